"""CPU oracle for mask-only logits -- test infrastructure, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it.
It shares no code with ``masked_token_lm_gb300`` and never imports it.
"""
from .mask_only_logits import (  # noqa: F401
    bf16_bits_to_f64,
    chunk_ranges,
    f64_to_bf16_bits,
    full_logits,
    logits_bytes,
    masked_logits,
    masked_logits_chunked,
    masked_sample,
    sample_from_logits,
    resolve_rows,
    round_output,
)
from .fp8_logits import (  # noqa: F401
    e4m3_bits_to_f64,
    f64_to_e4m3_bits,
    masked_logits_fp8,
    quantize_rows,
)
