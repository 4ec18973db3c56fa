"""Host-side argument checks of the torch wrappers (no GPU): a tensor whose size does not match
the extents the C ABI call implies is rejected before anything reaches the library, since the
kernels would read or write past it."""
import types

import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz

FAKE = types.SimpleNamespace(handle=None, device=0)  # never used: every case fails before


def bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def i32(*vals):
    return torch.tensor(vals, dtype=torch.int32)


H, W, IDX = bf(16, 32), bf(40, 32), i32(1, 2, 3)


@pytest.mark.parametrize("kw, what", [
    (dict(out=torch.zeros((3, 41), dtype=torch.bfloat16)), "shape"),
    (dict(out=torch.zeros((2, 40), dtype=torch.bfloat16)), "shape"),
    (dict(out=torch.zeros((3, 40), dtype=torch.float32), out_dtype=torch.bfloat16), "contiguous"),
    (dict(out=torch.zeros((40, 3), dtype=torch.bfloat16).t()), "contiguous"),
    (dict(out=torch.zeros((2, 40), dtype=torch.bfloat16), chunk_rows=1), "shape"),
    (dict(out_dtype=torch.float16), "out_dtype"),
    (dict(seq_offsets=i32(0, 16)), "both"),
    (dict(seq_offsets=i32(0, 8, 16), mask_offsets=i32(0, 3)), r"B \+ 1"),
    (dict(seq_offsets=i32(0), mask_offsets=i32(0)), r"B \+ 1"),
    (dict(seq_offsets=i32(0, 16).long(), mask_offsets=i32(0, 3)), "int32"),
])
def test_masked_logits_rejects_mismatched_tensors(kw, what):
    with pytest.raises(ValueError, match=what):
        mz.Mosaic.masked_logits(FAKE, H, IDX, W, **kw)


def test_masked_logits_rejects_bad_operands():
    with pytest.raises(ValueError, match="contiguous"):
        mz.Mosaic.masked_logits(FAKE, bf(32, 16).t(), IDX, W)
    with pytest.raises(ValueError, match="agree on d"):
        mz.Mosaic.masked_logits(FAKE, bf(16, 24), IDX, W)
    with pytest.raises(ValueError, match="int32"):
        mz.Mosaic.masked_logits(FAKE, H, IDX.long(), W)
    with pytest.raises(ValueError, match="one-dimensional"):
        mz.Mosaic.masked_logits(FAKE, H, IDX.view(1, 3), W)


def test_masked_logits_fp8_checks_scales_and_codes():
    hq, wq = torch.zeros((16, 32), dtype=torch.uint8), torch.zeros((40, 32), dtype=torch.uint8)
    sh, sw = torch.ones(16), torch.ones(40)
    call = lambda **kw: mz.Mosaic.masked_logits_fp8(
        FAKE, kw.get("hq", hq), kw.get("sh", sh), IDX, kw.get("wq", wq), kw.get("sw", sw),
        out=kw.get("out"))
    with pytest.raises(ValueError, match="hidden_scale"):
        call(sh=torch.ones(15))
    with pytest.raises(ValueError, match="w_scale"):
        call(sw=torch.ones(39))
    with pytest.raises(ValueError, match="w_scale"):
        call(sw=torch.ones(40, dtype=torch.float64))
    with pytest.raises(ValueError, match="W_q"):
        call(wq=bf(40, 32))
    with pytest.raises(ValueError, match="shape"):
        call(out=torch.zeros((4, 40), dtype=torch.bfloat16))


def test_quantize_masked_rows_checks_the_code_buffers():
    q, s = torch.zeros((16, 32), dtype=torch.uint8), torch.zeros(16)
    with pytest.raises(ValueError, match="hidden_q"):
        mz.quantize_masked_rows_e4m3(H, IDX, torch.zeros((15, 32), dtype=torch.uint8), s)
    with pytest.raises(ValueError, match="hidden_scale"):
        mz.quantize_masked_rows_e4m3(H, IDX, q, torch.zeros(8))
    with pytest.raises(ValueError, match="both"):
        mz.quantize_masked_rows_e4m3(H, IDX, q, s, seq_offsets=i32(0, 16))


def test_masked_sample_checks_operands():
    with pytest.raises(ValueError, match="W"):
        mz.Mosaic.masked_sample(FAKE, H, IDX, W.float())
    with pytest.raises(ValueError, match="B \\+ 1"):
        mz.Mosaic.masked_sample(FAKE, H, IDX, W, i32(0, 16), i32(0, 1, 3))
