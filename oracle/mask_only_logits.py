"""CPU oracle for mask-only logits -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
module. The product path (``masked_token_lm_gb300``) never imports it and shares no code with it.

What it computes, from the pages:

* "Mosaic: Unlocking Long-Context Inference for Diffusion LLMs via Global Memory" (paper review),
  section 3, observation #2: existing systems compute logits for every token at every step, yet
  only the masked tokens are sampled, so mask-only logits computes them for the masked tokens
  alone. Its "core components 1. Mask-only Logits Kernel" entry: the kernel takes the hidden
  states of all tokens plus the mask indices and addresses the hidden rows indirectly through
  them. The arXiv abstract page adds that the system preserves exact model outputs.
  => out[i, :] = H[row(i), :] @ W^T, i.e. row ``row(i)`` of the full logits H @ W^T.
* "扩散大语言模型内存优化：Mosaic系统突破与实践", section 2.3 (lazy chunking) and the dLLM-Serve
  article "扩散大语言模型内存优化：从理论到系统设计", section 3.2.2: when too many rows need
  logits, the rows are cut into consecutive slices, the LM head is applied per slice and the
  pieces are concatenated. => the chunked result equals the unchunked one.

Readings where the pages are silent (all listed in the design notes):

* logits = H @ W^T with no bias, scale or soft-cap (the pages never mention one);
* exact arithmetic is approximated by fp64 (the default) -- bf16 inputs make every product exact
  in fp64 and the only error is fp64 summation, far below any tolerance used against it; the
  "naive fp32-accumulate GEMM" variant (``accumulate="f32"``) adds the products in ascending k
  order in fp32 without fused multiply-add;
* CSR: ``mask_offsets[B+1]`` slices ``idx`` per sequence, ``idx`` values are local to their
  sequence and the hidden row is ``seq_offsets[b] + idx[i]``; output rows keep index order;
* an index outside its sequence (or outside H) is an error: the oracle raises ``IndexError``;
* bf16 output is round-to-nearest-even of the exact value.

Plain by design: a gather followed by one library matmul (fp64) or an explicit k loop (fp32);
nothing is blocked, fused or reordered beyond that.
"""
from __future__ import annotations

from typing import Iterator, Optional, Tuple

import numpy as np


# ---------------------------------------------------------------------------------------------
# bf16 <-> wider floats, written from the IEEE-754 binary16-brain-float definition:
# bf16 is the upper 16 bits of an IEEE binary32 (1 sign, 8 exponent, 7 fraction bits).
# ---------------------------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16, ties to even (finite inputs only).

    Done in two exact steps: scale by the bf16 ulp of each value's binade, round to an integer
    with numpy's ties-to-even ``rint``, then encode. bf16 keeps 8 significant bits; values below
    2**-126 use the fixed subnormal spacing 2**-133.
    """
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value")
    ax = np.abs(x)
    # exponent e with 2**e <= |x| < 2**(e+1); frexp gives |x| = f * 2**E, f in [0.5, 1)
    _, E = np.frexp(ax)
    e = E.astype(np.int64) - 1
    e = np.maximum(e, -126)                        # subnormal range shares the 2**-126 binade spacing
    ulp_exp = e - 7                                # 8 significant bits -> spacing 2**(e-7)
    q = np.rint(np.ldexp(ax, -ulp_exp))            # exact scaling by a power of two; RNE to integer
    r = np.ldexp(q, ulp_exp)                       # exact: q has <= 9 bits
    if np.any(r > np.float64(np.float32(3.3895313892515355e38))):
        raise OverflowError("value rounds beyond the largest finite bf16")
    r32 = (np.copysign(r, x)).astype(np.float32)   # r is representable in bf16, hence in f32
    return (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------------------------
# Mask indices -> hidden rows.
# ---------------------------------------------------------------------------------------------

def resolve_rows(idx: np.ndarray, L_tot: int, seq_offsets: Optional[np.ndarray] = None,
                 mask_offsets: Optional[np.ndarray] = None) -> np.ndarray:
    """Hidden-state row of every masked position, in output order.

    Flat mode (no offsets): row(i) = idx[i]. CSR mode: positions
    ``mask_offsets[b] <= i < mask_offsets[b+1]`` belong to sequence b and
    row(i) = seq_offsets[b] + idx[i], with 0 <= idx[i] < seq_offsets[b+1] - seq_offsets[b].
    Raises IndexError for any index outside its sequence or outside H, ValueError for
    malformed offsets.
    """
    idx = np.asarray(idx, dtype=np.int64)
    M = idx.shape[0]
    if (seq_offsets is None) != (mask_offsets is None):
        raise ValueError("CSR mode needs both seq_offsets and mask_offsets")
    if seq_offsets is None:
        rows = idx.copy()
    else:
        so = np.asarray(seq_offsets, dtype=np.int64)
        mo = np.asarray(mask_offsets, dtype=np.int64)
        if so.shape != mo.shape or so.ndim != 1 or so.shape[0] < 1:
            raise ValueError("offset arrays must both have B+1 entries")
        if mo[0] != 0 or mo[-1] != M or np.any(np.diff(mo) < 0):
            raise ValueError("mask_offsets must rise from 0 to M")
        if so[0] < 0 or so[-1] > L_tot or np.any(np.diff(so) < 0):
            raise ValueError("seq_offsets must rise within [0, L_tot]")
        rows = np.empty(M, dtype=np.int64)
        for b in range(so.shape[0] - 1):
            lo, hi = int(mo[b]), int(mo[b + 1])
            local = idx[lo:hi]
            seq_len = int(so[b + 1] - so[b])
            if np.any(local < 0) or np.any(local >= seq_len):
                raise IndexError(f"local index outside sequence {b}")
            rows[lo:hi] = so[b] + local
    if np.any(rows < 0) or np.any(rows >= L_tot):
        raise IndexError("mask index outside hidden states")
    return rows


# ---------------------------------------------------------------------------------------------
# Logits.
# ---------------------------------------------------------------------------------------------

def full_logits(H_bits: np.ndarray, W_bits: np.ndarray) -> np.ndarray:
    """All-token logits H @ W^T in float64: [L_tot, V]."""
    H = bf16_bits_to_f64(H_bits)
    W = bf16_bits_to_f64(W_bits)
    return H @ W.T


def _naive_f32(A: np.ndarray, W: np.ndarray) -> np.ndarray:
    """acc[i, v] = sum_k A[i, k] * W[v, k], added in ascending k, each step rounded to fp32."""
    M, d = A.shape
    V = W.shape[0]
    A32 = A.astype(np.float32)
    W32 = W.astype(np.float32)
    acc = np.zeros((M, V), dtype=np.float32)
    for k in range(d):
        # bf16 x bf16 has at most 16 significant bits, so this fp32 product is exact; the add
        # is a separate, rounded fp32 operation.
        acc += np.outer(A32[:, k], W32[:, k]).astype(np.float32)
    return acc


def masked_logits(H_bits: np.ndarray, idx: np.ndarray, W_bits: np.ndarray,
                  seq_offsets: Optional[np.ndarray] = None,
                  mask_offsets: Optional[np.ndarray] = None,
                  accumulate: str = "f64") -> np.ndarray:
    """Mask-only logits: gather the masked rows of H, then multiply by W^T.

    H_bits: uint16 bf16 patterns [L_tot, d]; W_bits: [V, d]; returns [M, V] float64
    (``accumulate="f64"``) or float32 (``accumulate="f32"``, naive ascending-k fp32 sums).
    """
    H_bits = np.asarray(H_bits)
    W_bits = np.asarray(W_bits)
    L_tot, d = H_bits.shape
    V, dw = W_bits.shape
    if dw != d:
        raise ValueError("H and W disagree on d")
    rows = resolve_rows(idx, L_tot, seq_offsets, mask_offsets)
    A = bf16_bits_to_f64(H_bits[rows])               # the gather: [M, d]
    W = bf16_bits_to_f64(W_bits)
    if accumulate == "f64":
        return A @ W.T
    if accumulate == "f32":
        return _naive_f32(A, W)
    raise ValueError(accumulate)


def round_output(acc: np.ndarray, out_dtype: str) -> np.ndarray:
    """Store the accumulated logits: fp32 (numpy's RNE cast) or bf16 bits (RNE)."""
    if out_dtype == "f32":
        return np.asarray(acc).astype(np.float32)
    if out_dtype == "bf16":
        return f64_to_bf16_bits(np.asarray(acc, dtype=np.float64))
    raise ValueError(out_dtype)


def chunk_ranges(M: int, chunk_rows: int) -> Iterator[Tuple[int, int]]:
    """Consecutive row slices [begin, end) of the flat index list. Chunking stays off (one
    slice) when ``chunk_rows <= 0`` or ``M <= chunk_rows``; no slice at all when M == 0."""
    if M == 0:
        return
    if chunk_rows <= 0 or M <= chunk_rows:
        yield 0, M
        return
    for b in range(0, M, chunk_rows):
        yield b, min(M, b + chunk_rows)


def masked_logits_chunked(H_bits, idx, W_bits, seq_offsets=None, mask_offsets=None,
                          chunk_rows: int = 0, accumulate: str = "f64") -> np.ndarray:
    """Slice the masked positions into chunks, compute each, concatenate in order."""
    idx = np.asarray(idx)
    L_tot = np.asarray(H_bits).shape[0]
    rows = resolve_rows(idx, L_tot, seq_offsets, mask_offsets)
    pieces = [masked_logits(H_bits, rows[b:e], W_bits, accumulate=accumulate)
              for b, e in chunk_ranges(rows.shape[0], chunk_rows)]
    V = np.asarray(W_bits).shape[0]
    if not pieces:
        return np.zeros((0, V), dtype=np.float64 if accumulate == "f64" else np.float32)
    return np.concatenate(pieces, axis=0)


def logits_bytes(rows: int, V: int, elt_bytes: int) -> int:
    """Bytes of a [rows, V] logit tensor with ``elt_bytes`` bytes per element."""
    return int(rows) * int(V) * int(elt_bytes)


# ---------------------------------------------------------------------------------------------
# Sampling the masked positions (the step after mask-only logits).
# ---------------------------------------------------------------------------------------------

def sample_from_logits(logits: np.ndarray):
    """Greedy token and its confidence for each row of a [M, V] logit matrix.

    "Mosaic: Unlocking Long-Context Inference for Diffusion LLMs via Global Memory" (paper review),
    section 3, observation #2: only the masked tokens are sampled. Reading (the pages give no
    sampler): greedy decoding, token = argmax_v logits[i, v] with ties going to the smallest v,
    and confidence = the softmax probability of that token, max_v softmax(logits[i])_v =
    1 / sum_v exp(logits[i, v] - max_v logits[i, v]). Returns (int64 [M], float64 [M]).
    """
    z = np.asarray(logits, dtype=np.float64)
    if z.shape[0] == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.float64)
    token = np.argmax(z, axis=1)  # numpy returns the first occurrence of the maximum
    zmax = z[np.arange(z.shape[0]), token]
    conf = 1.0 / np.sum(np.exp(z - zmax[:, None]), axis=1)
    return token.astype(np.int64), conf


def masked_sample(H_bits, idx, W_bits, seq_offsets=None, mask_offsets=None):
    """Token and confidence of every masked position: sampling applied to mask-only logits."""
    return sample_from_logits(masked_logits(H_bits, idx, W_bits, seq_offsets, mask_offsets))
