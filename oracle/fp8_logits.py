"""CPU oracle for the FP8 variant of mask-only logits -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
module. The product path (``masked_token_lm_gb300``) never imports it and shares no code with it.

The dLLM-Serve article "扩散大语言模型内存优化：从理论到系统设计", section 5 (extensions and
future directions), names combining the logit work with FP8 quantization as a next step; the pages
give no scheme. Readings taken here (all listed in the design notes):

* Format: FP8 E4M3 in its "fn" form -- 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits, no
  infinities, the single NaN pattern S.1111.111 per sign, largest finite value 448, smallest
  normal 2^-6, subnormal spacing 2^-9.
* Scaling per row (one scale per hidden-state row and per W row, i.e. per output row and column):
  a = max |x| over the row (exact), scale = fp32(a / 448), inv = fp32(448 / a) (IEEE fp32
  divisions, round to nearest even), q = e4m3(fp32(x * inv)) rounded to nearest even and clamped
  to +-448. A row of zeros has scale 0 and codes 0.
* Logits: out[i, v] = scale_H[row(i)] * scale_W[v] * sum_k q_H[row(i), k] * q_W[v, k], the sum
  exact (every product of two e4m3 values is exact in fp64 and the fp64 sum of d <= 2^20 of them
  is within fp64 rounding), then stored like the bf16 path (bf16 RNE or fp32).

Plain by design: the quantization is written element by element from the format definition, and
the logits are a gather plus one library matmul.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

from .mask_only_logits import bf16_bits_to_f64, resolve_rows

E4M3_MAX = 448.0
E4M3_BIAS = 7


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Value of E4M3 ("fn") codes (uint8) as float64; NaN for S.1111.111."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - E4M3_BIAS).astype(np.int64))
    subnormal = sign * np.ldexp(m / 8.0, 1 - E4M3_BIAS)
    out = np.where(e == 0, subnormal, normal)
    return np.where((e == 0xF) & ((b & 0x7) == 0x7), np.nan, out)


def f64_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round finite values to E4M3 codes: nearest, ties to even, results beyond 448 clamped to
    448 (the largest finite value). Values that are exact in float32 are rounded exactly."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value")
    ax = np.abs(x)
    _, E = np.frexp(ax)                     # ax = f * 2**E, f in [0.5, 1)
    e = np.maximum(E.astype(np.int64) - 1, 1 - E4M3_BIAS)  # binade; subnormals share 2**-6's
    ulp_exp = e - 3                          # 4 significant bits -> spacing 2**(e-3)
    q = np.rint(np.ldexp(ax, -ulp_exp))      # exact scaling, RNE to an integer
    r = np.minimum(np.ldexp(q, ulp_exp), E4M3_MAX)  # exact; clamp the overflow
    # encode the (now representable) magnitude r
    _, Er = np.frexp(r)
    er = Er.astype(np.int64) - 1
    sub = r < 2.0 ** (1 - E4M3_BIAS)
    man_sub = np.rint(np.ldexp(r, 9)).astype(np.int64)                 # r / 2**-9
    exp_n = np.where(sub, 0, er + E4M3_BIAS)
    man_n = np.rint((np.ldexp(r, -np.where(sub, 0, er)) - 1.0) * 8.0).astype(np.int64)
    code = np.where(sub, man_sub, (exp_n << 3) | man_n)
    code = np.where(r == 0, 0, code)
    code = code | np.where(np.signbit(x), 0x80, 0)          # rounding keeps the sign, even of 0
    return code.astype(np.uint8)


def quantize_rows(x_bits: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-row E4M3 quantization of a bf16 matrix (uint16 bit patterns [R, d]).

    Returns (codes uint8 [R, d], scale float32 [R]) with x ~= scale * decode(codes)."""
    x = bf16_bits_to_f64(x_bits).astype(np.float32)       # exact: bf16 is a subset of fp32
    a = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    a = a.astype(np.float32)
    zero = a == 0
    safe = np.where(zero, np.float32(1), a).astype(np.float32)
    scale = np.where(zero, np.float32(0), safe / np.float32(E4M3_MAX)).astype(np.float32)
    inv = np.where(zero, np.float32(0), np.float32(E4M3_MAX) / safe).astype(np.float32)
    y = (x * inv[:, None]).astype(np.float32)              # one fp32 multiply, RNE
    return f64_to_e4m3_bits(y.astype(np.float64)), scale


def masked_logits_fp8(qH: np.ndarray, sH: np.ndarray, idx: np.ndarray, qW: np.ndarray,
                      sW: np.ndarray, seq_offsets: Optional[np.ndarray] = None,
                      mask_offsets: Optional[np.ndarray] = None) -> np.ndarray:
    """Mask-only logits from quantized operands: [M, V] float64.

    qH: E4M3 codes [L_tot, d], sH: float32 [L_tot]; qW: [V, d], sW: [V]."""
    qH = np.asarray(qH)
    L_tot, d = qH.shape
    if np.asarray(qW).shape[1] != d:
        raise ValueError("H and W disagree on d")
    rows = resolve_rows(idx, L_tot, seq_offsets, mask_offsets)
    A = e4m3_bits_to_f64(qH[rows])                          # the gather: [M, d]
    B = e4m3_bits_to_f64(qW)
    acc = A @ B.T
    sa = np.asarray(sH, dtype=np.float64)[rows]
    sb = np.asarray(sW, dtype=np.float64)
    return acc * sa[:, None] * sb[None, :]
