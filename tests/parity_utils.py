"""Helpers shared by the GPU parity tests: bf16 bit views, the tolerance rule, and sampled
parity against the CPU oracle for workloads too large to check in full."""
from __future__ import annotations

import numpy as np
import torch

from oracle import mask_only_logits as orc

# max |gpu - ref| <= TOL * (1 + |ref|), ref = the oracle's exact (fp64) value before rounding
TOL = {torch.float32: 1e-3, torch.bfloat16: 1.5e-2}


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (copied to the host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy().astype(np.float64)


def assert_close(got: torch.Tensor, ref: np.ndarray, out_dtype, what=""):
    g = as_f64(got)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref) / (1.0 + np.abs(ref))
    worst = float(err.max()) if err.size else 0.0
    assert worst <= TOL[out_dtype], f"{what}: max scaled error {worst:.3e} > {TOL[out_dtype]}"
    return worst


def oracle_rows(mask, L_tot):
    so = None if mask.seq_offsets is None else mask.seq_offsets.cpu().numpy()
    mo = None if mask.mask_offsets is None else mask.mask_offsets.cpu().numpy()
    return orc.resolve_rows(mask.idx.cpu().numpy(), L_tot, so, mo)


def sampled_parity(H_bits, W_bits, rows, get_rows, out_dtype, seed, n_rows=48, must_rows=()):
    """Compare sampled output rows with the oracle, all V columns of each.

    H_bits/W_bits: host uint16 patterns of the full inputs; rows: the oracle's resolved hidden
    row per output row; get_rows(i_array) -> torch tensor [len(i), V] of GPU outputs. The rows are
    n_rows seeded ones, the first and the last, and must_rows."""
    M = rows.shape[0]
    g = np.random.default_rng(seed)
    ri = set(g.choice(M, min(n_rows, M), replace=False).tolist()) | {0, M - 1} | set(must_rows)
    ri = np.array(sorted(i for i in ri if 0 <= i < M))
    ref = orc.masked_logits(H_bits, rows[ri].astype(np.int32), W_bits)
    worst = assert_close(get_rows(ri), ref, out_dtype, "sampled rows")
    return ri, worst


def column_parity(H_bits, W_bits, rows, get_cols, out_dtype, seed, n_cols=256):
    V = W_bits.shape[0]
    g = np.random.default_rng(seed + 1)
    cols = np.sort(g.choice(V, min(n_cols, V), replace=False))
    ref = orc.masked_logits(H_bits, rows.astype(np.int32), W_bits[cols])
    return assert_close(get_cols(cols), ref, out_dtype, "sampled columns")
