"""GPU parity of the FP8 (E4M3) variant at the full workload sizes, in the launch configuration
`bench.py --mode fp8` times: W quantized once, only the masked hidden rows quantized, then one
fused call. Too large for the oracle to check every element, so sampled rows (all V columns, in
slices) and every row on a seeded set of columns are checked against the oracle's logits from the
same quantized operands; a chunked call must equal the unchunked call bit for bit.
"""
import numpy as np
import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz
from masked_token_lm_gb300 import workloads as wl
from oracle import fp8_logits as f8
from tests.parity_utils import TOL, oracle_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def mo():
    m = mz.Mosaic(0)
    yield m
    m.close()


def quantized_inputs(w):
    H, W, mask = w.hidden(DEV), w.weight(DEV), w.mask().to(DEV)
    qW, sW = mz.quantize_rows_e4m3(W)
    qH = torch.zeros(H.shape, dtype=torch.uint8, device=DEV)
    sH = torch.zeros(H.shape[0], dtype=torch.float32, device=DEV)
    mz.quantize_masked_rows_e4m3(H, mask.idx, qH, sH, mask.seq_offsets, mask.mask_offsets)
    torch.cuda.synchronize()
    del H, W
    return qH, sH, qW, sW, mask


def run(mo, w, qH, sH, qW, sW, mask, chunk_rows):
    M = mask.M
    if 0 < chunk_rows < M:
        full = torch.empty((M, w.V), dtype=torch.bfloat16, device=DEV)

        def on_chunk(c, rb, rows, out):
            full[rb:rb + rows].copy_(out[:rows])

        mo.masked_logits_fp8(qH, sH, mask.idx, qW, sW, mask.seq_offsets, mask.mask_offsets,
                             chunk_rows=chunk_rows, on_chunk=on_chunk)
        out = full
    else:
        out = mo.masked_logits_fp8(qH, sH, mask.idx, qW, sW, mask.seq_offsets, mask.mask_offsets)
    assert mo.check() == mz.MOSAIC_OK, mz.mosaic_last_error_string()
    return out


def check(w, qH, sH, qW, sW, mask, out, seed):
    rows = oracle_rows(mask, w.L_tot)
    M = rows.shape[0]
    qHn, sHn, qWn, sWn = qH.cpu().numpy(), sH.cpu().numpy(), qW.cpu().numpy(), sW.cpu().numpy()
    g = np.random.default_rng(seed)
    ri = np.array(sorted(set(g.choice(M, min(40, M), replace=False).tolist()) | {0, M - 1}))
    got = out[torch.from_numpy(ri).to(DEV)].float().cpu().numpy().astype(np.float64)
    worst = 0.0
    for c0 in range(0, w.V, 16384):           # all columns of the sampled rows, in slices
        c1 = min(w.V, c0 + 16384)
        ref = f8.masked_logits_fp8(qHn, sHn, rows[ri], qWn[c0:c1], sWn[c0:c1])
        worst = max(worst, float(np.max(np.abs(got[:, c0:c1] - ref) / (1 + np.abs(ref)))))
    assert worst <= TOL[torch.bfloat16], f"sampled rows: {worst:.3g}"
    cols = np.sort(np.random.default_rng(seed + 1).choice(w.V, 128, replace=False))
    ref = f8.masked_logits_fp8(qHn, sHn, rows, qWn[cols], sWn[cols])
    got = out[:, torch.from_numpy(cols).to(DEV)].float().cpu().numpy().astype(np.float64)
    err = float(np.max(np.abs(got - ref) / (1 + np.abs(ref))))
    assert err <= TOL[torch.bfloat16], f"sampled columns: {err:.3g}"


@pytest.mark.parametrize("w", [wl.LLADA[1], wl.DECODE], ids=lambda w: w.name)
def test_fp8_full_size_sampled_parity(mo, w):
    qH, sH, qW, sW, mask = quantized_inputs(w)
    out = run(mo, w, qH, sH, qW, sW, mask, w.chunk_rows)
    check(w, qH, sH, qW, sW, mask, out, seed=w.seed)


def test_fp8_long_context_chunked_equals_unchunked_and_oracle(mo):
    w = wl.LONG[0]   # L = 131072, r_m = 0.05: 6554 rows in two 4096-row chunks
    qH, sH, qW, sW, mask = quantized_inputs(w)
    chunked = run(mo, w, qH, sH, qW, sW, mask, w.chunk_rows)
    whole = run(mo, w, qH, sH, qW, sW, mask, 0)
    assert torch.equal(chunked.view(torch.int16), whole.view(torch.int16))
    del whole
    check(w, qH, sH, qW, sW, mask, chunked, seed=w.seed)


def test_fp8_dream_shape_chunked_equals_unchunked_and_oracle(mo):
    w = wl.DREAM     # ragged 8 x 32768, CSR, d = 3584, V = 152,064, chunks of 8192 rows
    qH, sH, qW, sW, mask = quantized_inputs(w)
    chunked = run(mo, w, qH, sH, qW, sW, mask, w.chunk_rows)
    whole = run(mo, w, qH, sH, qW, sW, mask, 0)
    assert torch.equal(chunked.view(torch.int16), whole.view(torch.int16))
    del whole
    check(w, qH, sH, qW, sW, mask, chunked, seed=w.seed)
