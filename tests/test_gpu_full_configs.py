"""GPU parity at the full workload sizes, in the launch configuration the benchmark times.

* The LLaDA-8B LM head at r_m = 0.1 / 0.5 / 0.9 and block decode: every element of the [M, V]
  output against the oracle (at most 3.8 TFLOP of fp64 on the host cores).
* Long context and the Dream-shaped batch (up to 10^2 TFLOP, too large for the oracle to check
  every element): 256 sampled rows (all V columns, with the first and last row of every chunk)
  plus every row on a seeded slice of 512 columns against the oracle; the chunked call (the workload's chunk_rows) equals the unchunked call
  bitwise; one-hot hidden states give out[i, v] == W[v, row(i) mod d] exactly, for every element.
"""
import numpy as np
import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz
from masked_token_lm_gb300 import workloads as wl
from oracle import mask_only_logits as orc
from tests.parity_utils import TOL, bits, column_parity, oracle_rows, sampled_parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def mo():
    m = mz.Mosaic(0)
    yield m
    m.close()


def call(mo, w, H, mask, W, chunk_rows):
    """Run one workload; returns the full [M, V] output (chunks copied out on-stream)."""
    odt = torch.float32 if w.out_dtype == "f32" else torch.bfloat16
    M = mask.M
    if 0 < chunk_rows < M:
        full = torch.empty((M, w.V), dtype=odt, device=DEV)

        def on_chunk(c, rb, rows, out):
            full[rb:rb + rows].copy_(out[:rows])

        mo.masked_logits(H, mask.idx, W, mask.seq_offsets, mask.mask_offsets, out_dtype=odt,
                         chunk_rows=chunk_rows, on_chunk=on_chunk)
        out = full
    else:
        out = mo.masked_logits(H, mask.idx, W, mask.seq_offsets, mask.mask_offsets, out_dtype=odt)
    assert mo.check() == mz.MOSAIC_OK, mz.mosaic_last_error_string()
    return out


def check_against_oracle(w, H, mask, W, out, seed):
    Hb, Wb = bits(H), bits(W)
    rows = oracle_rows(mask, w.L_tot)
    must = []
    if w.chunk_rows:
        for b in range(0, mask.M, w.chunk_rows):
            must += [b, min(mask.M, b + w.chunk_rows) - 1]
    # 256 seeded rows against all V columns (plus the first and last row of every chunk), and
    # every row on a seeded slice of 512 columns
    sampled_parity(Hb, Wb, rows, lambda ri: out[torch.from_numpy(ri).to(DEV)], torch.bfloat16
                   if w.out_dtype == "bf16" else torch.float32, seed, n_rows=256, must_rows=must)
    column_parity(Hb, Wb, rows, lambda cols: out[:, torch.from_numpy(cols).to(DEV)],
                  torch.bfloat16 if w.out_dtype == "bf16" else torch.float32, seed, n_cols=512)


@pytest.mark.parametrize("w", wl.LLADA + [wl.DECODE], ids=lambda w: w.name)
def test_unchunked_configs_every_element_matches_the_oracle(mo, w):
    H, W, mask = w.hidden(DEV), w.weight(DEV), w.mask().to(DEV)
    out = call(mo, w, H, mask, W, w.chunk_rows)
    rows = oracle_rows(mask, w.L_tot).astype(np.int32)
    ref = orc.masked_logits(bits(H), rows, bits(W))          # fp64 [M, V], every element
    tol = TOL[torch.bfloat16]
    worst = 0.0
    for r0 in range(0, mask.M, 512):                          # compare in row blocks
        r1 = min(mask.M, r0 + 512)
        got = out[r0:r1].float().cpu().numpy().astype(np.float64)
        err = np.abs(got - ref[r0:r1]) / (1.0 + np.abs(ref[r0:r1]))
        worst = max(worst, float(err.max()))
        assert worst <= tol, f"rows {r0}..{r1}: max scaled error {worst:.3e} > {tol}"
    # rounding to bf16 is the dominant error: well inside the tolerance, yet not vacuous
    assert 0.0 < worst <= 2.0 ** -8


@pytest.mark.parametrize("w", [wl.LONG[0], wl.LONG[3], wl.DREAM], ids=lambda w: w.name)
def test_chunked_configs_equal_unchunked_and_oracle(mo, w):
    H, W, mask = w.hidden(DEV), w.weight(DEV), w.mask().to(DEV)
    chunked = call(mo, w, H, mask, W, w.chunk_rows)
    whole = call(mo, w, H, mask, W, 0)
    assert torch.equal(chunked.view(torch.int16), whole.view(torch.int16))
    del whole
    check_against_oracle(w, H, mask, W, chunked, seed=w.seed)


def test_long_config_middle_ratios_chunked_equal_unchunked(mo):
    for w in wl.LONG[1:3]:
        H, W, mask = w.hidden(DEV), w.weight(DEV), w.mask().to(DEV)
        chunked = call(mo, w, H, mask, W, w.chunk_rows)
        whole = call(mo, w, H, mask, W, 0)
        assert torch.equal(chunked.view(torch.int16), whole.view(torch.int16)), w.name
        del chunked, whole


@pytest.mark.parametrize("w", [wl.DECODE, wl.DREAM], ids=lambda w: w.name)
def test_one_hot_full_size_is_bit_exact(mo, w):
    # H[r, :] = e_(r mod d) at the workload's full shape: every output element is one weight.
    r = torch.arange(w.L_tot, device=DEV)
    H = torch.zeros((w.L_tot, w.d), dtype=torch.bfloat16, device=DEV)
    H[r, r % w.d] = 1.0
    W = w.weight(DEV)
    m = w.mask()
    rows = torch.from_numpy(oracle_rows(m, w.L_tot)).to(DEV)
    out = call(mo, w, H, m.to(DEV), W, w.chunk_rows)
    want = W.t()[rows % w.d]  # [M, V]: row i is column (row(i) mod d) of W
    assert torch.equal(out.view(torch.int16), want.contiguous().view(torch.int16))
