"""GPU parity of the fused gather-GEMM + greedy sampling (token = argmax, confidence = max
softmax probability) against the CPU oracle.

The argmax is an integer decided by floating point, so it is compared this way: the GPU's token
must be a valid argmax of the oracle's exact logits within the fp32 tolerance (its logit within
1e-3 * (1 + |max|) of the maximum), and must equal the oracle's token wherever the top two
logits are further apart than twice that. On inputs where fp32 accumulation is exact (integer
values, one-hot hidden states) the token must match exactly, ties going to the smallest index.
"""
import numpy as np
import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz
from masked_token_lm_gb300 import workloads as wl
from oracle import mask_only_logits as orc
from tests.parity_utils import bits, oracle_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 1e-3   # fp32 logits
CONF_RTOL = 1e-2


@pytest.fixture(scope="module")
def mo():
    m = mz.Mosaic(0)
    yield m
    m.close()


def check_against_logits(token, conf, logits):
    """token/conf from the GPU, logits: the oracle's fp64 [M, V]."""
    token = token.cpu().numpy().astype(np.int64)
    conf = conf.cpu().numpy().astype(np.float64)
    M = logits.shape[0]
    assert np.all((token >= 0) & (token < logits.shape[1]))
    zmax = logits.max(axis=1)
    tol = TOL * (1 + np.abs(zmax))
    assert np.all(logits[np.arange(M), token] >= zmax - tol), "token is not a valid argmax"
    part = np.partition(logits, -2, axis=1)
    gap = part[:, -1] - part[:, -2]
    t_ref, c_ref = orc.sample_from_logits(logits)
    clear = gap > 2 * tol
    assert np.array_equal(token[clear], t_ref[clear])
    np.testing.assert_allclose(conf, c_ref, rtol=CONF_RTOL, atol=0)
    return int(clear.sum())


@pytest.mark.parametrize("L,d,V,M", [
    (1000, 512, 1000, 300),    # V not a multiple of 256: padded columns must not count
    (777, 200, 520, 129),      # K tail, M tail
    (300, 64, 256, 100),       # single M tile (one CTA per tile)
    (2000, 1024, 8200, 700),
    (600, 256, 520, 300),      # one-panel unit column, split last round with an empty half
    (2000, 256, 15104, 700),   # 90 units over 76 pairs: split last round, odd panels
])
def test_sample_matches_oracle(mo, L, d, V, M):
    H = wl.make_hidden(L, d, 3 + L, DEV)
    W = wl.make_weight(V, d, 4 + V, DEV) * 8  # wider logits: a sharper softmax
    W = W.to(torch.bfloat16)
    idx = wl.uniform_positions(L, M, seed=M)
    token, conf = mo.masked_sample(H, idx.to(DEV), W)
    assert mo.check() == mz.MOSAIC_OK
    logits = orc.masked_logits(bits(H), idx.numpy(), bits(W))
    assert check_against_logits(token, conf, logits) > 0.9 * M


def test_sample_integer_inputs_exact_with_ties(mo):
    L, d, V, M = 600, 64, 1000, 257
    g = torch.Generator().manual_seed(8)
    Hi = torch.randint(-1, 2, (L, d), generator=g)
    Wi = torch.randint(-1, 2, (V, d), generator=g)   # small range: many exact ties
    H, W = Hi.to(torch.bfloat16).to(DEV), Wi.to(torch.bfloat16).to(DEV)
    idx = wl.uniform_positions(L, M, seed=6)
    token, conf = mo.masked_sample(H, idx.to(DEV), W)
    assert mo.check() == mz.MOSAIC_OK
    exact = (Hi[idx.long()].long() @ Wi.long().T).numpy()
    first = np.array([int(np.flatnonzero(r == r.max())[0]) for r in exact])
    assert np.array_equal(token.cpu().numpy(), first)
    t_ref, c_ref = orc.sample_from_logits(exact.astype(np.float64))
    np.testing.assert_allclose(conf.cpu().numpy(), c_ref, rtol=1e-5)


def test_sample_one_hot_exact(mo):
    L, d, V, M = 900, 128, 1032, 333
    Hf = torch.zeros((L, d))
    Hf[torch.arange(L), torch.arange(L) % d] = 1.0
    H = Hf.to(torch.bfloat16).to(DEV)
    W = wl.make_weight(V, d, 21, DEV)
    idx = torch.randint(0, L, (M,), generator=torch.Generator().manual_seed(2), dtype=torch.int32)
    token, _ = mo.masked_sample(H, idx.to(DEV), W)
    Wf = orc.bf16_bits_to_f64(bits(W))
    want = [int(np.argmax(Wf[:, r % d])) for r in idx.numpy()]
    assert token.cpu().tolist() == want


def test_sample_agrees_with_the_logits_path_bit_for_bit(mo):
    # both read the same fp32 accumulators: the token is the first maximum of the fp32 logits
    L, d, V, M = 1500, 768, 4104, 600
    H, W = wl.make_hidden(L, d, 31, DEV), wl.make_weight(V, d, 32, DEV)
    idx = wl.uniform_positions(L, M, seed=33).to(DEV)
    token, conf = mo.masked_sample(H, idx, W)
    logits = mo.masked_logits(H, idx, W, out_dtype=torch.float32)
    assert mo.check() == mz.MOSAIC_OK
    lg = logits.double().cpu().numpy()
    first = np.array([int(np.flatnonzero(r == r.max())[0]) for r in lg])
    assert np.array_equal(token.cpu().numpy(), first)
    _, c_ref = orc.sample_from_logits(lg)
    np.testing.assert_allclose(conf.cpu().numpy(), c_ref, rtol=1e-4)


@pytest.mark.parametrize("chunk_rows", [1, 100, 128, 300])
def test_sample_chunked_equals_unchunked(mo, chunk_rows):
    L, d, V, M = 1200, 320, 1288, 300
    H, W = wl.make_hidden(L, d, 17, DEV), wl.make_weight(V, d, 18, DEV)
    idx = wl.uniform_positions(L, M, seed=18).to(DEV)
    t0, c0 = mo.masked_sample(H, idx, W)
    t1, c1 = mo.masked_sample(H, idx, W, chunk_rows=chunk_rows)
    assert torch.equal(t0, t1) and torch.equal(c0, c1)


def test_sample_csr_and_bad_index(mo):
    m = wl.ragged_mask(4, 300, seed=9)
    d, V = 128, 520
    H, W = wl.make_hidden(1200, d, 41, DEV), wl.make_weight(V, d, 42, DEV)
    mm = m.to(DEV)
    token, conf = mo.masked_sample(H, mm.idx, W, mm.seq_offsets, mm.mask_offsets)
    assert mo.check() == mz.MOSAIC_OK
    logits = orc.masked_logits(bits(H), m.idx.numpy(), bits(W), m.seq_offsets.numpy(), m.mask_offsets.numpy())
    check_against_logits(token, conf, logits)
    bad = m.idx.clone()
    bad[3] = 10_000
    token, conf = mo.masked_sample(H, bad.to(DEV), W, mm.seq_offsets, mm.mask_offsets)
    assert mo.check() == mz.MOSAIC_ERR_INDEX
    assert int(token[3]) == -1 and float(conf[3]) == 0.0
    assert int(token[4]) >= 0


def test_sample_workspace_too_small_is_rejected(mo):
    H, W = wl.make_hidden(64, 64, 1, DEV), wl.make_weight(256, 64, 2, DEV)
    idx = torch.arange(8, dtype=torch.int32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(mz.MosaicError) as e:
        mo.masked_sample(H, idx, W, workspace=ws)
    assert e.value.status == mz.MOSAIC_ERR_INVALID_ARG


@pytest.mark.parametrize("w", [wl.LLADA[2], wl.DECODE], ids=lambda w: w.name)
def test_sample_full_size_sampled_rows(mo, w):
    H, W, mask = w.hidden(DEV), w.weight(DEV), w.mask().to(DEV)
    token, conf = mo.masked_sample(H, mask.idx, W, mask.seq_offsets, mask.mask_offsets)
    assert mo.check() == mz.MOSAIC_OK
    rows = oracle_rows(mask, w.L_tot)
    ri = np.sort(np.random.default_rng(w.seed).choice(mask.M, 48, replace=False))
    logits = orc.masked_logits(bits(H), rows[ri].astype(np.int32), bits(W))
    check_against_logits(token[torch.from_numpy(ri).to(DEV)], conf[torch.from_numpy(ri).to(DEV)], logits)


def test_sample_full_size_every_row_llada_r05(mo):
    """Every masked row of the LLaDA-8B r_m = 0.5 shape (M = 2048) against the oracle's logits."""
    w = wl.LLADA[1]
    H, W, mask = w.hidden(DEV), w.weight(DEV), w.mask().to(DEV)
    token, conf = mo.masked_sample(H, mask.idx, W)
    assert mo.check() == mz.MOSAIC_OK
    rows = oracle_rows(mask, w.L_tot).astype(np.int32)
    logits = orc.masked_logits(bits(H), rows, bits(W))
    clear = check_against_logits(token, conf, logits)
    assert clear > 0.8 * mask.M  # the exact-token comparison covers most rows


def test_sample_dream_shape_chunked_equals_unchunked_and_oracle(mo):
    """The Dream-shaped ragged batch (CSR, M = 172,201) sampled in the bench's chunks of 8192
    rows equals the unchunked call bit for bit; sampled rows against the oracle."""
    w = wl.DREAM
    H, W, mask = w.hidden(DEV), w.weight(DEV), w.mask().to(DEV)
    t1, c1 = mo.masked_sample(H, mask.idx, W, mask.seq_offsets, mask.mask_offsets,
                              chunk_rows=w.chunk_rows)
    t0, c0 = mo.masked_sample(H, mask.idx, W, mask.seq_offsets, mask.mask_offsets)
    assert mo.check() == mz.MOSAIC_OK
    assert torch.equal(t0, t1) and torch.equal(c0, c1)
    rows = oracle_rows(mask, w.L_tot)
    M = mask.M
    # rows of every sequence (first and last rows included) and of every chunk boundary
    ri = set(np.random.default_rng(w.seed).choice(M, 40, replace=False).tolist()) | {0, M - 1}
    ri |= {b for b in range(0, M, w.chunk_rows)} | {min(M, b + w.chunk_rows) - 1 for b in range(0, M, w.chunk_rows)}
    ri = np.array(sorted(ri))
    logits = orc.masked_logits(bits(H), rows[ri].astype(np.int32), bits(W))
    sel = torch.from_numpy(ri).to(DEV)
    check_against_logits(t1[sel], c1[sel], logits)


def test_sample_timeout_reports_and_the_next_call_is_exact(mo):
    """A bounded wait that runs out inside the sampling kernel of a CTA pair (the epilogue holds
    a whole slot in registers) reports a timeout; the next call on the same context is exact."""
    L, d, V, M = 2048, 1024, 8200, 700
    H = wl.make_hidden(L, d, 51, DEV)
    W = wl.make_weight(V, d, 52, DEV)
    idx = wl.uniform_positions(L, M, seed=53).to(DEV)
    mo.set_wait_timeout(0)  # every wait that is not already satisfied gives up at once
    try:
        mo.masked_sample(H, idx, W)
        assert mo.check() == mz.MOSAIC_ERR_TIMEOUT
    finally:
        mo.set_wait_timeout(2_000_000_000)
    token, conf = mo.masked_sample(H, idx, W)
    assert mo.check() == mz.MOSAIC_OK
    check_against_logits(token, conf, orc.masked_logits(bits(H), idx.cpu().numpy(), bits(W)))
