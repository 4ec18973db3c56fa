"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle, at sizes the oracle
checks in full: several tiles in M, N and K with ragged tails, CSR batches, exact pins
(one-hot, integer-valued inputs), lazy chunking, and the error paths."""
import numpy as np
import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz
from masked_token_lm_gb300 import workloads as wl
from oracle import mask_only_logits as orc
from tests.parity_utils import as_f64, assert_close, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def mo():
    m = mz.Mosaic(0)
    yield m
    m.close()


def run(mo, H, idx, W, out_dtype, so=None, moff=None, chunk_rows=0):
    """Call through the C ABI and return the full [M, V] result (chunks gathered on-stream)."""
    M, V = int(idx.numel()), int(W.shape[0])
    if 0 < chunk_rows < M:
        result = torch.empty((M, V), dtype=out_dtype, device=DEV)
        seen = []

        def on_chunk(c, rb, rows, out):
            seen.append((c, rb, rows))
            result[rb:rb + rows].copy_(out[:rows])

        mo.masked_logits(H, idx, W, so, moff, out_dtype=out_dtype, chunk_rows=chunk_rows,
                         on_chunk=on_chunk)
        assert [s[1:] for s in seen] == [(b, e - b) for b, e in orc.chunk_ranges(M, chunk_rows)]
        out = result
    else:
        out = mo.masked_logits(H, idx, W, so, moff, out_dtype=out_dtype)
    assert mo.check() == mz.MOSAIC_OK, mz.mosaic_last_error_string()
    return out


def rand_inputs(L, d, V, seed):
    return (wl.make_hidden(L, d, seed, DEV), wl.make_weight(V, d, seed + 1, DEV))


def test_tiny_config_full_parity(mo):
    w = wl.TINY
    H, W, mask = w.hidden(DEV), w.weight(DEV), w.mask()
    out = run(mo, H, mask.idx.to(DEV), W, torch.float32)
    ref = orc.masked_logits(bits(H), mask.idx.numpy(), bits(W))
    assert_close(out, ref, torch.float32, "tiny")
    # lazy chunking on the same workload: 128 one-row launches, 19 launches of 7 rows, and
    # chunk_rows = M (chunking stays off); each equals the unchunked call bit for bit
    for chunk_rows in (1, 7, 128):
        before = mo.launches
        ch = run(mo, H, mask.idx.to(DEV), W, torch.float32, chunk_rows=chunk_rows)
        assert mo.launches - before == -(-mask.M // chunk_rows)
        assert torch.equal(ch.view(torch.int32), out.view(torch.int32)), chunk_rows


@pytest.mark.parametrize("L,d,V,M,dt", [
    (1000, 512, 1000, 300, torch.float32),   # 3 M tiles (last 44 rows), 4 N tiles (last 232 cols)
    (1000, 512, 1000, 300, torch.bfloat16),
    (777, 200, 520, 129, torch.bfloat16),    # K tail (200 = 3*64 + 8), M tail of 1 row
    (4096, 4096, 2048, 1, torch.bfloat16),   # a single masked row
    (300, 64, 256, 257, torch.float32),      # one K block, exact N tile
    (2000, 1024, 8200, 700, torch.bfloat16), # many tiles: 6 x 33, persistent loop > 1 tile/CTA
    # Schedule paths of the 256 x 512 pair units (76 pairs resident on a GB300):
    (600, 256, 520, 300, torch.bfloat16),    # 3 panels: a one-panel unit column; 4 units, all
                                             # split into halves, one half empty (skipped)
    (2000, 256, 15104, 700, torch.bfloat16), # 3 x 30 units = 76 + 14: split last round, odd panels
    (1500, 64, 16384, 1024, torch.bfloat16), # one K block (fewer than the stages) over 2 rounds
    (1500, 128, 16384, 1024, torch.float32), # two K blocks, fp32 out
])
def test_ragged_tiles_full_parity(mo, L, d, V, M, dt):
    H, W = rand_inputs(L, d, V, seed=L + d + V + M)
    idx = wl.uniform_positions(L, M, seed=M)
    out = run(mo, H, idx.to(DEV), W, dt)
    ref = orc.masked_logits(bits(H), idx.numpy(), bits(W))
    assert_close(out, ref, dt, f"L={L} d={d} V={V} M={M}")


def test_unsorted_and_duplicate_indices(mo):
    L, d, V = 500, 256, 512
    H, W = rand_inputs(L, d, V, seed=3)
    g = torch.Generator().manual_seed(9)
    idx = torch.randint(0, L, (333,), generator=g, dtype=torch.int32)  # unsorted, duplicates
    out = run(mo, H, idx.to(DEV), W, torch.float32)
    ref = orc.masked_logits(bits(H), idx.numpy(), bits(W))
    assert_close(out, ref, torch.float32, "unsorted/duplicates")
    dup = (idx[:, None] == idx[None, :]).nonzero()
    o = out.cpu()
    assert all(torch.equal(o[i], o[j]) for i, j in dup.tolist()[:200])


def test_csr_golden_example_on_gpu(mo, golden_dir):
    import json, os
    gd = json.load(open(os.path.join(golden_dir, "csr_small.json")))
    d, V = 64, 256
    H, W = rand_inputs(gd["L_tot"], d, V, seed=11)
    t = lambda a: torch.tensor(a, dtype=torch.int32, device=DEV)
    out = run(mo, H, t(gd["idx"]), W, torch.float32, t(gd["seq_offsets"]), t(gd["mask_offsets"]))
    flat = run(mo, H, t(gd["rows"]), W, torch.float32)
    assert torch.equal(out, flat)  # index handling is bit-exact
    ref = orc.masked_logits(bits(H), np.array(gd["idx"]), bits(W), np.array(gd["seq_offsets"]),
                            np.array(gd["mask_offsets"]))
    assert_close(out, ref, torch.float32, "csr golden")


def test_csr_ragged_with_empty_sequences(mo):
    counts, Ls = [3, 0, 130, 0, 1, 200], [10, 7, 300, 5, 2, 999]
    so = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    moff = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    g = np.random.default_rng(4)
    idx = np.concatenate([np.sort(g.choice(L, c, replace=False)) for L, c in zip(Ls, counts)]).astype(np.int32)
    d, V = 192, 776
    H, W = rand_inputs(int(so[-1]), d, V, seed=5)
    t = lambda a: torch.from_numpy(a).to(DEV)
    out = run(mo, H, t(idx), W, torch.bfloat16, t(so), t(moff))
    ref = orc.masked_logits(bits(H), idx, bits(W), so, moff)
    assert_close(out, ref, torch.bfloat16, "csr ragged")


def test_csr_many_sequences_offsets_from_global_memory(mo):
    # B = 200 > 128: the kernel searches the offsets in global memory instead of shared memory
    g = np.random.default_rng(12)
    B = 200
    Ls = g.integers(1, 40, B)
    counts = np.minimum(Ls, g.integers(0, 6, B))
    counts[::17] = 0  # some empty sequences
    so = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    moff = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    idx = np.concatenate([np.sort(g.choice(L, c, replace=False)) for L, c in zip(Ls, counts)]).astype(np.int32)
    d, V = 128, 520
    H, W = rand_inputs(int(so[-1]), d, V, seed=13)
    t = lambda a: torch.from_numpy(a).to(DEV)
    out = run(mo, H, t(idx), W, torch.float32, t(so), t(moff))
    ref = orc.masked_logits(bits(H), idx, bits(W), so, moff)
    assert_close(out, ref, torch.float32, "csr B=200")
    flat = run(mo, H, t(orc.resolve_rows(idx, int(so[-1]), so, moff).astype(np.int32)), W, torch.float32)
    assert torch.equal(out, flat)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_one_hot_hidden_is_bit_exact(mo, dt):
    # H[r, :] = e_(r mod d): out[i, v] = W[v, row(i) mod d] exactly, in any dtype.
    L, d, V, M = 900, 128, 1032, 333
    Hf = torch.zeros((L, d))
    Hf[torch.arange(L), torch.arange(L) % d] = 1.0
    H = Hf.to(torch.bfloat16).to(DEV)
    W = wl.make_weight(V, d, 21, DEV)
    idx = torch.randint(0, L, (M,), generator=torch.Generator().manual_seed(2), dtype=torch.int32)
    out = run(mo, H, idx.to(DEV), W, dt)
    want = orc.bf16_bits_to_f64(bits(W))[:, idx.numpy() % d].T
    assert np.array_equal(as_f64(out), want)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_integer_valued_inputs_are_bit_exact(mo, dt):
    # H, W in {-2..2}: fp32 accumulation is exact in any order; bf16 out = RNE(exact).
    L, d, V, M = 600, 512, 1000, 257
    g = torch.Generator().manual_seed(8)
    Hi = torch.randint(-2, 3, (L, d), generator=g)
    Wi = torch.randint(-2, 3, (V, d), generator=g)
    H, W = Hi.to(torch.bfloat16).to(DEV), Wi.to(torch.bfloat16).to(DEV)
    idx = wl.uniform_positions(L, M, seed=6)
    out = run(mo, H, idx.to(DEV), W, dt)
    exact = (Hi[idx.long()].long() @ Wi.long().T).numpy()
    if dt == torch.float32:
        assert np.array_equal(as_f64(out), exact.astype(np.float64))
    else:
        assert np.array_equal(bits(out), orc.f64_to_bf16_bits(exact.astype(np.float64)))


@pytest.mark.parametrize("chunk_rows", [1, 7, 128, 129, 299, 300, 1000])
def test_chunked_equals_unchunked_bitwise(mo, chunk_rows):
    L, d, V, M = 1200, 320, 1288, 300
    H, W = rand_inputs(L, d, V, seed=17)
    idx = wl.uniform_positions(L, M, seed=18).to(DEV)
    full = run(mo, H, idx, W, torch.bfloat16)
    chunked = run(mo, H, idx, W, torch.bfloat16, chunk_rows=chunk_rows)
    assert torch.equal(full.view(torch.int16), chunked.view(torch.int16))


def test_chunked_csr_crosses_sequence_boundaries(mo):
    m = wl.ragged_mask(4, 400, seed=3)
    d, V = 128, 512
    H, W = rand_inputs(1600, d, V, seed=23)
    mm = m.to(DEV)
    full = run(mo, H, mm.idx, W, torch.float32, mm.seq_offsets, mm.mask_offsets)
    ch = run(mo, H, mm.idx, W, torch.float32, mm.seq_offsets, mm.mask_offsets, chunk_rows=100)
    assert torch.equal(full, ch)
    ref = orc.masked_logits(bits(H), m.idx.numpy(), bits(W), m.seq_offsets.numpy(), m.mask_offsets.numpy())
    assert_close(ch, ref, torch.float32, "chunked csr")


def test_zero_masked_rows_launch_nothing(mo):
    H, W = rand_inputs(64, 64, 256, seed=1)
    calls = []
    before = mo.launches
    out = mo.masked_logits(H, torch.zeros(0, dtype=torch.int32, device=DEV), W,
                           out_dtype=torch.float32, chunk_rows=8, on_chunk=lambda *a: calls.append(a))
    assert out.shape == (0, 256) and calls == [] and mo.launches == before
    assert mo.check() == mz.MOSAIC_OK


def test_out_of_range_index_sets_status_and_zero_fills_row(mo):
    L, d, V = 300, 128, 512
    H, W = rand_inputs(L, d, V, seed=31)
    idx = torch.tensor([5, L, 7, -1, 299], dtype=torch.int32)
    out = mo.masked_logits(H, idx.to(DEV), W, out_dtype=torch.float32)
    assert mo.check() == mz.MOSAIC_ERR_INDEX
    o = out.cpu()
    assert torch.all(o[1] == 0) and torch.all(o[3] == 0)
    good = np.array([0, 2, 4])
    ref = orc.masked_logits(bits(H), idx.numpy()[good], bits(W))
    assert_close(out[good.tolist()], ref, torch.float32, "valid rows next to bad ones")
    assert mo.check() == mz.MOSAIC_OK  # the status word was cleared


@pytest.mark.parametrize("chunk_rows", [0, 200])
def test_bad_indices_in_both_pair_tiles_bf16(mo, chunk_rows):
    """The CTA-pair kernel with bf16 output (both accumulator slots read before any store):
    bad rows in the first and in the ragged second M tile, next to a bad row in the last chunk,
    come out as zeros with the status set; every other row matches the oracle."""
    L, d, V = 700, 256, 1032
    H, W = rand_inputs(L, d, V, seed=41)
    rng = np.random.default_rng(41)
    idx = rng.integers(0, L, size=300).astype(np.int32)
    bad = [3, 130, 257, 299]  # CTA 0 / CTA 1 of tile 0, tile 1 (44 valid rows), the last row
    idx[bad] = [L, -5, L + 1000, 2 ** 30]
    idx_t = torch.from_numpy(idx).to(DEV)
    if chunk_rows:
        result = torch.empty((300, V), dtype=torch.bfloat16, device=DEV)

        def on_chunk(c, rb, rows, out):
            result[rb:rb + rows].copy_(out[:rows])

        mo.masked_logits(H, idx_t, W, chunk_rows=chunk_rows, on_chunk=on_chunk)
        out = result
    else:
        out = mo.masked_logits(H, idx_t, W)
    assert mo.check() == mz.MOSAIC_ERR_INDEX
    o = out.cpu()
    for r in bad:
        assert torch.all(o[r].view(torch.int16) == 0), r
    good = np.setdiff1d(np.arange(300), bad)
    ref = orc.masked_logits(bits(H), idx[good], bits(W))
    assert_close(out[torch.from_numpy(good).to(DEV)], ref, torch.bfloat16, "valid rows next to bad ones")
    assert mo.check() == mz.MOSAIC_OK


def test_csr_local_index_past_its_sequence_is_flagged(mo):
    d, V = 64, 256
    H, W = rand_inputs(16, d, V, seed=2)
    t = lambda a: torch.tensor(a, dtype=torch.int32, device=DEV)
    out = mo.masked_logits(H, t([5, 0, 6, 1, 3]), W, t([0, 5, 9, 16]), t([0, 2, 2, 5]),
                           out_dtype=torch.float32)
    assert mo.check() == mz.MOSAIC_ERR_INDEX
    assert torch.all(out[0] == 0) and not torch.all(out[1] == 0)


def test_csr_offsets_not_ending_at_M_are_flagged(mo):
    d, V = 64, 256
    H, W = rand_inputs(16, d, V, seed=2)
    t = lambda a: torch.tensor(a, dtype=torch.int32, device=DEV)
    mo.masked_logits(H, t([4, 0, 6, 1, 3]), W, t([0, 5, 9, 16]), t([0, 2, 2, 4]), out_dtype=torch.float32)
    assert mo.check() == mz.MOSAIC_ERR_INDEX


def test_argument_errors_enqueue_nothing(mo):
    H, W = rand_inputs(64, 64, 256, seed=1)
    idx = torch.arange(8, dtype=torch.int32, device=DEV)
    out = torch.empty((8, 256), dtype=torch.bfloat16, device=DEV)
    before = mo.launches
    s = torch.cuda.current_stream().cuda_stream
    call = lambda **kw: mz.mosaic_masked_logits(**{**dict(
        handle=mo.handle, hidden=H.data_ptr(), L_tot=64, d=64, mask_idx=idx.data_ptr(), M=8,
        seq_offsets=None, mask_offsets=None, B=0, W=W.data_ptr(), V=256, out=out.data_ptr(),
        out_dtype=mz.MOSAIC_BF16, chunk_rows=0, cb=None, user=None, stream=s), **kw})
    assert call() == mz.MOSAIC_OK
    assert mo.check() == mz.MOSAIC_OK
    before = mo.launches
    assert call(d=60) == mz.MOSAIC_ERR_UNSUPPORTED              # 120-byte rows
    assert call(V=250) == mz.MOSAIC_ERR_UNSUPPORTED
    assert call(hidden=H.data_ptr() + 2) == mz.MOSAIC_ERR_INVALID_ARG  # misaligned
    assert call(out=None) == mz.MOSAIC_ERR_INVALID_ARG
    assert call(M=-1) == mz.MOSAIC_ERR_INVALID_ARG
    assert call(out_dtype=7) == mz.MOSAIC_ERR_INVALID_ARG
    assert call(seq_offsets=idx.data_ptr()) == mz.MOSAIC_ERR_INVALID_ARG   # half a CSR pair
    assert call(chunk_rows=3) == mz.MOSAIC_ERR_INVALID_ARG        # chunking without a callback
    host = torch.empty((8, 256), dtype=torch.bfloat16)
    assert call(out=host.data_ptr()) == mz.MOSAIC_ERR_INVALID_ARG  # not device memory
    assert mo.launches == before


def test_bounded_wait_timeout_reports_and_context_survives(mo):
    L, d, V, M = 2048, 4096, 32768, 1024
    H, W = rand_inputs(L, d, V, seed=41)
    idx = wl.uniform_positions(L, M, seed=42).to(DEV)
    mo.set_wait_timeout(0)  # every wait that is not already satisfied gives up at once
    try:
        mo.masked_logits(H, idx, W, out_dtype=torch.bfloat16)
        assert mo.check() == mz.MOSAIC_ERR_TIMEOUT
    finally:
        mo.set_wait_timeout(2_000_000_000)
    out = run(mo, H[:256], idx[:100] % 256, W[:1024], torch.float32)
    ref = orc.masked_logits(bits(H[:256]), (idx[:100] % 256).cpu().numpy(), bits(W[:1024]))
    assert_close(out, ref, torch.float32, "after timeout")
    # the CTA-pair kernel with bf16 output (the one whose warpgroups trade registers) runs again
    sub = idx[:300] % 256
    out = run(mo, H[:256], sub, W[:1024], torch.bfloat16)
    ref = orc.masked_logits(bits(H[:256]), sub.cpu().numpy(), bits(W[:1024]))
    assert_close(out, ref, torch.bfloat16, "pair kernel after timeout")


def test_min_chunk_rows_drives_a_chunked_call_within_budget(mo):
    # lazy chunking with the minimum sufficient chunk count for a 250-row output budget
    L, d, V, M = 2000, 256, 1032, 900
    H, W = rand_inputs(L, d, V, seed=51)
    idx = wl.uniform_positions(L, M, seed=52).to(DEV)
    st, cr, nc = mz.mosaic_min_chunk_rows(M, V, mz.MOSAIC_BF16, 250 * V * 2 + 100)
    assert (st, cr, nc) == (mz.MOSAIC_OK, 225, 4)
    full = run(mo, H, idx, W, torch.bfloat16)
    chunked = run(mo, H, idx, W, torch.bfloat16, chunk_rows=cr)
    assert torch.equal(full.view(torch.int16), chunked.view(torch.int16))


@pytest.mark.parametrize("L,d,V,M,dt", [
    (1, 8, 8, 1, torch.float32),        # smallest shape: one row, one 16-byte K piece, 8 columns
    (50, 8, 8, 300, torch.float32),     # K far below one block, CTA pairs, duplicates
    (512, 8192, 1024, 200, torch.bfloat16),  # 128 K blocks
    (64, 24, 264, 130, torch.float32),  # K tail only (24 = 3 pieces), N tail of 8 columns
])
def test_extreme_shapes(mo, L, d, V, M, dt):
    H, W = rand_inputs(L, d, V, seed=L * 7 + d + V)
    g = torch.Generator().manual_seed(M)
    idx = torch.randint(0, L, (M,), generator=g, dtype=torch.int32)
    out = run(mo, H, idx.to(DEV), W, dt)
    ref = orc.masked_logits(bits(H), idx.numpy(), bits(W))
    assert_close(out, ref, dt, f"L={L} d={d} V={V} M={M}")


def test_all_positions_masked_equals_the_full_gemm(mo):
    L, d, V = 700, 256, 1288
    H, W = rand_inputs(L, d, V, seed=91)
    out = run(mo, H, torch.arange(L, dtype=torch.int32, device=DEV), W, torch.float32)
    assert_close(out, orc.full_logits(bits(H), bits(W)), torch.float32, "all masked")


def test_csr_duplicates_and_unsorted_local_indices(mo):
    so = np.array([0, 100, 180, 400], np.int32)
    moff = np.array([0, 5, 5, 12], np.int32)
    idx = np.array([99, 3, 3, 50, 0, 219, 0, 7, 7, 100, 219, 1], np.int32)
    d, V = 96, 776
    H, W = rand_inputs(400, d, V, seed=93)
    t = lambda a: torch.from_numpy(a).to(DEV)
    out = run(mo, H, t(idx), W, torch.float32, t(so), t(moff))
    ref = orc.masked_logits(bits(H), idx, bits(W), so, moff)
    assert_close(out, ref, torch.float32, "csr duplicates")
    assert torch.equal(out[1], out[2]) and torch.equal(out[5], out[10])


def test_fp32_output_chunked_pairs_bitwise(mo):
    L, d, V, M = 1500, 384, 2056, 700
    H, W = rand_inputs(L, d, V, seed=95)
    idx = wl.uniform_positions(L, M, seed=96).to(DEV)
    full = run(mo, H, idx, W, torch.float32)
    for cr in (129, 256, 500):
        assert torch.equal(full, run(mo, H, idx, W, torch.float32, chunk_rows=cr))
