"""GPU parity of the FP8 (E4M3) variant against the CPU oracle.

* mosaic_quantize_rows_e4m3 must equal the oracle's per-row quantization bit for bit (codes and
  scales: every step is a single IEEE fp32 operation or a round-to-nearest-even conversion).
* mosaic_masked_logits_fp8 must match the oracle's logits from the same quantized operands
  (exact products, fp64 sums, the two scales) within the bf16 / fp32 output tolerance of the bf16
  path; on inputs whose fp32 accumulation is exact the fp32 output must match bit for bit.
* Chunked calls equal the unchunked call bit for bit.
"""
import numpy as np
import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz
from masked_token_lm_gb300 import workloads as wl
from oracle import fp8_logits as f8
from tests.parity_utils import TOL, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def mo():
    m = mz.Mosaic(0)
    yield m
    m.close()


def quantize(x):
    q, s = mz.quantize_rows_e4m3(x)
    torch.cuda.synchronize()
    return q, s


def assert_close(out, ref, dt, what):
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref) / (1 + np.abs(ref))
    assert err.max() <= TOL[dt], f"{what}: max scaled error {err.max():.3g}"


@pytest.mark.parametrize("rows,d,scale", [(1, 16, 1.0), (37, 64, 1.0), (300, 4096, 0.02),
                                          (64, 144, 1000.0), (5, 32, 1e-30)])
def test_quantize_rows_is_bitwise_the_oracle(rows, d, scale):
    g = torch.Generator().manual_seed(rows * 7 + d)
    x = (torch.randn(rows, d, generator=g) * scale).to(torch.bfloat16)
    x[0, : d // 2] = 0.0
    if rows > 3:
        x[3] = 0.0                                   # a zero row: scale 0, codes 0
    q, s = quantize(x.to(DEV))
    q_ref, s_ref = f8.quantize_rows(bits(x))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("L,d,V,M,dt", [
    (1000, 512, 1000, 300, torch.bfloat16),   # 3 M tiles, N tail of 232 columns
    (1000, 512, 1000, 300, torch.float32),
    (777, 144, 520, 129, torch.bfloat16),     # K tail (144 = 128 + 16), M tail of one row
    (300, 128, 256, 100, torch.bfloat16),     # one M tile: single CTA, one K block
    (300, 272, 264, 100, torch.float32),      # single CTA, fp32 out, K tail, N tail of 8 columns
    (600, 256, 520, 300, torch.bfloat16),     # one-panel unit column, split last round
    (2000, 1024, 8200, 700, torch.bfloat16),  # many units, persistent loop
])
def test_fp8_logits_match_the_oracle(mo, L, d, V, M, dt):
    H = wl.make_hidden(L, d, 100 + L, DEV)
    W = wl.make_weight(V, d, 101 + V, DEV)
    idx = wl.uniform_positions(L, M, seed=M + 1)
    qH, sH = quantize(H)
    qW, sW = quantize(W)
    out = mo.masked_logits_fp8(qH, sH, idx.to(DEV), qW, sW, out_dtype=dt)
    assert mo.check() == mz.MOSAIC_OK
    ref = f8.masked_logits_fp8(qH.cpu().numpy(), sH.cpu().numpy(), idx.numpy(),
                               qW.cpu().numpy(), sW.cpu().numpy())
    assert_close(out, ref, dt, f"L={L} d={d} V={V} M={M}")


def test_fp8_exact_inputs_are_bit_exact(mo):
    """Rows holding one +-448 get scale exactly 1 and keep their (E4M3-exact) integer values, and
    every partial sum stays below 2^24: fp32 accumulation is exact, so the output is the oracle's
    value bit for bit."""
    L, d, V, M = 200, 32, 264, 150
    g = torch.Generator().manual_seed(5)
    def ints(rows):
        x = torch.randint(-16, 17, (rows, d), generator=g).float()
        x[torch.arange(rows), torch.randint(0, d, (rows,), generator=g)] = 448.0
        return x.to(torch.bfloat16)
    H, W = ints(L), ints(V)
    idx = torch.randint(0, L, (M,), generator=g, dtype=torch.int32)
    qH, sH = quantize(H.to(DEV))
    qW, sW = quantize(W.to(DEV))
    assert torch.all(sH == 1.0) and torch.all(sW == 1.0)
    out = mo.masked_logits_fp8(qH, sH, idx.to(DEV), qW, sW, out_dtype=torch.float32)
    ref = f8.masked_logits_fp8(qH.cpu().numpy(), sH.cpu().numpy(), idx.numpy(),
                               qW.cpu().numpy(), sW.cpu().numpy())
    assert np.array_equal(out.cpu().numpy(), ref.astype(np.float32))


def test_fp8_csr_and_bad_index(mo):
    m = wl.ragged_mask(4, 300, seed=9)
    d, V = 256, 1032
    H = wl.make_hidden(1200, d, 3, DEV)
    W = wl.make_weight(V, d, 4, DEV)
    qH, sH = quantize(H)
    qW, sW = quantize(W)
    out = mo.masked_logits_fp8(qH, sH, m.idx.to(DEV), qW, sW, m.seq_offsets.to(DEV),
                               m.mask_offsets.to(DEV))
    assert mo.check() == mz.MOSAIC_OK
    ref = f8.masked_logits_fp8(qH.cpu().numpy(), sH.cpu().numpy(), m.idx.numpy(), qW.cpu().numpy(),
                               sW.cpu().numpy(), m.seq_offsets.numpy(), m.mask_offsets.numpy())
    assert_close(out, ref, torch.bfloat16, "CSR")
    bad = m.idx.clone()
    bad[2] = 10 ** 6
    out = mo.masked_logits_fp8(qH, sH, bad.to(DEV), qW, sW, m.seq_offsets.to(DEV),
                               m.mask_offsets.to(DEV))
    assert mo.check() == mz.MOSAIC_ERR_INDEX
    assert torch.all(out[2] == 0)


@pytest.mark.parametrize("chunk_rows", [1, 100, 256])
def test_fp8_chunked_equals_unchunked_bitwise(mo, chunk_rows):
    L, d, V, M = 900, 256, 776, 513
    H = wl.make_hidden(L, d, 21, DEV)
    W = wl.make_weight(V, d, 22, DEV)
    idx = wl.uniform_positions(L, M, seed=23).to(DEV)
    qH, sH = quantize(H)
    qW, sW = quantize(W)
    full = mo.masked_logits_fp8(qH, sH, idx, qW, sW)
    got = torch.empty_like(full)

    def on_chunk(c, rb, rows, out):
        got[rb:rb + rows].copy_(out[:rows])

    mo.masked_logits_fp8(qH, sH, idx, qW, sW, chunk_rows=chunk_rows, on_chunk=on_chunk)
    torch.cuda.synchronize()
    assert torch.equal(got, full)


@pytest.mark.parametrize("csr", [False, True])
def test_quantize_masked_rows_touches_only_the_masked_rows(csr):
    d = 256
    if csr:
        m = wl.ragged_mask(5, 200, seed=4)
        L = int(m.seq_offsets[-1])
        idx, so, mo_ = m.idx, m.seq_offsets, m.mask_offsets
        rows = np.concatenate([
            so[b].item() + idx[mo_[b]:mo_[b + 1]].numpy() for b in range(5)])
    else:
        L = 700
        g = torch.Generator().manual_seed(8)
        idx = torch.randint(0, L, (300,), generator=g, dtype=torch.int32)  # with duplicates
        idx[7] = 10 ** 6                                                   # out of range: skipped
        so = mo_ = None
        rows = idx.numpy()[idx.numpy() < L]
    H = wl.make_hidden(L, d, 12, DEV)
    q = torch.full((L, d), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((L,), -1.0, dtype=torch.float32, device=DEV)
    mz.quantize_masked_rows_e4m3(H, idx.to(DEV), q, s, so.to(DEV) if csr else None,
                                 mo_.to(DEV) if csr else None)
    torch.cuda.synchronize()
    q_ref, s_ref = f8.quantize_rows(bits(H.cpu()))
    qc, sc = q.cpu().numpy(), s.cpu().numpy()
    touched = np.zeros(L, bool)
    touched[rows] = True
    assert np.array_equal(qc[touched], q_ref[touched])
    assert np.array_equal(sc[touched].view(np.uint32), s_ref[touched].view(np.uint32))
    assert np.all(qc[~touched] == 0xAB) and np.all(sc[~touched] == -1.0)


def test_fp8_argument_errors():
    x = torch.zeros((4, 24), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mz.MosaicError):
        mz.quantize_rows_e4m3(x)                      # d % 16 != 0


@pytest.mark.parametrize("csr", [False, True])
def test_fp8_whole_chain_against_the_oracle_from_bf16_inputs(mo, csr):
    """The expected side is all oracle: it quantizes the bf16 inputs itself (rows of H and W)
    and computes the quantized logits; the GPU side runs its own quantization kernels and the
    FP8 logits. No GPU-produced value enters the expected side."""
    d, V = 512, 1544
    if csr:
        m = wl.ragged_mask(3, 400, seed=31)
        L = 1200
        so, mo_ = m.seq_offsets, m.mask_offsets
        idx = m.idx
    else:
        L = 900
        idx = wl.uniform_positions(L, 333, seed=32)
        so = mo_ = None
    H = wl.make_hidden(L, d, 33, DEV)
    W = wl.make_weight(V, d, 34, DEV)
    # oracle: quantize from the bf16 bit patterns, then the FP8 logits
    qH_ref, sH_ref = f8.quantize_rows(bits(H))
    qW_ref, sW_ref = f8.quantize_rows(bits(W))
    ref = f8.masked_logits_fp8(qH_ref, sH_ref, idx.numpy(), qW_ref, sW_ref,
                               None if so is None else so.numpy(),
                               None if mo_ is None else mo_.numpy())
    # GPU: W quantized once, the masked hidden rows quantized, then the fused FP8 logits
    qW, sW = mz.quantize_rows_e4m3(W)
    qH = torch.zeros((L, d), dtype=torch.uint8, device=DEV)
    sH = torch.zeros((L,), dtype=torch.float32, device=DEV)
    dev = lambda t: None if t is None else t.to(DEV)  # noqa: E731
    mz.quantize_masked_rows_e4m3(H, idx.to(DEV), qH, sH, dev(so), dev(mo_))
    for dt in (torch.bfloat16, torch.float32):
        out = mo.masked_logits_fp8(qH, sH, idx.to(DEV), qW, sW, dev(so), dev(mo_), out_dtype=dt)
        assert mo.check() == mz.MOSAIC_OK
        assert_close(out, ref, dt, f"whole FP8 chain, csr={csr}, {dt}")
