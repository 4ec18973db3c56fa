"""Pins for the FP8 (E4M3) oracle, checked against facts that do not come from the oracle: an
independent library implementation of the format (torch.float8_e4m3fn), hand-worked encodings
and row quantizations (tests/golden/fp8_quantize_rows.json), exact rational arithmetic, and the
error bound of E4M3 rounding against the unquantized logits.

Cited page: the dLLM-Serve article "扩散大语言模型内存优化：从理论到系统设计", section 5
(extensions and future directions), which names FP8 quantization of the logit computation as
future work.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8_logits as f8
from oracle import mask_only_logits as orc

rng = np.random.default_rng(20261203)


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module")
def golden(golden_dir):
    return json.load(open(os.path.join(golden_dir, "fp8_quantize_rows.json")))


def test_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = f8.e4m3_bits_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    assert np.isnan(mine).sum() == 2                       # S.1111.111 only
    assert np.nanmax(mine) == 448.0 and np.nanmin(mine) == -448.0


def test_encode_matches_torch_in_range():
    x = (rng.standard_normal(300000) * np.exp(rng.uniform(-14, 6.2, 300000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    mine = f8.f64_to_e4m3_bits(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_encode_ties_go_to_even():
    vals = f8.e4m3_bits_to_f64(np.arange(0, 0x7E, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    codes = f8.f64_to_e4m3_bits(mids)
    # every midpoint lands on the neighbour with an even code (even fraction)
    assert np.all(codes % 2 == 0)
    assert np.array_equal(codes, torch.from_numpy(mids.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_encode_golden(golden):
    for e in golden["encode"]:
        assert int(f8.f64_to_e4m3_bits(np.array([e["x"]]))[0]) == e["code"], e


def test_quantize_rows_golden(golden):
    for r in golden["rows"]:
        q, s = f8.quantize_rows(bf16_bits([r["x"]]))
        assert q[0].tolist() == r["q_code"], r
        assert f8.e4m3_bits_to_f64(q[0]).tolist() == r["q_value"]
        assert s[0] == np.float32(r["absmax"]) / np.float32(448.0)


def test_quantize_rows_properties():
    x = rng.standard_normal((64, 300)).astype(np.float32) * np.exp(rng.uniform(-8, 8, (64, 1))).astype(np.float32)
    x[3] = 0.0
    xb = bf16_bits(x)
    xv = orc.bf16_bits_to_f64(xb)
    q, s = f8.quantize_rows(xb)
    dq = f8.e4m3_bits_to_f64(q)
    assert not np.any(np.isnan(dq))
    nz = s > 0
    assert not nz[3] and np.all(q[3] == 0)
    # the largest magnitude of every nonzero row maps to +-448
    assert np.all(np.max(np.abs(dq[nz]), axis=1) == 448.0)
    # E4M3 rounding: relative error <= 2^-4 in the normal range, absolute <= 2^-10 below it
    y = xv[nz] * (448.0 / np.max(np.abs(xv[nz]), axis=1, keepdims=True))
    err = np.abs(dq[nz] - y)
    bound = np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) + np.abs(y) * 2.0 ** -22
    assert np.all(err <= bound)


def test_masked_logits_fp8_exact_rationals():
    L, d, V = 9, 40, 7
    qH, sH = f8.quantize_rows(bf16_bits(rng.standard_normal((L, d))))
    qW, sW = f8.quantize_rows(bf16_bits(rng.standard_normal((V, d)) * 0.02))
    idx = np.array([4, 0, 8, 4], np.int64)
    out = f8.masked_logits_fp8(qH, sH, idx, qW, sW)
    A = f8.e4m3_bits_to_f64(qH)
    B = f8.e4m3_bits_to_f64(qW)
    for i, r in enumerate(idx):
        for v in range(V):
            exact = sum(Fraction(a) * Fraction(b) for a, b in zip(A[r].tolist(), B[v].tolist()))
            exact *= Fraction(float(sH[r])) * Fraction(float(sW[v]))
            assert abs(out[i, v] - float(exact)) <= 1e-12 * (1 + abs(float(exact)))


def test_masked_logits_fp8_within_the_quantization_bound():
    """Against the unquantized exact logits: with x = s*q + e, |e| <= 2^-4 |x| + s 2^-10, each
    product's error is below (2^-3 + 2^-8)|a||b| + 2^-10 (s_b |a| + s_a |b|) + 2^-20 s_a s_b."""
    L, d, V = 50, 256, 40
    Hb = bf16_bits(rng.standard_normal((L, d)))
    Wb = bf16_bits(rng.standard_normal((V, d)) * 0.02)
    qH, sH = f8.quantize_rows(Hb)
    qW, sW = f8.quantize_rows(Wb)
    idx = rng.integers(0, L, 30)
    out = f8.masked_logits_fp8(qH, sH, idx, qW, sW)
    ref = orc.masked_logits(Hb, idx, Wb)
    a = np.abs(orc.bf16_bits_to_f64(Hb)[idx])
    b = np.abs(orc.bf16_bits_to_f64(Wb))
    sa = sH[idx].astype(np.float64)[:, None]
    sb = sW.astype(np.float64)[None, :]
    bound = ((2.0 ** -3 + 2.0 ** -8) * (a @ b.T) + 2.0 ** -10 * (a.sum(1)[:, None] * sb + sa * b.sum(1)[None, :])
             + 2.0 ** -20 * d * sa * sb) * (1 + 1e-6)
    assert np.all(np.abs(out - ref) <= bound)
    # and the bound is not vacuous: the error is a small fraction of the logits' scale
    assert np.abs(out - ref).max() < 0.1 * np.abs(ref).max()


def test_masked_logits_fp8_csr_rows():
    qH, sH = f8.quantize_rows(bf16_bits(rng.standard_normal((10, 32))))
    qW, sW = f8.quantize_rows(bf16_bits(rng.standard_normal((8, 32))))
    so = np.array([0, 4, 10]); mo = np.array([0, 2, 3]); idx = np.array([3, 0, 5])
    out = f8.masked_logits_fp8(qH, sH, idx, qW, sW, so, mo)
    flat = f8.masked_logits_fp8(qH, sH, np.array([3, 0, 9]), qW, sW)
    assert np.array_equal(out, flat)
    with pytest.raises(IndexError):
        f8.masked_logits_fp8(qH, sH, np.array([3, 0, 6]), qW, sW, so, mo)


def test_planted_mistakes_fail_the_pins():
    """A transposed scale, a dropped scale or a truncating (not rounding) encoder is caught."""
    qH, sH = f8.quantize_rows(bf16_bits(rng.standard_normal((6, 64))))
    qW, sW = f8.quantize_rows(bf16_bits(rng.standard_normal((5, 64)) * 0.02))
    idx = np.array([1, 5, 2])
    good = f8.masked_logits_fp8(qH, sH, idx, qW, sW)
    A = f8.e4m3_bits_to_f64(qH[idx]); B = f8.e4m3_bits_to_f64(qW)
    assert not np.allclose(A @ B.T * sW[None, :], good)          # dropped H scale
    assert not np.allclose((A @ B.T) * sH[idx][:, None], good)   # dropped W scale
    x = np.array([1.0625 + 1e-9, 300.0, 0.01])
    trunc = np.array([56, 0x79, 0x05], np.uint8)                 # truncation, not rounding
    assert not np.array_equal(f8.f64_to_e4m3_bits(x), trunc)
