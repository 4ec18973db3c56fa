"""Pins for the CPU oracle, checked against facts that do not come from the oracle itself:
printed worked examples, exact rational arithmetic, exact integer arithmetic, closed forms
(one-hot inputs), the IEEE format definition, library routines, and the identities the pages
state (mask-only rows == rows of the full logits; chunked == unchunked).

Cited pages: "Mosaic: Unlocking Long-Context Inference for Diffusion LLMs via Global Memory"
(paper review), section 3 observation #2 and core component 1; the dLLM-Serve article
"扩散大语言模型内存优化：从理论到系统设计", sections 2.2 and 3.2.2; the Mosaic news article
"扩散大语言模型内存优化：Mosaic系统突破与实践", section 2.3.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mask_only_logits as orc
from masked_token_lm_gb300 import workloads as wl

rng = np.random.default_rng(20261202)


def rand_bf16(shape, scale=1.0):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale)
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def exact_dot(a_bits, b_bits):
    """Exact sum_k a_k * b_k with Python Fractions (bf16 values are dyadic rationals)."""
    a = orc.bf16_bits_to_f64(a_bits)
    b = orc.bf16_bits_to_f64(b_bits)
    s = Fraction(0)
    for x, y in zip(a.tolist(), b.tolist()):
        s += Fraction(x) * Fraction(y)
    return s


# --------------------------------------------------------------------------------- bf16 format

def test_bf16_decode_known_patterns():
    bits = np.array([0x3F80, 0x4049, 0x0001, 0x7F7F, 0x8000, 0xC0A0], dtype=np.uint16)
    want = [1.0, 3.140625, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, -0.0, -5.0]
    got = orc.bf16_bits_to_f64(bits)
    assert got.tolist() == want
    assert np.signbit(got[4])


def test_bf16_rne_golden(golden_dir):
    cases = json.load(open(os.path.join(golden_dir, "bf16_rne.json")))["cases"]
    xs = np.array([float.fromhex(c["x"]) for c in cases])
    want = np.array([int(c["bits"], 16) for c in cases], dtype=np.uint16)
    got = orc.f64_to_bf16_bits(xs)
    assert got.tolist() == want.tolist(), [c["why"] for c, g, w in zip(cases, got, want) if g != w]


def test_bf16_rne_matches_torch_on_float32_values():
    # For values that are exactly fp32, RNE to bf16 must agree with torch's conversion.
    x32 = (rng.standard_normal(200_000) * np.exp(rng.uniform(-30, 30, 200_000))).astype(np.float32)
    x32 = np.concatenate([x32, np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 2 ** -130], np.float32)])
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f64_to_bf16_bits(x32.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_round_trip_is_identity():
    bits = np.arange(0, 0x7F80, 7, dtype=np.uint16)  # all finite positive patterns, sampled
    bits = np.concatenate([bits, bits | np.uint16(0x8000)])
    assert np.array_equal(orc.f64_to_bf16_bits(orc.bf16_bits_to_f64(bits)), bits)


# ------------------------------------------------------------------------ logits: exact values

def test_full_logits_against_exact_rationals():
    L, d, V = 5, 37, 6
    H, W = rand_bf16((L, d)), rand_bf16((V, d), 0.02)
    got = orc.full_logits(H, W)
    for r in range(L):
        for v in range(V):
            ex = exact_dot(H[r], W[v])
            mag = float(sum(abs(Fraction(a) * Fraction(b)) for a, b in
                            zip(orc.bf16_bits_to_f64(H[r]).tolist(), orc.bf16_bits_to_f64(W[v]).tolist())))
            # recursive fp64 summation: |err| <= d * 2^-53 * sum |a_k b_k| (first order)
            assert abs(got[r, v] - float(ex)) <= d * 2.0 ** -53 * mag * 1.01 + 1e-300


def test_naive_f32_within_recursive_summation_bound():
    L, d, V = 4, 300, 5
    H, W = rand_bf16((L, d)), rand_bf16((V, d), 0.02)
    idx = np.arange(L, dtype=np.int32)
    got = orc.masked_logits(H, idx, W, accumulate="f32")
    assert got.dtype == np.float32
    for r in range(L):
        for v in range(V):
            ex = float(exact_dot(H[r], W[v]))
            mag = float(np.sum(np.abs(orc.bf16_bits_to_f64(H[r]) * orc.bf16_bits_to_f64(W[v]))))
            assert abs(float(got[r, v]) - ex) <= d * 2.0 ** -24 * mag * 1.01


@pytest.mark.parametrize("accumulate", ["f64", "f32"])
def test_integer_valued_inputs_are_exact(accumulate):
    # H, W in {-2..2}: every partial sum is an integer of magnitude <= 4d < 2^24, so any
    # fp32/fp64 accumulation is exact; compare with exact int64 arithmetic.
    L, d, V = 40, 512, 33
    Hi = rng.integers(-2, 3, (L, d))
    Wi = rng.integers(-2, 3, (V, d))
    H = torch.from_numpy(Hi.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    W = torch.from_numpy(Wi.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    idx = rng.choice(L, 17, replace=False).astype(np.int32)
    got = orc.masked_logits(H, idx, W, accumulate=accumulate)
    exact = Hi[idx] @ Wi.T
    assert np.array_equal(got.astype(np.int64), exact)
    assert np.array_equal(got, exact.astype(got.dtype))
    # and bf16 storage of an exact integer is RNE of that integer
    assert np.array_equal(orc.round_output(got, "bf16"), orc.f64_to_bf16_bits(exact.astype(np.float64)))


@pytest.mark.parametrize("accumulate", ["f64", "f32"])
def test_one_hot_hidden_selects_weight_columns(accumulate):
    # H[r, :] = e_(r mod d)  =>  out[i, v] = W[v, row(i) mod d] exactly (one nonzero product).
    L, d, V = 70, 32, 19
    Hf = np.zeros((L, d), np.float32)
    Hf[np.arange(L), np.arange(L) % d] = 1.0
    H = torch.from_numpy(Hf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    W = rand_bf16((V, d), 0.02)
    idx = np.array([3, 69, 0, 31, 32, 33, 3, 64], dtype=np.int32)
    got = orc.masked_logits(H, idx, W, accumulate=accumulate)
    want = orc.bf16_bits_to_f64(W)[:, idx % d].T
    assert np.array_equal(got.astype(np.float64), want)


# ------------------------------------------------------------- the pages' identities / shapes

def test_mask_only_equals_rows_of_full_logits():
    L, d, V = 64, 96, 40
    H, W = rand_bf16((L, d)), rand_bf16((V, d), 0.02)
    idx = np.sort(rng.choice(L, 23, replace=False)).astype(np.int32)
    full32 = orc.masked_logits(H, np.arange(L, dtype=np.int32), W, accumulate="f32")
    assert np.array_equal(orc.masked_logits(H, idx, W, accumulate="f32"), full32[idx])
    full64 = orc.full_logits(H, W)
    np.testing.assert_allclose(orc.masked_logits(H, idx, W), full64[idx], rtol=1e-12, atol=1e-13)


def test_all_masked_equals_full_gemm():
    L, d, V = 33, 64, 24
    H, W = rand_bf16((L, d)), rand_bf16((V, d), 0.02)
    all_idx = np.arange(L, dtype=np.int32)
    np.testing.assert_allclose(orc.masked_logits(H, all_idx, W), orc.full_logits(H, W), rtol=1e-12, atol=1e-13)
    Hf, Wf = orc.bf16_bits_to_f64(H), orc.bf16_bits_to_f64(W)
    np.testing.assert_allclose(orc.masked_logits(H, all_idx, W), np.einsum("lk,vk->lv", Hf, Wf),
                               rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("accumulate", ["f64", "f32"])
def test_zero_masked_rows_give_empty_output(accumulate):
    H, W = rand_bf16((8, 16)), rand_bf16((12, 16))
    out = orc.masked_logits(H, np.zeros(0, np.int32), W, accumulate=accumulate)
    assert out.shape == (0, 12)
    assert orc.masked_logits_chunked(H, np.zeros(0, np.int32), W, chunk_rows=4).shape == (0, 12)
    assert list(orc.chunk_ranges(0, 4)) == []


@pytest.mark.parametrize("chunk_rows", [0, 1, 7, 128, 200, 205])
def test_chunked_equals_unchunked_bitwise(chunk_rows):
    L, d, V = 256, 64, 48
    H, W = rand_bf16((L, d)), rand_bf16((V, d), 0.02)
    idx = np.sort(rng.choice(L, 200, replace=False)).astype(np.int32)
    ref = orc.masked_logits(H, idx, W, accumulate="f32")
    got = orc.masked_logits_chunked(H, idx, W, chunk_rows=chunk_rows, accumulate="f32")
    assert np.array_equal(got, ref)


def test_chunk_ranges_are_lazy_and_cover_in_order():
    assert list(orc.chunk_ranges(10, 0)) == [(0, 10)]
    assert list(orc.chunk_ranges(10, 10)) == [(0, 10)]      # off when M <= chunk_rows
    assert list(orc.chunk_ranges(10, 4)) == [(0, 4), (4, 8), (8, 10)]
    assert list(orc.chunk_ranges(1, 1)) == [(0, 1)]


def test_permuted_and_duplicate_indices():
    L, d, V = 50, 40, 30
    H, W = rand_bf16((L, d)), rand_bf16((V, d), 0.02)
    idx = rng.choice(L, 20, replace=False).astype(np.int32)
    perm = rng.permutation(20)
    a = orc.masked_logits(H, idx, W, accumulate="f32")
    assert np.array_equal(orc.masked_logits(H, idx[perm], W, accumulate="f32"), a[perm])
    dup = np.array([idx[0], idx[0], idx[5], idx[0]], np.int32)
    b = orc.masked_logits(H, dup, W, accumulate="f32")
    assert np.array_equal(b[0], b[1]) and np.array_equal(b[0], b[3]) and np.array_equal(b[2], a[5])


def test_csr_golden_rows(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "csr_small.json")))
    rows = orc.resolve_rows(np.array(g["idx"]), g["L_tot"], np.array(g["seq_offsets"]), np.array(g["mask_offsets"]))
    assert rows.tolist() == g["rows"]
    for bad in g["bad_cases"]:
        with pytest.raises(IndexError):
            orc.resolve_rows(np.array(bad["idx"]), g["L_tot"], np.array(g["seq_offsets"]), np.array(g["mask_offsets"]))


def test_csr_logits_equal_flat_logits_on_resolved_rows(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "csr_small.json")))
    H, W = rand_bf16((g["L_tot"], 24)), rand_bf16((10, 24), 0.02)
    a = orc.masked_logits(H, np.array(g["idx"], np.int32), W, np.array(g["seq_offsets"]),
                          np.array(g["mask_offsets"]), accumulate="f32")
    b = orc.masked_logits(H, np.array(g["rows"], np.int32), W, accumulate="f32")
    assert np.array_equal(a, b)


def test_malformed_offsets_and_indices_raise():
    with pytest.raises(ValueError):
        orc.resolve_rows(np.array([0, 1]), 10, np.array([0, 5, 10]), None)
    with pytest.raises(ValueError):  # mask_offsets must end at M
        orc.resolve_rows(np.array([0, 1]), 10, np.array([0, 5, 10]), np.array([0, 1, 3]))
    with pytest.raises(ValueError):  # not monotone
        orc.resolve_rows(np.array([0, 1]), 10, np.array([0, 5, 10]), np.array([0, 3, 2]))
    with pytest.raises(IndexError):
        orc.resolve_rows(np.array([10]), 10)
    with pytest.raises(IndexError):
        orc.resolve_rows(np.array([-1]), 10)


def test_logit_tensor_size_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "logit_tensor_size.json")))
    full = orc.logits_bytes(g["B"] * g["L"], g["V"], g["bytes_per_element"])
    assert full == g["exact_bytes_hand_computed"]
    assert round(full / 1e9, 1) == g["printed_approx_GB"]
    blk = wl.DECODE.mask()
    assert orc.logits_bytes(blk.M, g["V"], 2) == g["mask_only_one_32_token_block_per_sequence_bytes_hand_computed"]


# -------------------------------------------------------- planted mistakes must fail the pins

def _pins_pass(fn):
    """Run three pins (integer exactness, one-hot, CSR golden rows) against a candidate."""
    L, d, V = 24, 64, 10
    Hi, Wi = rng.integers(-2, 3, (L, d)), rng.integers(-2, 3, (V, d))
    to_b = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    idx = np.array([5, 0, 23, 7], np.int32)
    ok = np.array_equal(fn(to_b(Hi), idx, to_b(Wi)), (Hi[idx] @ Wi.T).astype(np.float64))
    Hf = np.zeros((L, d)); Hf[np.arange(L), np.arange(L) % d] = 1
    ok &= np.array_equal(fn(to_b(Hf), idx, to_b(Wi)), Wi[:, idx % d].T.astype(np.float64))
    so, mo = np.array([0, 10, 24]), np.array([0, 2, 4])
    ok &= np.array_equal(fn(to_b(Hi), idx % 10, to_b(Wi), so, mo),
                         (Hi[np.array([5, 0, 13, 17])] @ Wi.T).astype(np.float64))
    return bool(ok)


def test_pins_accept_the_oracle():
    assert _pins_pass(orc.masked_logits)


def test_pins_reject_planted_mistakes():
    def dropped_last_term(H, idx, W, so=None, mo=None):
        rows = orc.resolve_rows(idx, H.shape[0], so, mo)
        A, Wf = orc.bf16_bits_to_f64(H[rows]), orc.bf16_bits_to_f64(W)
        return A[:, :-1] @ Wf[:, :-1].T

    def transposed_weight_index(H, idx, W, so=None, mo=None):
        rows = orc.resolve_rows(idx, H.shape[0], so, mo)
        A, Wf = orc.bf16_bits_to_f64(H[rows]), orc.bf16_bits_to_f64(W)
        return A @ Wf[::-1].T  # rows of W taken in the wrong order

    def csr_base_off_by_one(H, idx, W, so=None, mo=None):
        if so is not None:
            so = np.asarray(so).copy(); so[1:-1] -= 1
        return orc.masked_logits(H, idx, W, so, mo)

    def sign_flip(H, idx, W, so=None, mo=None):
        return -orc.masked_logits(H, idx, W, so, mo)

    for mutant in (dropped_last_term, transposed_weight_index, csr_base_off_by_one, sign_flip):
        assert not _pins_pass(mutant), mutant.__name__


# ------------------------------------------------------------------- the input recipe itself

def test_workload_mask_counts():
    assert wl.TINY.mask().M == 128
    assert [w.mask().M for w in wl.LLADA] == [410, 2048, 3686]
    assert wl.DECODE.mask().M == 512
    assert [wl.mask_count(w.r_m, w.L) for w in wl.LONG] == [6554, 39322, 91750, 117965]


def test_workload_masks_are_valid_and_seeded():
    for w in [wl.TINY, wl.LLADA[0], wl.DECODE]:
        m1, m2 = w.mask(), w.mask()
        assert torch.equal(m1.idx, m2.idx)
        rows = orc.resolve_rows(m1.idx.numpy(), w.L_tot,
                                None if m1.seq_offsets is None else m1.seq_offsets.numpy(),
                                None if m1.mask_offsets is None else m1.mask_offsets.numpy())
        assert len(np.unique(rows)) == len(rows)
        assert np.all(np.diff(rows) > 0)  # sorted within and across sequences
    blk = wl.DECODE.mask()
    local = blk.idx.view(16, 32)
    assert torch.all(local[:, 1:] - local[:, :-1] == 1)  # one contiguous block per sequence


def test_ragged_mask_structure():
    m = wl.ragged_mask(8, 1000, seed=5)
    assert m.mask_offsets[0] == 0 and int(m.mask_offsets[-1]) == m.M
    counts = (m.mask_offsets[1:] - m.mask_offsets[:-1]).tolist()
    assert len(set(counts)) > 1  # ragged
    rows = orc.resolve_rows(m.idx.numpy(), 8000, m.seq_offsets.numpy(), m.mask_offsets.numpy())
    assert np.all(np.diff(rows) > 0)


# ------------------------------------------------------------------ sampling the masked rows

def test_sample_closed_forms():
    # all logits equal: token 0 (first), confidence 1/V
    t, c = orc.sample_from_logits(np.zeros((3, 7)))
    assert t.tolist() == [0, 0, 0] and np.allclose(c, 1 / 7, rtol=0, atol=1e-15)
    # two-way tie at the top: the smaller index wins; confidence from the definition by hand
    z = np.array([[0.0, 2.0, -1.0, 2.0]])
    t, c = orc.sample_from_logits(z)
    assert t.tolist() == [1]
    assert abs(c[0] - 1.0 / (np.exp(-2.0) + 1 + np.exp(-3.0) + 1)) < 1e-15
    # a dominant logit: confidence tends to 1
    t, c = orc.sample_from_logits(np.array([[0.0, 50.0, 0.0]]))
    assert t.tolist() == [1] and 1 - c[0] < 1e-20
    assert orc.sample_from_logits(np.zeros((0, 5)))[0].shape == (0,)


def test_sample_confidence_matches_logsumexp_library():
    from scipy.special import logsumexp

    z = rng.standard_normal((50, 300)) * 3
    t, c = orc.sample_from_logits(z)
    assert np.array_equal(t, np.argmax(z, axis=1))
    np.testing.assert_allclose(np.log(c), z.max(axis=1) - logsumexp(z, axis=1), rtol=0, atol=1e-12)


def test_sample_integer_inputs_exact_argmax():
    L, d, V = 30, 256, 77
    Hi, Wi = rng.integers(-2, 3, (L, d)), rng.integers(-2, 3, (V, d))
    to_b = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    idx = np.array([3, 0, 29, 3, 11], np.int32)
    t, c = orc.masked_sample(to_b(Hi), idx, to_b(Wi))
    exact = Hi[idx] @ Wi.T
    first = np.array([int(np.flatnonzero(row == row.max())[0]) for row in exact])
    assert np.array_equal(t, first)
    want = np.array([1.0 / sum(np.exp(float(v - row.max())) for v in row) for row in exact])
    np.testing.assert_allclose(c, want, rtol=1e-14)


def test_sample_one_hot_picks_the_weight_column_maximum():
    L, d, V = 40, 32, 50
    Hf = np.zeros((L, d)); Hf[np.arange(L), np.arange(L) % d] = 1
    H = torch.from_numpy(Hf.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    W = rand_bf16((V, d), 0.02)
    idx = np.array([0, 5, 33, 39], np.int32)
    t, _ = orc.masked_sample(H, idx, W)
    Wf = orc.bf16_bits_to_f64(W)
    assert t.tolist() == [int(np.argmax(Wf[:, r % d])) for r in idx]
