"""The allocation-free entry point, mosaic_masked_logits_noalloc.

It serves callers that cannot allocate device memory (a global memory planner owns the whole
workspace, or an allocation would synchronise the device), so it takes no handle and keeps its
per-chunk status words in a fixed array inside the library. These tests call it through the C
ABI and compare its logits with the handle-based mosaic_masked_logits, twice in a row (the
array keeps the previous call's contents, so the second call checks that it is cleared).
This file is collected last so a failure here does not hide the other tests' results.
"""
import ctypes

import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz
from masked_token_lm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _noalloc(H, idx, W, out, chunk_rows=0, cb=None, so=None, moff=None, status=None):
    stream = torch.cuda.current_stream().cuda_stream
    csr = so is not None
    return mz.mosaic_masked_logits_noalloc(
        H.data_ptr(), H.shape[0], H.shape[1], idx.data_ptr(), idx.numel(),
        so.data_ptr() if csr else None, moff.data_ptr() if csr else None,
        so.numel() - 1 if csr else 0, W.data_ptr(), W.shape[0], out.data_ptr(),
        mz.MOSAIC_F32 if out.dtype == torch.float32 else mz.MOSAIC_BF16, chunk_rows, cb, None,
        status, stream)


def test_noalloc_matches_handle_entry_point_twice_in_a_row():
    torch.cuda.set_device(0)
    L, d, V, M = 3000, 1024, 4104, 700
    H = wl.make_hidden(L, d, 71, DEV)
    W = wl.make_weight(V, d, 72, DEV)
    idx = wl.uniform_positions(L, M, 73).to(DEV)
    mo = mz.Mosaic(0)
    ref = mo.masked_logits(H, idx, W, out_dtype=torch.bfloat16)
    assert mo.check() == mz.MOSAIC_OK
    mo.close()
    for _ in range(2):
        out = torch.full((M, V), 7.0, dtype=torch.bfloat16, device=DEV)
        status = (ctypes.c_uint32 * 1)(0xFFFF)
        st = _noalloc(H, idx, W, out, status=status)
        assert st == mz.MOSAIC_OK, mz.mosaic_last_error_string()
        assert status[0] == 0
        # same kernel: the logits agree bit for bit (well within the 1.5e-2 bf16 tolerance)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_noalloc_chunked_status_per_chunk_and_limit():
    torch.cuda.set_device(0)
    L, d, V, M = 1200, 256, 1032, 300
    H = wl.make_hidden(L, d, 81, DEV)
    W = wl.make_weight(V, d, 82, DEV)
    idx = wl.uniform_positions(L, M, 83)
    idx[150] = L  # out of range: chunk 1 of 3 (chunk_rows 128) must report it
    idx = idx.to(DEV)
    full = torch.empty((M, V), dtype=torch.float32, device=DEV)
    out = torch.empty((128, V), dtype=torch.float32, device=DEV)

    def on_chunk(c, rb, rows, ptr, user):
        full[rb:rb + rows].copy_(out[:rows])

    cb = mz.mosaic_chunk_cb(on_chunk)
    for _ in range(2):
        status = (ctypes.c_uint32 * 3)(0, 0, 0)
        st = _noalloc(H, idx, W, out, chunk_rows=128, cb=cb, status=status)
        assert st == mz.MOSAIC_ERR_INDEX
        assert list(status) == [0, 1, 0]
        assert torch.all(full[150] == 0)
    good = idx.clone()
    good[150] = 0
    status = (ctypes.c_uint32 * 3)(9, 9, 9)
    assert _noalloc(H, good, W, out, chunk_rows=128, cb=cb, status=status) == mz.MOSAIC_OK
    assert list(status) == [0, 0, 0]  # the earlier call's words were cleared
    mo = mz.Mosaic(0)
    ref = mo.masked_logits(H, good, W, out_dtype=torch.float32)
    assert mo.check() == mz.MOSAIC_OK
    mo.close()
    assert torch.equal(full, ref)
    # more chunks than the fixed array holds: rejected before anything is enqueued
    many = torch.zeros(mz.MOSAIC_NOALLOC_MAX_CHUNKS + 1, dtype=torch.int32, device=DEV)
    st = _noalloc(H, many, W, out, chunk_rows=1, cb=cb)
    assert st == mz.MOSAIC_ERR_UNSUPPORTED
    assert "status words" in mz.mosaic_last_error_string()


def test_noalloc_csr_chunked_matches_handle_and_reports_bad_offsets():
    """A CSR batch of three sequences, one of them empty, cut into chunks that cross sequence
    boundaries: bit for bit the handle entry point's result. Then mask_offsets that do not end at
    M: the kernel's offsets check (made by the first chunk's launch) sets chunk 0's word only."""
    torch.cuda.set_device(0)
    d, V, L = 512, 1032, 500
    so = torch.tensor([0, 500, 500, 1000], dtype=torch.int32)     # sequence 1 is empty
    a = wl.uniform_positions(L, 300, 91)
    b = wl.uniform_positions(L, 250, 92)
    idx = torch.cat([a, b])
    M = idx.numel()
    moff = torch.tensor([0, 300, 300, M], dtype=torch.int32)
    H = wl.make_hidden(1000, d, 93, DEV)
    W = wl.make_weight(V, d, 94, DEV)
    idx, so, moff = idx.to(DEV), so.to(DEV), moff.to(DEV)
    mo = mz.Mosaic(0)
    ref = mo.masked_logits(H, idx, W, so, moff, out_dtype=torch.bfloat16)
    assert mo.check() == mz.MOSAIC_OK
    mo.close()
    chunk = 256
    n_chunks = (M + chunk - 1) // chunk
    full = torch.empty((M, V), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((chunk, V), dtype=torch.bfloat16, device=DEV)

    def on_chunk(c, rb, rows, ptr, user):
        full[rb:rb + rows].copy_(out[:rows])

    cb = mz.mosaic_chunk_cb(on_chunk)
    for _ in range(2):
        status = (ctypes.c_uint32 * n_chunks)(*([7] * n_chunks))
        st = _noalloc(H, idx, W, out, chunk_rows=chunk, cb=cb, so=so, moff=moff, status=status)
        assert st == mz.MOSAIC_OK, mz.mosaic_last_error_string()
        assert list(status) == [0] * n_chunks
        assert torch.equal(full.view(torch.int16), ref.view(torch.int16))
    # mask_offsets[B] = M - 1 (not M): every access stays bounded (rows are resolved through the
    # offsets and range-checked against their sequence), and the offsets check flags chunk 0
    bad = moff.clone()
    bad[-1] = M - 1
    status = (ctypes.c_uint32 * n_chunks)(*([0] * n_chunks))
    st = _noalloc(H, idx, W, out, chunk_rows=chunk, cb=cb, so=so, moff=bad, status=status)
    assert st == mz.MOSAIC_ERR_INDEX
    assert status[0] & 1 and all(w == 0 for w in list(status)[1:])
