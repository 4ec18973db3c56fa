"""Python binding of libmosaic.so (ctypes). Argument marshalling only: every step of the
mask-only logits path runs in the library's CUDA kernels.

The ``mosaic_*`` functions mirror the C ABI in ``include/mosaic.h`` one to one (raw pointers,
integer status). ``Mosaic`` is a small convenience wrapper that takes torch tensors (torch is
used for device memory and streams only) and raises ``MosaicError`` on a non-OK status.

There is no CPU fallback: if the library is missing or no sm_103 GPU is present, the calls
fail loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Callable, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libmosaic.so")

MOSAIC_OK = 0
MOSAIC_ERR_INVALID_ARG = 1
MOSAIC_ERR_UNSUPPORTED = 2
MOSAIC_ERR_CUDA = 3
MOSAIC_ERR_INDEX = 4
MOSAIC_ERR_TIMEOUT = 5
STATUS_NAMES = {0: "MOSAIC_OK", 1: "MOSAIC_ERR_INVALID_ARG", 2: "MOSAIC_ERR_UNSUPPORTED",
                3: "MOSAIC_ERR_CUDA", 4: "MOSAIC_ERR_INDEX", 5: "MOSAIC_ERR_TIMEOUT"}

MOSAIC_BF16 = 0
MOSAIC_F32 = 1
MOSAIC_NOALLOC_MAX_CHUNKS = 4096

mosaic_chunk_cb = ctypes.CFUNCTYPE(None, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_void_p, ctypes.c_void_p)

_lib = None


class MosaicError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmosaic.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m masked_token_lm_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.mosaic_create.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
    lib.mosaic_create.restype = ctypes.c_int
    lib.mosaic_destroy.argtypes = [P]
    lib.mosaic_destroy.restype = ctypes.c_int
    lib.mosaic_masked_logits.argtypes = [P, P, I64, I64, P, I64, P, P, I32, P, I64, P,
                                         ctypes.c_int, I64, mosaic_chunk_cb, P, P]
    lib.mosaic_masked_logits.restype = ctypes.c_int
    lib.mosaic_check.argtypes = [P, P]
    lib.mosaic_check.restype = ctypes.c_int
    lib.mosaic_set_wait_timeout.argtypes = [P, ctypes.c_uint64]
    lib.mosaic_set_wait_timeout.restype = ctypes.c_int
    lib.mosaic_launch_count.argtypes = [P]
    lib.mosaic_launch_count.restype = ctypes.c_int64
    lib.mosaic_last_error_string.argtypes = []
    lib.mosaic_last_error_string.restype = ctypes.c_char_p
    lib.mosaic_masked_logits_noalloc.argtypes = [P, I64, I64, P, I64, P, P, I32, P, I64, P,
                                                 ctypes.c_int, I64, mosaic_chunk_cb, P,
                                                 ctypes.POINTER(ctypes.c_uint32), P]
    lib.mosaic_masked_logits_noalloc.restype = ctypes.c_int
    lib.mosaic_min_chunk_rows.argtypes = [I64, I64, ctypes.c_int, I64,
                                          ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_int64)]
    lib.mosaic_min_chunk_rows.restype = ctypes.c_int
    lib.mosaic_masked_sample_workspace_bytes.argtypes = [I64, I64, I64]
    lib.mosaic_masked_sample_workspace_bytes.restype = ctypes.c_int64
    lib.mosaic_masked_sample.argtypes = [P, P, I64, I64, P, I64, P, P, I32, P, I64, P, P, P, I64,
                                         I64, P]
    lib.mosaic_masked_sample.restype = ctypes.c_int
    lib.mosaic_workspace_create.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, I64]
    lib.mosaic_workspace_create.restype = ctypes.c_int
    lib.mosaic_workspace_bind.argtypes = [P, I64, ctypes.POINTER(ctypes.c_void_p)]
    lib.mosaic_workspace_bind.restype = ctypes.c_int
    lib.mosaic_workspace_trim.argtypes = [P, I64]
    lib.mosaic_workspace_trim.restype = ctypes.c_int
    lib.mosaic_workspace_bound_bytes.argtypes = [P]
    lib.mosaic_workspace_bound_bytes.restype = ctypes.c_int64
    lib.mosaic_workspace_reserved_bytes.argtypes = [P]
    lib.mosaic_workspace_reserved_bytes.restype = ctypes.c_int64
    lib.mosaic_workspace_destroy.argtypes = [P]
    lib.mosaic_workspace_destroy.restype = ctypes.c_int
    lib.mosaic_masked_logits_fp8.argtypes = [P, P, P, I64, I64, P, I64, P, P, I32, P, P, I64, P,
                                             ctypes.c_int, I64, mosaic_chunk_cb, P, P]
    lib.mosaic_masked_logits_fp8.restype = ctypes.c_int
    lib.mosaic_quantize_rows_e4m3.argtypes = [P, I64, I64, P, P, P]
    lib.mosaic_quantize_rows_e4m3.restype = ctypes.c_int
    lib.mosaic_quantize_masked_rows_e4m3.argtypes = [P, I64, I64, P, I64, P, P, I32, P, P, P]
    lib.mosaic_quantize_masked_rows_e4m3.restype = ctypes.c_int
    _lib = lib
    return lib


# ------------------------------------------------------------------ C-ABI mirrors (same names)

def mosaic_create(device: int = 0):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    st = load_library().mosaic_create(ctypes.byref(h), int(device))
    return st, h


def mosaic_destroy(handle) -> int:
    return load_library().mosaic_destroy(handle)


def mosaic_masked_logits(handle, hidden, L_tot, d, mask_idx, M, seq_offsets, mask_offsets, B,
                         W, V, out, out_dtype, chunk_rows, cb, user, stream) -> int:
    """Raw call; pointer arguments are ints (device addresses) or None."""
    cb_c = cb if isinstance(cb, mosaic_chunk_cb) else (mosaic_chunk_cb(cb) if cb else mosaic_chunk_cb())
    return load_library().mosaic_masked_logits(handle, hidden, L_tot, d, mask_idx, M, seq_offsets,
                                               mask_offsets, B, W, V, out, out_dtype, chunk_rows,
                                               cb_c, user, stream)


def mosaic_masked_logits_fp8(handle, hidden_q, hidden_scale, L_tot, d, mask_idx, M, seq_offsets,
                             mask_offsets, B, W_q, w_scale, V, out, out_dtype, chunk_rows, cb,
                             user, stream) -> int:
    """Raw call; pointer arguments are ints (device addresses) or None."""
    cb_c = cb if isinstance(cb, mosaic_chunk_cb) else (mosaic_chunk_cb(cb) if cb else mosaic_chunk_cb())
    return load_library().mosaic_masked_logits_fp8(handle, hidden_q, hidden_scale, L_tot, d,
                                                   mask_idx, M, seq_offsets, mask_offsets, B,
                                                   W_q, w_scale, V, out, out_dtype, chunk_rows,
                                                   cb_c, user, stream)


def mosaic_quantize_rows_e4m3(x, rows, d, q, scale, stream) -> int:
    """Raw call; pointer arguments are ints (device addresses) or None."""
    return load_library().mosaic_quantize_rows_e4m3(x, rows, d, q, scale, stream)


def mosaic_quantize_masked_rows_e4m3(hidden, L_tot, d, mask_idx, M, seq_offsets, mask_offsets, B,
                                     hidden_q, hidden_scale, stream) -> int:
    """Raw call; pointer arguments are ints (device addresses) or None."""
    return load_library().mosaic_quantize_masked_rows_e4m3(hidden, L_tot, d, mask_idx, M,
                                                           seq_offsets, mask_offsets, B, hidden_q,
                                                           hidden_scale, stream)


def quantize_masked_rows_e4m3(hidden, mask_idx, hidden_q, hidden_scale, seq_offsets=None,
                              mask_offsets=None, stream=None):
    """Quantize, in place in hidden_q (uint8 [L_tot, d]) / hidden_scale (float32 [L_tot]), the
    hidden rows the masked positions name (see mosaic_quantize_masked_rows_e4m3)."""
    import torch

    if hidden.dim() != 2:
        raise ValueError("hidden must be [L_tot, d]")
    L_tot, d = int(hidden.shape[0]), int(hidden.shape[1])
    _require("hidden", hidden, torch.bfloat16)
    _require("hidden_q", hidden_q, torch.uint8, (L_tot, d))
    _require("hidden_scale", hidden_scale, torch.float32, (L_tot,))
    _check_mask(mask_idx, seq_offsets, mask_offsets)
    M = int(mask_idx.numel())
    csr = seq_offsets is not None
    s = stream if stream is not None else torch.cuda.current_stream(hidden.device)
    with torch.cuda.device(hidden.device):
        st = mosaic_quantize_masked_rows_e4m3(
            hidden.data_ptr(), L_tot, d, mask_idx.data_ptr() if M else None, M,
            seq_offsets.data_ptr() if csr else None, mask_offsets.data_ptr() if csr else None,
            int(seq_offsets.numel()) - 1 if csr else 0, hidden_q.data_ptr(),
            hidden_scale.data_ptr(), s.cuda_stream)
    if st != MOSAIC_OK:
        raise MosaicError(st, mosaic_last_error_string())
    return hidden_q, hidden_scale


def quantize_rows_e4m3(x, stream=None):
    """Per-row E4M3 quantization of a contiguous bf16 [rows, d] tensor (see
    mosaic_quantize_rows_e4m3 in include/mosaic.h). Returns (codes uint8 [rows, d],
    scale float32 [rows]) on x's device; d must be a multiple of 16."""
    import torch

    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 [rows, d] tensor")
    rows, d = int(x.shape[0]), int(x.shape[1])
    q = torch.empty((rows, d), dtype=torch.uint8, device=x.device)
    scale = torch.empty((rows,), dtype=torch.float32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        st = mosaic_quantize_rows_e4m3(x.data_ptr() if rows else None, rows, d,
                                       q.data_ptr() if rows else None,
                                       scale.data_ptr() if rows else None, s.cuda_stream)
    if st != MOSAIC_OK:
        raise MosaicError(st, mosaic_last_error_string())
    return q, scale


def mosaic_masked_logits_noalloc(hidden, L_tot, d, mask_idx, M, seq_offsets, mask_offsets, B,
                                 W, V, out, out_dtype, chunk_rows, cb, user, chunk_status,
                                 stream) -> int:
    """Raw call of the allocation-free entry point (current CUDA device, no handle).
    chunk_status: None (asynchronous) or a ctypes uint32 array with one word per chunk."""
    cb_c = cb if isinstance(cb, mosaic_chunk_cb) else (mosaic_chunk_cb(cb) if cb else mosaic_chunk_cb())
    return load_library().mosaic_masked_logits_noalloc(hidden, L_tot, d, mask_idx, M, seq_offsets,
                                                       mask_offsets, B, W, V, out, out_dtype,
                                                       chunk_rows, cb_c, user, chunk_status,
                                                       stream)


def mosaic_min_chunk_rows(M: int, V: int, out_dtype: int, budget_bytes: int):
    """Returns (status, chunk_rows, n_chunks): the fewest chunks whose live output fits."""
    cr, nc = ctypes.c_int64(), ctypes.c_int64()
    st = load_library().mosaic_min_chunk_rows(int(M), int(V), int(out_dtype), int(budget_bytes),
                                              ctypes.byref(cr), ctypes.byref(nc))
    return st, cr.value, nc.value


def mosaic_masked_sample_workspace_bytes(M: int, V: int, chunk_rows: int = 0) -> int:
    return load_library().mosaic_masked_sample_workspace_bytes(int(M), int(V), int(chunk_rows))


def mosaic_masked_sample(handle, hidden, L_tot, d, mask_idx, M, seq_offsets, mask_offsets, B, W,
                         V, token, confidence, workspace, workspace_bytes, chunk_rows,
                         stream) -> int:
    """Raw call of the fused gather-GEMM + greedy sampling; pointers are ints or None."""
    return load_library().mosaic_masked_sample(handle, hidden, L_tot, d, mask_idx, M, seq_offsets,
                                               mask_offsets, B, W, V, token, confidence,
                                               workspace, workspace_bytes, chunk_rows, stream)


def mosaic_check(handle, stream) -> int:
    return load_library().mosaic_check(handle, stream)


def mosaic_set_wait_timeout(handle, timeout_ns: int) -> int:
    return load_library().mosaic_set_wait_timeout(handle, int(timeout_ns))


def mosaic_launch_count(handle) -> int:
    return load_library().mosaic_launch_count(handle)


def mosaic_last_error_string() -> str:
    return load_library().mosaic_last_error_string().decode()


# ------------------------------------------------------------------ host-side argument checks
# The kernels read and write exactly the extents the sizes passed to the C ABI imply; the library
# cannot see a tensor's real size, so the wrappers check every tensor against those extents here.

def _require(name, t, dtype, shape=None):
    """t must be a contiguous tensor of `dtype` (and of exactly `shape`, if given)."""
    if t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check_mask(mask_idx, seq_offsets, mask_offsets):
    """mask_idx int32 [M]; the CSR pair both or neither, int32 [B + 1] each with B >= 1.
    Returns B (0 in flat mode)."""
    import torch

    _require("mask_idx", mask_idx, torch.int32)
    if mask_idx.dim() != 1:
        raise ValueError("mask_idx must be one-dimensional")
    if (seq_offsets is None) != (mask_offsets is None):
        raise ValueError("CSR mode needs both seq_offsets and mask_offsets")
    if seq_offsets is None:
        return 0
    _require("seq_offsets", seq_offsets, torch.int32)
    _require("mask_offsets", mask_offsets, torch.int32)
    if seq_offsets.dim() != 1 or mask_offsets.shape != seq_offsets.shape or seq_offsets.numel() < 2:
        raise ValueError("seq_offsets and mask_offsets must both be int32 [B + 1] with B >= 1")
    return int(seq_offsets.numel()) - 1


def _check_out(out, rows_out, V, out_dtype):
    import torch

    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    if out is not None:
        _require("out", out, out_dtype, (rows_out, V))


# ------------------------------------------------------------------ torch convenience wrapper

class Mosaic:
    """Owns a handle on one CUDA device; takes torch tensors."""

    def __init__(self, device: int = 0):
        import torch  # noqa: F401  (device memory and streams)

        st, h = mosaic_create(device)
        if st != MOSAIC_OK:
            raise MosaicError(st, mosaic_last_error_string())
        self.handle = h
        self.device = device

    def close(self):
        if self.handle:
            mosaic_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _stream_ptr(self, stream):
        import torch

        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return s.cuda_stream

    def masked_logits(self, hidden, mask_idx, W, seq_offsets=None, mask_offsets=None,
                      out=None, out_dtype=None, chunk_rows: int = 0,
                      on_chunk: Optional[Callable] = None, stream=None):
        """Mask-only logits. Returns ``out`` ([M, V], or [chunk_rows, V] holding the last chunk
        when chunking is on). ``on_chunk(chunk, row_begin, rows, out)`` runs on the host after
        each chunk is enqueued; it must enqueue its use of ``out`` on the same stream."""
        import torch

        _require("hidden", hidden, torch.bfloat16)
        _require("W", W, torch.bfloat16)
        if hidden.dim() != 2 or W.dim() != 2 or hidden.shape[1] != W.shape[1]:
            raise ValueError("hidden [L_tot, d] and W [V, d] must agree on d")
        B = _check_mask(mask_idx, seq_offsets, mask_offsets)
        M = int(mask_idx.numel())
        V, d = int(W.shape[0]), int(W.shape[1])
        if out_dtype is None:
            out_dtype = out.dtype if out is not None else torch.bfloat16
        chunked = 0 < chunk_rows < M
        rows_out = chunk_rows if chunked else M
        _check_out(out, rows_out, V, out_dtype)
        code = MOSAIC_F32 if out_dtype == torch.float32 else MOSAIC_BF16
        if out is None:
            out = torch.empty((rows_out, V), dtype=out_dtype, device=W.device)
        csr = seq_offsets is not None

        def _cb(c, rb, rows, _ptr, _user):
            on_chunk(int(c), int(rb), int(rows), out)

        cb = mosaic_chunk_cb(_cb) if on_chunk is not None else mosaic_chunk_cb()
        st = mosaic_masked_logits(
            self.handle, hidden.data_ptr(), int(hidden.shape[0]), d,
            mask_idx.data_ptr() if M > 0 else None, M,
            seq_offsets.data_ptr() if csr else None, mask_offsets.data_ptr() if csr else None, B,
            W.data_ptr(), V, out.data_ptr(), code, int(chunk_rows), cb, None,
            self._stream_ptr(stream))
        if st != MOSAIC_OK:
            raise MosaicError(st, mosaic_last_error_string())
        return out

    def masked_logits_fp8(self, hidden_q, hidden_scale, mask_idx, W_q, w_scale,
                          seq_offsets=None, mask_offsets=None, out=None, out_dtype=None,
                          chunk_rows: int = 0, on_chunk: Optional[Callable] = None, stream=None):
        """FP8 variant of masked_logits: E4M3 codes (uint8 tensors) with per-row fp32 scales, as
        produced by quantize_rows_e4m3; same chunking and output as masked_logits."""
        import torch

        _require("hidden_q", hidden_q, torch.uint8)
        _require("W_q", W_q, torch.uint8)
        if hidden_q.dim() != 2 or W_q.dim() != 2 or hidden_q.shape[1] != W_q.shape[1]:
            raise ValueError("hidden_q [L_tot, d] and W_q [V, d] must agree on d")
        _require("hidden_scale", hidden_scale, torch.float32, (hidden_q.shape[0],))
        _require("w_scale", w_scale, torch.float32, (W_q.shape[0],))
        B = _check_mask(mask_idx, seq_offsets, mask_offsets)
        M = int(mask_idx.numel())
        V, d = int(W_q.shape[0]), int(W_q.shape[1])
        if out_dtype is None:
            out_dtype = out.dtype if out is not None else torch.bfloat16
        chunked = 0 < chunk_rows < M
        rows_out = chunk_rows if chunked else M
        _check_out(out, rows_out, V, out_dtype)
        code = MOSAIC_F32 if out_dtype == torch.float32 else MOSAIC_BF16
        if out is None:
            out = torch.empty((rows_out, V), dtype=out_dtype, device=W_q.device)
        csr = seq_offsets is not None

        def _cb(c, rb, rows, _ptr, _user):
            on_chunk(int(c), int(rb), int(rows), out)

        cb = mosaic_chunk_cb(_cb) if on_chunk is not None else mosaic_chunk_cb()
        st = mosaic_masked_logits_fp8(
            self.handle, hidden_q.data_ptr(), hidden_scale.data_ptr(), int(hidden_q.shape[0]), d,
            mask_idx.data_ptr() if M > 0 else None, M,
            seq_offsets.data_ptr() if csr else None, mask_offsets.data_ptr() if csr else None, B,
            W_q.data_ptr(), w_scale.data_ptr(), V, out.data_ptr(), code, int(chunk_rows), cb,
            None, self._stream_ptr(stream))
        if st != MOSAIC_OK:
            raise MosaicError(st, mosaic_last_error_string())
        return out

    def masked_sample(self, hidden, mask_idx, W, seq_offsets=None, mask_offsets=None,
                      chunk_rows: int = 0, workspace=None, stream=None):
        """Greedy token (int32 [M]) and confidence (fp32 [M]) of every masked position, without
        writing the [M, V] logits. ``workspace`` (uint8 device tensor) is allocated with torch if
        not given."""
        import torch

        _require("hidden", hidden, torch.bfloat16)
        _require("W", W, torch.bfloat16)
        if hidden.dim() != 2 or W.dim() != 2 or hidden.shape[1] != W.shape[1]:
            raise ValueError("hidden [L_tot, d] and W [V, d] must agree on d")
        B = _check_mask(mask_idx, seq_offsets, mask_offsets)
        M = int(mask_idx.numel())
        V, d = int(W.shape[0]), int(W.shape[1])
        need = mosaic_masked_sample_workspace_bytes(M, V, chunk_rows)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=W.device)
        elif not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor")
        token = torch.empty(M, dtype=torch.int32, device=W.device)
        conf = torch.empty(M, dtype=torch.float32, device=W.device)
        csr = seq_offsets is not None
        st = mosaic_masked_sample(
            self.handle, hidden.data_ptr(), int(hidden.shape[0]), d,
            mask_idx.data_ptr() if M > 0 else None, M,
            seq_offsets.data_ptr() if csr else None, mask_offsets.data_ptr() if csr else None,
            B, W.data_ptr(), V,
            token.data_ptr() if M > 0 else None, conf.data_ptr() if M > 0 else None,
            workspace.data_ptr(), workspace.numel() * workspace.element_size(), int(chunk_rows),
            self._stream_ptr(stream))
        if st != MOSAIC_OK:
            raise MosaicError(st, mosaic_last_error_string())
        return token, conf

    def check(self, stream=None) -> int:
        """Synchronise and return the device status (MOSAIC_OK / _INDEX / _TIMEOUT / _CUDA)."""
        return mosaic_check(self.handle, self._stream_ptr(stream))

    def set_wait_timeout(self, ns: int):
        mosaic_set_wait_timeout(self.handle, ns)

    @property
    def launches(self) -> int:
        return mosaic_launch_count(self.handle)


# ------------------------------------------------------------------ VMM-backed output workspace

def mosaic_workspace_create(device: int, reserve_bytes: int):
    """Returns (status, workspace handle)."""
    ws = ctypes.c_void_p()
    st = load_library().mosaic_workspace_create(ctypes.byref(ws), int(device), int(reserve_bytes))
    return st, ws


def mosaic_workspace_bind(ws, nbytes: int):
    """Returns (status, base address)."""
    p = ctypes.c_void_p()
    st = load_library().mosaic_workspace_bind(ws, int(nbytes), ctypes.byref(p))
    return st, p.value


def mosaic_workspace_trim(ws, keep_bytes: int) -> int:
    return load_library().mosaic_workspace_trim(ws, int(keep_bytes))


def mosaic_workspace_bound_bytes(ws) -> int:
    return load_library().mosaic_workspace_bound_bytes(ws)


def mosaic_workspace_reserved_bytes(ws) -> int:
    return load_library().mosaic_workspace_reserved_bytes(ws)


def mosaic_workspace_destroy(ws) -> int:
    return load_library().mosaic_workspace_destroy(ws)


class Workspace:
    """Virtual range reserved once; physical pages bound only as far as `bind` asks."""

    def __init__(self, reserve_bytes: int, device: int = 0):
        st, ws = mosaic_workspace_create(device, reserve_bytes)
        if st != MOSAIC_OK:
            raise MosaicError(st, mosaic_last_error_string())
        self.ws, self.device = ws, device

    def bind(self, nbytes: int) -> int:
        st, ptr = mosaic_workspace_bind(self.ws, nbytes)
        if st != MOSAIC_OK:
            raise MosaicError(st, mosaic_last_error_string())
        return ptr

    def tensor(self, shape, dtype):
        """Bind enough pages for a contiguous tensor of `shape` and return a view of it."""
        import torch

        n = 1
        for x in shape:
            n *= int(x)
        ptr = self.bind(n * torch.empty(0, dtype=dtype).element_size())
        from .dlpack import device_view

        return device_view(ptr, shape, dtype, self.device)

    def trim(self, keep_bytes: int = 0):
        st = mosaic_workspace_trim(self.ws, keep_bytes)
        if st != MOSAIC_OK:
            raise MosaicError(st, mosaic_last_error_string())

    @property
    def bound_bytes(self) -> int:
        return mosaic_workspace_bound_bytes(self.ws)

    @property
    def reserved_bytes(self) -> int:
        return mosaic_workspace_reserved_bytes(self.ws)

    def close(self):
        if self.ws:
            mosaic_workspace_destroy(self.ws)
            self.ws = None
