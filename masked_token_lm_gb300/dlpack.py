"""Torch tensor views of raw device memory owned elsewhere (e.g. a VMM workspace), through the
DLPack protocol. No copy and no ownership: the memory must outlive the tensor."""
from __future__ import annotations

import ctypes

_KDL_CUDA = 2
_CODES = {"float32": (2, 32), "bfloat16": (4, 16), "int32": (0, 32), "uint8": (1, 8),
          "float16": (2, 16)}


class _DLDevice(ctypes.Structure):
    _fields_ = [("device_type", ctypes.c_int), ("device_id", ctypes.c_int)]


class _DLDataType(ctypes.Structure):
    _fields_ = [("code", ctypes.c_uint8), ("bits", ctypes.c_uint8), ("lanes", ctypes.c_uint16)]


class _DLTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("device", _DLDevice), ("ndim", ctypes.c_int),
                ("dtype", _DLDataType), ("shape", ctypes.POINTER(ctypes.c_int64)),
                ("strides", ctypes.POINTER(ctypes.c_int64)), ("byte_offset", ctypes.c_uint64)]


class _DLManagedTensor(ctypes.Structure):
    pass


_DELETER = ctypes.CFUNCTYPE(None, ctypes.POINTER(_DLManagedTensor))
_DLManagedTensor._fields_ = [("dl_tensor", _DLTensor), ("manager_ctx", ctypes.c_void_p),
                             ("deleter", _DELETER)]

_alive = {}  # id -> (managed tensor, shape array): kept until the consumer calls the deleter


@_DELETER
def _release(ptr):
    _alive.pop(ctypes.addressof(ptr.contents), None)


_capsule_new = ctypes.pythonapi.PyCapsule_New
_capsule_new.restype = ctypes.py_object
_capsule_new.argtypes = [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_void_p]


def device_view(ptr: int, shape, dtype, device: int = 0):
    """A contiguous torch tensor of `shape` and `dtype` over device memory at `ptr`."""
    import torch

    name = str(dtype).replace("torch.", "")
    code, bits = _CODES[name]
    shp = (ctypes.c_int64 * len(shape))(*[int(x) for x in shape])
    mt = _DLManagedTensor()
    mt.dl_tensor.data = ctypes.c_void_p(int(ptr))
    mt.dl_tensor.device = _DLDevice(_KDL_CUDA, int(device))
    mt.dl_tensor.ndim = len(shape)
    mt.dl_tensor.dtype = _DLDataType(code, bits, 1)
    mt.dl_tensor.shape = shp
    mt.dl_tensor.strides = None
    mt.dl_tensor.byte_offset = 0
    mt.deleter = _release
    _alive[ctypes.addressof(mt)] = (mt, shp)
    capsule = _capsule_new(ctypes.addressof(mt), b"dltensor", None)
    return torch.utils.dlpack.from_dlpack(capsule)
