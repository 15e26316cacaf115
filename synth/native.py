"""ctypes bindings of synth_kernels.cu: GPU fill and fast host evaluation of the same generator."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_kernels.cu")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off", "-fmad=false", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i, u, ll, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_longlong, ctypes.c_double
            lib.synth_fill_device.argtypes = [vp, i, i, ctypes.c_ulonglong, u, ll, ll, d, d, vp]
            lib.synth_fill_device.restype = i
            lib.synth_values_host.argtypes = [vp, i, i, ctypes.c_ulonglong, u, vp, ll, d, d]
            lib.synth_values_host.restype = None
            _lib = lib
    return _lib


def fill_device(tensor, seed: int, tensor_id: int, dist, offset: int = 0, stream=None):
    """Fill a contiguous CUDA tensor (float32 or bfloat16) with elements offset .. offset+numel-1."""
    import torch
    if tensor.dtype == torch.float32:
        dt = 0
    elif tensor.dtype == torch.bfloat16:
        dt = 1
    else:
        raise ValueError("float32 or bfloat16 tensors only")
    if not (tensor.is_cuda and tensor.is_contiguous()):
        raise ValueError("contiguous CUDA tensor expected")
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _load().synth_fill_device(tensor.data_ptr(), dt, int(dist.kind), int(seed), int(tensor_id), int(offset),
                                   int(tensor.numel()), float(dist.p0), float(dist.p1), s or None)
    if rc != 0:
        raise RuntimeError("synth fill failed with CUDA error %d" % rc)
    return tensor


def values_host(seed: int, tensor_id: int, dist, e, dtype: str) -> np.ndarray:
    """Like synth.raw(): float32 values or bfloat16 bit patterns at global indices e (fast C path)."""
    e = np.ascontiguousarray(np.asarray(e, dtype=np.int64))
    shape = e.shape
    e = e.reshape(-1)
    if dtype == "f32":
        out = np.empty(e.shape, dtype=np.float32)
        dt = 0
    elif dtype == "bf16":
        out = np.empty(e.shape, dtype=np.uint16)
        dt = 1
    else:
        raise ValueError(dtype)
    _load().synth_values_host(out.ctypes.data, dt, int(dist.kind), int(seed), int(tensor_id), e.ctypes.data,
                              int(e.size), float(dist.p0), float(dist.p1))
    return out.reshape(shape)
