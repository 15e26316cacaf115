"""Chunked causal 3-D convolution for GB300 (sm_103a): Python binding of libcc3d.so.

This module only marshals arguments: every step of the convolution (the
implicit-GEMM tensor-core kernel, its fused bias / residual epilogue, the
temporal-cache update, the float32 CUDA-core kernel) runs in the CUDA kernels
of ``libcc3d.so``.  PyTorch is used for device memory and streams only.  There
is no CPU or library fallback: if the shared library is missing, every call
raises.

The functions carry the C ABI's names (``include/cc3d.h``):

    plan = cc3d_plan_create(Cin, Cout, H, W, kt, kh, kw, dtype)
    cc3d_forward_chunk(plan, T, x, w, b, residual, cache_in, cache_out, y, stream)
    cc3d_reset(plan, cache, stream); cc3d_get_status(plan, stream); cc3d_destroy(plan)

where tensor arguments are CUDA tensors (or raw device addresses as ints, or
None) and ``stream`` is a ``torch.cuda.Stream``, a raw handle or None (the
current stream).  :class:`CausalConv3dPlan` wraps the same calls.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "CC3D_F32", "CC3D_BF16", "CC3DError", "CausalConv3dPlan",
    "cc3d_plan_create", "cc3d_plan_create_upsample2x", "cc3d_forward_chunk", "cc3d_forward_chunk_u8",
    "cc3d_reset", "cc3d_get_status", "cc3d_destroy", "cc3d_status_string", "cc3d_plan_kernel",
    "cc3d_plan_launches_per_chunk", "cc3d_plan_describe", "cc3d_debug_set_wait_budget_ns",
    "cc3d_debug_set_fault", "cc3d_debug_set_schedule", "SCHEDULE_KNOBS", "cc3d_last_error_detail",
    "library_path", "Upsample2xConvPlan",
    "load_library", "FrameWriter",
    "cc3d_writer_create", "cc3d_writer_submit", "cc3d_writer_wait_copied", "cc3d_writer_close",
    "cc3d_group_create", "cc3d_group_workspace_bytes", "cc3d_group_forward_chunk", "cc3d_group_destroy",
    "LayerGroup", "weights_from_torch_layout", "EXPORTED_SYMBOLS",
]

CC3D_F32 = 0
CC3D_BF16 = 1

STATUS_NAMES = {
    0: "CC3D_OK", 1: "CC3D_ERR_INVALID_ARG", 2: "CC3D_ERR_UNSUPPORTED", 3: "CC3D_ERR_ALIGNMENT",
    4: "CC3D_ERR_ALIAS", 5: "CC3D_ERR_CUDA", 6: "CC3D_ERR_OOM", 7: "CC3D_ERR_DEVICE_TIMEOUT",
    8: "CC3D_ERR_NOT_DEVICE_MEMORY", 9: "CC3D_ERR_IO", 10: "CC3D_ERR_SCRATCH_TOO_SMALL",
}

EXPORTED_SYMBOLS = (
    "cc3d_plan_create", "cc3d_plan_create_upsample2x", "cc3d_forward_chunk", "cc3d_forward_chunk_u8", "cc3d_reset", "cc3d_get_status",
    "cc3d_destroy",
    "cc3d_status_string", "cc3d_plan_kernel", "cc3d_plan_launches_per_chunk", "cc3d_plan_describe",
    "cc3d_debug_set_wait_budget_ns", "cc3d_debug_set_fault", "cc3d_debug_set_schedule", "cc3d_last_error_detail",
    "cc3d_writer_create", "cc3d_writer_submit", "cc3d_writer_wait_copied", "cc3d_writer_close",
    "cc3d_group_create", "cc3d_group_workspace_bytes", "cc3d_group_forward_chunk", "cc3d_group_destroy",
    "cc3d_group_forward_chunk_static",
)

# the CC3D_SCHED_* knobs of cc3d.h, by name (value -1 restores the measured default)
SCHEDULE_KNOBS = {
    "pair": 0, "two_frame": 1, "split_tail": 2, "channel_blocks": 3, "mma_warps": 4, "row_groups": 5,
    "acc_stages": 6, "tap_rows": 7, "window_stages": 8, "weight_stages": 9, "prefetch": 10, "channel_block": 11,
}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None
_lock = threading.Lock()


class CC3DError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        self.name = STATUS_NAMES.get(code, str(code))
        msg = "%s (%s)" % (self.name, _status_text(code))
        if code == 5:
            msg += ": " + cc3d_last_error_detail()
        super().__init__("%s: %s" % (what, msg) if what else msg)


def library_path() -> str:
    return os.path.join(_HERE, "libcc3d.so")


def load_library():
    """Load libcc3d.so (built in-tree by ``build.py``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("libcc3d.so is not built (expected at %s); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
        lib = ctypes.CDLL(path)
        vp, i, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong
        lib.cc3d_plan_create.argtypes = [i] * 8 + [ctypes.POINTER(vp)]
        lib.cc3d_plan_create_upsample2x.argtypes = [i] * 6 + [ctypes.POINTER(vp)]
        lib.cc3d_forward_chunk.argtypes = [vp, i] + [vp] * 8
        lib.cc3d_forward_chunk_u8.argtypes = [vp, i] + [vp] * 8
        lib.cc3d_reset.argtypes = [vp, vp, vp]
        lib.cc3d_get_status.argtypes = [vp, vp]
        lib.cc3d_destroy.argtypes = [vp]
        lib.cc3d_destroy.restype = None
        lib.cc3d_status_string.argtypes = [i]
        lib.cc3d_status_string.restype = ctypes.c_char_p
        lib.cc3d_plan_kernel.argtypes = [vp]
        lib.cc3d_plan_kernel.restype = ctypes.c_char_p
        lib.cc3d_plan_launches_per_chunk.argtypes = [vp]
        lib.cc3d_plan_describe.argtypes = [vp, i, i, ctypes.c_char_p, ctypes.c_size_t]
        lib.cc3d_debug_set_wait_budget_ns.argtypes = [vp, u64]
        lib.cc3d_debug_set_fault.argtypes = [vp, i]
        lib.cc3d_debug_set_schedule.argtypes = [vp, i, i]
        lib.cc3d_writer_create.argtypes = [ctypes.c_char_p, ctypes.c_size_t, ctypes.POINTER(vp)]
        lib.cc3d_writer_submit.argtypes = [vp, vp, ctypes.c_size_t, vp, ctypes.POINTER(ctypes.c_longlong)]
        lib.cc3d_writer_wait_copied.argtypes = [vp, ctypes.c_longlong, vp]
        lib.cc3d_writer_close.argtypes = [vp, ctypes.POINTER(ctypes.c_longlong)]
        for f in (lib.cc3d_writer_create, lib.cc3d_writer_submit, lib.cc3d_writer_wait_copied,
                  lib.cc3d_writer_close):
            f.restype = i
        lib.cc3d_group_create.argtypes = [i, ctypes.POINTER(vp), i, ctypes.POINTER(vp)]
        lib.cc3d_group_workspace_bytes.argtypes = [vp, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.cc3d_group_forward_chunk.argtypes = [vp, i, vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                 ctypes.POINTER(vp), vp, vp, ctypes.c_size_t, vp]
        lib.cc3d_group_forward_chunk_static.argtypes = [vp, i, vp, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                        ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp]
        lib.cc3d_group_forward_chunk_static.restype = i
        lib.cc3d_group_destroy.argtypes = [vp]
        lib.cc3d_group_destroy.restype = None
        for f in (lib.cc3d_group_create, lib.cc3d_group_workspace_bytes, lib.cc3d_group_forward_chunk):
            f.restype = i
        lib.cc3d_last_error_detail.argtypes = []
        lib.cc3d_last_error_detail.restype = ctypes.c_char_p
        for f in (lib.cc3d_plan_create, lib.cc3d_plan_create_upsample2x, lib.cc3d_forward_chunk, lib.cc3d_forward_chunk_u8, lib.cc3d_reset,
                  lib.cc3d_get_status,
                  lib.cc3d_plan_launches_per_chunk, lib.cc3d_plan_describe, lib.cc3d_debug_set_wait_budget_ns,
                  lib.cc3d_debug_set_fault, lib.cc3d_debug_set_schedule):
            f.restype = i
        _lib = lib
        return lib


def _status_text(code: int) -> str:
    try:
        return load_library().cc3d_status_string(code).decode()
    except Exception:
        return STATUS_NAMES.get(code, "?")


def _check(code: int, what: str):
    if code != 0:
        raise CC3DError(code, what)


def _dtype_code(dtype) -> int:
    if dtype in (CC3D_F32, CC3D_BF16):
        return dtype
    s = str(dtype)
    if s in ("bf16", "bfloat16", "torch.bfloat16"):
        return CC3D_BF16
    if s in ("f32", "float32", "torch.float32"):
        return CC3D_F32
    raise ValueError("unsupported dtype %r" % (dtype,))


def _addr(t):
    """Device address of a tensor argument (tensor, int address or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t or None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    _check_device(t)
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr() or None


def _check_device(t):
    """The library launches on the current device; a tensor of another device would be read
    through that device's addresses, so it is refused here (the C ABI refuses it too)."""
    import torch
    cur = torch.cuda.current_device()
    if t.device.index is not None and t.device.index != cur:
        raise ValueError("tensor on %s, but the current device is cuda:%d" % (t.device, cur))


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


# ---------------------------------------------------------------- C-ABI names
def cc3d_plan_create(Cin, Cout, H, W, kt=3, kh=3, kw=3, dtype=CC3D_BF16):
    h = ctypes.c_void_p()
    _check(load_library().cc3d_plan_create(int(Cin), int(Cout), int(H), int(W), int(kt), int(kh), int(kw),
                                           _dtype_code(dtype), ctypes.byref(h)), "cc3d_plan_create")
    return h.value


def cc3d_plan_create_upsample2x(Cin, Cout, H, W, kt=3, dtype=CC3D_BF16):
    h = ctypes.c_void_p()
    _check(load_library().cc3d_plan_create_upsample2x(int(Cin), int(Cout), int(H), int(W), int(kt),
                                                      _dtype_code(dtype), ctypes.byref(h)),
           "cc3d_plan_create_upsample2x")
    return h.value


def cc3d_forward_chunk(plan, T, x, w, b, residual, cache_in, cache_out, y, stream=None):
    _check(load_library().cc3d_forward_chunk(plan, int(T), _addr(x), _addr(w), _addr(b), _addr(residual),
                                             _addr(cache_in), _addr(cache_out), _addr(y), _stream(stream)),
           "cc3d_forward_chunk")


def cc3d_forward_chunk_u8(plan, T, x, w, b, residual, cache_in, cache_out, y_u8, stream=None):
    _check(load_library().cc3d_forward_chunk_u8(plan, int(T), _addr(x), _addr(w), _addr(b), _addr(residual),
                                                _addr(cache_in), _addr(cache_out), _addr(y_u8), _stream(stream)),
           "cc3d_forward_chunk_u8")


def cc3d_writer_create(path: str, slot_bytes: int):
    h = ctypes.c_void_p()
    _check(load_library().cc3d_writer_create(os.fsencode(path), int(slot_bytes), ctypes.byref(h)),
           "cc3d_writer_create")
    return h.value


def cc3d_writer_submit(writer, src, nbytes, stream=None) -> int:
    seq = ctypes.c_longlong(-1)
    _check(load_library().cc3d_writer_submit(writer, _addr(src), int(nbytes), _stream(stream), ctypes.byref(seq)),
           "cc3d_writer_submit")
    return seq.value


def cc3d_writer_wait_copied(writer, seq, stream=None):
    _check(load_library().cc3d_writer_wait_copied(writer, int(seq), _stream(stream)), "cc3d_writer_wait_copied")


def cc3d_writer_close(writer) -> int:
    n = ctypes.c_longlong(0)
    _check(load_library().cc3d_writer_close(writer, ctypes.byref(n)), "cc3d_writer_close")
    return n.value


def _ptr_array(items):
    """A host array of device pointers (tensors, int addresses or None) for the group calls."""
    if items is None:
        return None
    return (ctypes.c_void_p * len(items))(*[_addr(t) for t in items])


def cc3d_group_create(plans, frame_batch: int):
    """plans: C plan handles (or CausalConv3dPlan objects), first layer first."""
    hs = [p.handle if hasattr(p, "handle") else p for p in plans]
    arr = (ctypes.c_void_p * len(hs))(*hs)
    g = ctypes.c_void_p()
    _check(load_library().cc3d_group_create(len(hs), arr, int(frame_batch), ctypes.byref(g)), "cc3d_group_create")
    return g.value


def cc3d_group_workspace_bytes(group, T_max: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().cc3d_group_workspace_bytes(group, int(T_max), ctypes.byref(n)), "cc3d_group_workspace_bytes")
    return n.value


def cc3d_group_forward_chunk(group, T, x, w, b, cache_in, cache_out, y, workspace, workspace_bytes, stream=None):
    """w, b, cache_in, cache_out: per-layer lists (b, cache_in may be None; entries may be None)."""
    _check(load_library().cc3d_group_forward_chunk(group, int(T), _addr(x), _ptr_array(w), _ptr_array(b),
                                                   _ptr_array(cache_in), _ptr_array(cache_out), _addr(y),
                                                   _addr(workspace), int(workspace_bytes), _stream(stream)),
           "cc3d_group_forward_chunk")


def cc3d_group_forward_chunk_static(group, T, x, w, b, cache_in, cache_out, y, stream=None):
    """cc3d_group_forward_chunk with the library's fixed device scratch array as its workspace:
    allocates nothing, for callers that cannot allocate device memory (see include/cc3d.h)."""
    _check(load_library().cc3d_group_forward_chunk_static(group, int(T), _addr(x), _ptr_array(w), _ptr_array(b),
                                                          _ptr_array(cache_in), _ptr_array(cache_out), _addr(y),
                                                          _stream(stream)),
           "cc3d_group_forward_chunk_static")


def cc3d_group_destroy(group):
    if group:
        load_library().cc3d_group_destroy(group)


class FrameWriter:
    """The C ABI's asynchronous chunk writer: `submit` a device buffer after the chunk that fills it
    is enqueued; call `wait_copied(seq, stream)` before that buffer is overwritten; `close` writes
    everything and returns the bytes written."""

    def __init__(self, path, slot_bytes):
        self.handle = cc3d_writer_create(path, slot_bytes)

    def submit(self, src, nbytes=None, stream=None) -> int:
        return cc3d_writer_submit(self.handle, src, src.numel() * src.element_size() if nbytes is None else nbytes,
                                  stream)

    def wait_copied(self, seq, stream=None):
        cc3d_writer_wait_copied(self.handle, seq, stream)

    def close(self) -> int:
        h, self.handle = self.handle, None
        return cc3d_writer_close(h) if h else 0


def cc3d_reset(plan, cache, stream=None):
    _check(load_library().cc3d_reset(plan, _addr(cache), _stream(stream)), "cc3d_reset")


def cc3d_get_status(plan, stream=None) -> int:
    """Synchronise the stream and return the status code (0 = ok); never raises on device errors."""
    return int(load_library().cc3d_get_status(plan, _stream(stream)))


def cc3d_destroy(plan):
    if plan:
        load_library().cc3d_destroy(plan)


def cc3d_last_error_detail() -> str:
    return load_library().cc3d_last_error_detail().decode()


def cc3d_status_string(code: int) -> str:
    return load_library().cc3d_status_string(int(code)).decode()


def cc3d_plan_kernel(plan) -> str:
    s = load_library().cc3d_plan_kernel(plan)
    return s.decode() if s else ""


def cc3d_plan_launches_per_chunk(plan) -> int:
    return int(load_library().cc3d_plan_launches_per_chunk(plan))


def cc3d_plan_describe(plan, T, has_residual=True) -> dict:
    """The launch configuration of a T-frame chunk as {key: value} (ints where the value is one)."""
    buf = ctypes.create_string_buffer(1024)
    _check(load_library().cc3d_plan_describe(plan, int(T), 1 if has_residual else 0, buf, len(buf)),
           "cc3d_plan_describe")
    out = {}
    for item in buf.value.decode().split():
        k, v = item.split("=", 1)
        out[k] = int(v) if v.lstrip("-").isdigit() else v
    return out


def cc3d_debug_set_wait_budget_ns(plan, ns: int):
    _check(load_library().cc3d_debug_set_wait_budget_ns(plan, int(ns)), "cc3d_debug_set_wait_budget_ns")


def cc3d_debug_set_fault(plan, mode: int):
    _check(load_library().cc3d_debug_set_fault(plan, int(mode)), "cc3d_debug_set_fault")


def cc3d_debug_set_schedule(plan, knob, value: int):
    """Override one schedule knob of the plan (a CC3D_SCHED_* number or a SCHEDULE_KNOBS name);
    -1 restores the measured default."""
    k = SCHEDULE_KNOBS[knob] if isinstance(knob, str) else int(knob)
    _check(load_library().cc3d_debug_set_schedule(plan, k, int(value)), "cc3d_debug_set_schedule")


# ---------------------------------------------------------------- convenience
def weights_from_torch_layout(w_oikkk):
    """PyTorch Conv3d weights [Cout][Cin][kt][kh][kw] -> this library's [Cout][kt][kh][kw][Cin]."""
    return w_oikkk.permute(0, 2, 3, 4, 1).contiguous()


class CausalConv3dPlan:
    """One layer shape; owns the C plan.  Tensors are NDHWC (batch 1) CUDA tensors."""

    def __init__(self, Cin, Cout, H, W, kt=3, kh=3, kw=3, dtype="bf16"):
        self.Cin, self.Cout, self.H, self.W = int(Cin), int(Cout), int(H), int(W)
        self.kt, self.kh, self.kw = int(kt), int(kh), int(kw)
        self.dtype = _dtype_code(dtype)
        self.Ho, self.Wo = self.H, self.W  # output frame size
        self.handle = cc3d_plan_create(Cin, Cout, H, W, kt, kh, kw, self.dtype)

    @property
    def kernel(self) -> str:
        return cc3d_plan_kernel(self.handle)

    @property
    def launches_per_chunk(self) -> int:
        return cc3d_plan_launches_per_chunk(self.handle)

    def describe(self, T, has_residual=True) -> dict:
        """The launch configuration a T-frame chunk of this plan would use (host-only)."""
        return cc3d_plan_describe(self.handle, T, has_residual)

    def torch_dtype(self):
        import torch
        return torch.float32 if self.dtype == CC3D_F32 else torch.bfloat16

    def new_cache(self, device="cuda"):
        """A zeroed history buffer [kt-1][H][W][Cin] (allocated by PyTorch, zeroed by the library)."""
        import torch
        c = torch.empty((self.kt - 1, self.H, self.W, self.Cin), dtype=self.torch_dtype(), device=device)
        if self.kt > 1:
            self.reset(c)
        return c

    def _check_sizes(self, T, y_dtype, **tensors):
        """Element counts and dtypes of the tensor arguments against the plan.  The C ABI takes
        bare pointers and cannot see a buffer's size, so a tensor of the wrong shape would be read
        or written past its end; this catches it before the call (integer addresses and None are
        passed through unchecked)."""
        dt = self.torch_dtype()
        hist = (self.kt - 1) * self.H * self.W * self.Cin
        out = T * self.Ho * self.Wo * self.Cout
        need = {"x": (T * self.H * self.W * self.Cin, dt),
                "w": (self.Cout * self.kt * self.kh * self.kw * self.Cin, dt),
                "b": (self.Cout, dt), "residual": (out, dt), "cache_in": (hist, dt), "cache_out": (hist, dt),
                "cache": (hist, dt), "y": (out, y_dtype)}
        for name, t in tensors.items():
            if t is None or isinstance(t, int):
                continue
            n, d = need[name]
            if t.dtype != d:
                raise ValueError("%s has dtype %s; this plan takes %s" % (name, t.dtype, d))
            if t.numel() != n:
                raise ValueError("%s has %d elements (shape %s); this plan takes %d"
                                 % (name, t.numel(), tuple(t.shape), n))

    def forward_chunk(self, x, w, b=None, residual=None, cache_in=None, cache_out=None, y=None, stream=None):
        """Enqueue one chunk; returns y ([T][H][W][Cout]).  cache_out receives the new history."""
        import torch
        T = 0 if x is None else int(x.shape[0])
        if y is None and T > 0:
            y = torch.empty((T, self.Ho, self.Wo, self.Cout), dtype=self.torch_dtype(), device=x.device)
        self._check_sizes(T, self.torch_dtype(), x=x, w=w, b=b, residual=residual, cache_in=cache_in,
                          cache_out=cache_out, y=y)
        cc3d_forward_chunk(self.handle, T, x, w, b, residual, cache_in, cache_out, y, stream)
        return y

    def forward_chunk_u8(self, x, w, b=None, residual=None, cache_in=None, cache_out=None, y=None, stream=None):
        """Enqueue one chunk of a narrow-output plan with 8-bit pixels out; returns y (uint8)."""
        import torch
        T = 0 if x is None else int(x.shape[0])
        if y is None and T > 0:
            y = torch.empty((T, self.Ho, self.Wo, self.Cout), dtype=torch.uint8, device=x.device)
        self._check_sizes(T, torch.uint8, x=x, w=w, b=b, residual=residual, cache_in=cache_in,
                          cache_out=cache_out, y=y)
        cc3d_forward_chunk_u8(self.handle, T, x, w, b, residual, cache_in, cache_out, y, stream)
        return y

    def reset(self, cache, stream=None):
        self._check_sizes(0, self.torch_dtype(), cache=cache)
        cc3d_reset(self.handle, cache, stream)

    def status(self, stream=None) -> int:
        return cc3d_get_status(self.handle, stream)

    def set_wait_budget_ns(self, ns):
        cc3d_debug_set_wait_budget_ns(self.handle, ns)

    def set_fault(self, mode):
        cc3d_debug_set_fault(self.handle, mode)

    def set_schedule(self, knob, value):
        """Override one schedule knob (name from SCHEDULE_KNOBS); -1 restores the default."""
        cc3d_debug_set_schedule(self.handle, knob, value)

    def close(self):
        if getattr(self, "handle", None):
            cc3d_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LayerGroup:
    """Consecutive layers (plans, first layer first) run frame batch by frame batch through the
    C ABI's layer-group runtime: each batch of `frame_batch` frames (0: the whole chunk) passes
    through every layer before the next batch starts, so only one batch of intermediate frames is
    held; layers with a history keep it from batch to batch.  The plans must outlive the group."""

    def __init__(self, plans, frame_batch: int = 1):
        self.plans = list(plans)
        self.frame_batch = int(frame_batch)
        self.handle = cc3d_group_create(self.plans, self.frame_batch)

    def workspace_bytes(self, T_max: int) -> int:
        return cc3d_group_workspace_bytes(self.handle, T_max)

    def new_workspace(self, T_max: int, device="cuda"):
        """A workspace for chunks of up to T_max frames (allocated by PyTorch; 256-byte aligned)."""
        import torch
        n = self.workspace_bytes(T_max)
        buf = torch.empty(n + 256, dtype=torch.uint8, device=device)
        off = (-buf.data_ptr()) % 256
        return buf[off:off + n]

    def forward_chunk(self, x, ws, bs=None, caches_in=None, caches_out=None, y=None, workspace=None, stream=None):
        """One chunk through the group; returns the last layer's output.  ws / bs / caches_in /
        caches_out are per-layer lists (caches_in None: zero histories)."""
        import torch
        T = 0 if x is None else int(x.shape[0])
        first, last = self.plans[0], self.plans[-1]
        if y is None and T > 0:
            y = torch.empty((T, last.Ho, last.Wo, last.Cout), dtype=last.torch_dtype(), device=x.device)
        first._check_sizes(T, first.torch_dtype(), x=x)
        last._check_sizes(T, last.torch_dtype(), y=y)
        for j, p in enumerate(self.plans):
            p._check_sizes(0, p.torch_dtype(), w=ws[j], b=None if bs is None else bs[j],
                           cache_in=None if caches_in is None else caches_in[j],
                           cache_out=None if caches_out is None else caches_out[j])
        if workspace is None:
            workspace = self.new_workspace(T, x.device if x is not None else "cuda")
        nbytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
        cc3d_group_forward_chunk(self.handle, T, x, ws, bs, caches_in, caches_out, y, workspace, nbytes, stream)
        return y

    def close(self):
        if getattr(self, "handle", None):
            cc3d_group_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Upsample2xConvPlan(CausalConv3dPlan):
    """A causal kt x 3 x 3 conv reading its H x W input through a fused nearest-2x upsample:
    outputs (and the residual) are 2H x 2W, histories hold source frames."""

    def __init__(self, Cin, Cout, H, W, kt=3, dtype="bf16"):
        self.Cin, self.Cout, self.H, self.W = int(Cin), int(Cout), int(H), int(W)
        self.kt, self.kh, self.kw = int(kt), 3, 3
        self.dtype = _dtype_code(dtype)
        self.Ho, self.Wo = 2 * self.H, 2 * self.W
        self.handle = cc3d_plan_create_upsample2x(Cin, Cout, H, W, kt, self.dtype)
