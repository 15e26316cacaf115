"""fp64 CPU oracle for the chunked causal 3-D convolution.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg import this module.  The product library
(``chunked_causal_convolution_gb300``) never imports, loads or calls it, and it
shares no code with the CUDA path: the arithmetic lives in ``cc3d_oracle.c``,
a direct nested loop in double precision, wrapped here with ``ctypes``.

What it computes is stated in ``cc3d_oracle.c``.  In short (NDHWC, batch 1):

    Y[t,h,w,co] = b[co] + sum_{dt,dh,dw,ci} W[co,dt,dh,dw,ci]
                              * Xz[t+dt-(kt-1), h+dh-(kh-1)/2, w+dw-(kw-1)/2, ci]
                  (+ R[t,h,w,co])

with Xz zero outside the video (causal zero history, spatial zero padding).
Sources: "SwiftVR Inference Optimization" (LightX2V blog), section "ReAE:
Causal Halo Exchange" (current frame paired with previous input frames; cache
of input features; zeros before the first chunk) and "SGLang-Diffusion advanced
optimizations", section 3 "Parallel VAE" (chunked / halo-split work equals the
unsplit dense 3-D convolution).

Every function here takes and returns float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "cc3d_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library (gcc, -O2, no FMA contraction)."""
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
           "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``cc3d_oracle.c`` into ``liboracle.so`` next to it when stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE)):
        return _LIB
    return compile_source(SOURCE, _LIB)


class OracleLib:
    """The oracle entry points bound to one compiled library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        i = ctypes.c_int
        lib.cc3d_oracle_whole.argtypes = [i] * 8 + [dp] * 5 + [i]
        lib.cc3d_oracle_chunk.argtypes = [i] * 8 + [dp] * 7 + [i]
        lib.cc3d_oracle_points.argtypes = [i] * 9 + [ip] + [dp] * 5 + [i]
        for f in (lib.cc3d_oracle_whole, lib.cc3d_oracle_chunk, lib.cc3d_oracle_points):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    conv_whole = lambda self, *a, **k: conv_whole(*a, _lib=self.lib, **k)  # noqa: E731
    conv_chunk = lambda self, *a, **k: conv_chunk(*a, _lib=self.lib, **k)  # noqa: E731
    conv_chunked = lambda self, *a, **k: conv_chunked(*a, _lib=self.lib, **k)  # noqa: E731
    conv_points = lambda self, *a, **k: conv_points(*a, _lib=self.lib, **k)  # noqa: E731


def _load():
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default.lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f64(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError("expected shape %s, got %s" % (tuple(shape), a.shape))
    return a


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc):
    if rc != 0:
        raise ValueError("oracle rejected its arguments (code %d)" % rc)


def conv_whole(x, w, b=None, r=None, nthreads=None, _lib=None):
    """Causal conv of a whole sequence.

    x: [T][H][W][Cin]; w: [Cout][kt][kh][kw][Cin]; b: [Cout] or None;
    r: [T][H][W][Cout] or None.  Returns y: [T][H][W][Cout] (float64).
    """
    x = _f64(x)
    w = _f64(w)
    T, H, W, Cin = x.shape
    Cout, kt, kh, kw, Cin_w = w.shape
    if Cin_w != Cin:
        raise ValueError("Cin mismatch")
    b = _f64(b, (Cout,))
    r = _f64(r, (T, H, W, Cout))
    y = np.empty((T, H, W, Cout), dtype=np.float64)
    _check((_lib or _load()).cc3d_oracle_whole(T, H, W, Cin, Cout, kt, kh, kw, _ptr(x), _ptr(w), _ptr(b),
                                     _ptr(r), _ptr(y), nthreads or default_threads()))
    return y


def conv_chunk(x_chunk, w, b=None, r=None, cache_in=None, nthreads=None, _lib=None):
    """One chunk with a carried cache.

    x_chunk: [Tc][H][W][Cin]; cache_in: [kt-1][H][W][Cin] or None (zero history).
    Returns (y [Tc][H][W][Cout], cache_out [kt-1][H][W][Cin]).
    """
    x_chunk = _f64(x_chunk)
    w = _f64(w)
    Tc, H, W, Cin = x_chunk.shape
    Cout, kt, kh, kw, Cin_w = w.shape
    if Cin_w != Cin:
        raise ValueError("Cin mismatch")
    P = kt - 1
    b = _f64(b, (Cout,))
    r = _f64(r, (Tc, H, W, Cout))
    cache_in = _f64(cache_in, (P, H, W, Cin))
    y = np.empty((Tc, H, W, Cout), dtype=np.float64)
    cache_out = np.empty((P, H, W, Cin), dtype=np.float64)
    _check((_lib or _load()).cc3d_oracle_chunk(Tc, H, W, Cin, Cout, kt, kh, kw, _ptr(x_chunk), _ptr(w),
                                     _ptr(b), _ptr(r), _ptr(cache_in),
                                     _ptr(cache_out) if P > 0 else None, _ptr(y),
                                     nthreads or default_threads()))
    return y, cache_out


def conv_chunked(x, w, b=None, r=None, chunks=None, nthreads=None, _lib=None):
    """Run the chunk form over a whole sequence split into ``chunks`` (list of lengths).

    Returns (y [T][H][W][Cout], list of cache_out after each chunk).
    """
    x = _f64(x)
    T = x.shape[0]
    chunks = list(chunks) if chunks is not None else [T]
    if sum(chunks) != T or any(c < 1 for c in chunks):
        raise ValueError("chunk lengths must be >= 1 and sum to T")
    ys, caches = [], []
    cache = None
    s = 0
    for c in chunks:
        rc = None if r is None else np.asarray(r)[s:s + c]
        y, cache = conv_chunk(x[s:s + c], w, b, rc, cache, nthreads, _lib=_lib)
        ys.append(y)
        caches.append(cache)
        s += c
    return np.concatenate(ys, axis=0), caches


def conv_points(shape, pts, xwin, w, b=None, rpts=None, nthreads=None, _lib=None):
    """Y of the whole-sequence definition at chosen output positions.

    shape: (T, H, W) of the video; pts: int array [n][3] of (t, h, w);
    xwin: [n][kt][kh][kw][Cin] input values around each point (entries that
    fall outside the video are ignored); rpts: [n][Cout] or None.
    Returns [n][Cout].
    """
    T, H, W = (int(v) for v in shape)
    w = _f64(w)
    Cout, kt, kh, kw, Cin = w.shape
    pts = np.ascontiguousarray(np.asarray(pts, dtype=np.int32).reshape(-1, 3))
    n = pts.shape[0]
    xwin = _f64(xwin, (n, kt, kh, kw, Cin))
    b = _f64(b, (Cout,))
    rpts = _f64(rpts, (n, Cout))
    y = np.empty((n, Cout), dtype=np.float64)
    _check((_lib or _load()).cc3d_oracle_points(T, H, W, Cin, Cout, kt, kh, kw, n,
                                      pts.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                      _ptr(xwin), _ptr(w), _ptr(b), _ptr(rpts), _ptr(y),
                                      nthreads or default_threads()))
    return y


def upsample_nearest2x(x):
    """Nearest-neighbour 2x spatial upsampling of [T][H][W][C] frames: every input position's
    features are copied to the 2 x 2 block of output positions it covers ("SwiftVR Inference
    Optimization" (LightX2V blog), the TemporalGrow section: the nearest-neighbour upsample that
    feeds the decoder's spatial convolution)."""
    x = _f64(x)
    return np.repeat(np.repeat(x, 2, axis=1), 2, axis=2)


def conv_upsample2x_whole(x, w, b=None, r=None, nthreads=None, _lib=None):
    """The convolution of the nearest-2x upsampled sequence: conv_whole(upsample_nearest2x(x))."""
    return conv_whole(upsample_nearest2x(x), w, b, r, nthreads=nthreads, _lib=_lib)


def round_bf16(y):
    """Round float64 values to the nearest bfloat16 value, ties to even, returned as float64.

    bfloat16 keeps 8 significant bits and float32's 8-bit exponent.  For y = m * 2**e with
    0.5 <= |m| < 1 the representable neighbours of y are spaced 2**(e - 8) apart (the spacing stays
    2**-133 below the normal range, e < -125); y is scaled by that spacing, rounded half to even and
    scaled back, which is exact in float64.  Magnitudes that round to 2**128 or beyond become inf;
    NaN stays NaN.  (The outputs of the decoder's convolution are stored as bfloat16: "SwiftVR
    Inference Optimization" (LightX2V blog) runs the VAE in BF16.)"""
    y = _f64(y)
    with np.errstate(invalid="ignore"):
        _, e = np.frexp(y)
        step = np.maximum(e, -125) - 8
        r = np.ldexp(np.rint(np.ldexp(y, -step)), step)
        return np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, y), r)


def quantize_u8(y):
    """8-bit pixels of the decoder's output frames (the device-side half of the asynchronous frame
    output path: "How Synthesia optimizes generative AI video inference on Amazon EC2 G7e
    instances" copies finished frames to the host while the next chunk computes, and 8-bit frames
    halve those copies).  The pages name 8-bit frames but not the mapping; the reading taken is the
    plain one for decoder outputs in [-1, 1]:

        v = round_bf16(y)                            (the value the bf16 output stores)
        t = fp32(fp32(v + 1) * 127.5)                 (float32, one rounding per operation)
        q = clamp(round_half_even(t), 0, 255)

    y: float64 array of exact convolution outputs.  Returns uint8 of the same shape.  NaN inputs
    have no defined pixel."""
    v = round_bf16(y).astype(np.float32)  # exact: every bfloat16 value is a float32 value
    t = (v + np.float32(1.0)).astype(np.float32)
    t = (t * np.float32(127.5)).astype(np.float32)
    with np.errstate(invalid="ignore"):
        return np.clip(np.rint(t), 0.0, 255.0).astype(np.uint8)
