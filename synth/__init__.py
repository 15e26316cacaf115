"""Seeded synthetic inputs shared by the tests and the benchmark.

This module holds the input generators and nothing of the convolution's
arithmetic.  It is the one place both sides of a parity check draw their
inputs from: the CPU side here (numpy, and a C copy of it in ``synth_kernels.cu``'s host
code), the GPU side in the fill kernel of ``synth_kernels.cu`` (loaded through
``synth.native``), all implementing the same counter-based
definition so that every element is a pure function of
(seed, tensor id, global element index) and therefore independent of how a
video is split into chunks or of which device produced it.

Definition
----------
Counter-based SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast Splittable
Pseudorandom Number Generators", OOPSLA 2014): the n-th output (n >= 1) of a
generator seeded with s is ``mix64(s + n * GOLDEN)`` with

    mix64(z): z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
              z = (z ^ (z >> 27)) * 0x94D049BB133111EB
              return z ^ (z >> 31)

(all arithmetic modulo 2**64, GOLDEN = 0x9E3779B97F4A7C15).

* tensor key:  key = mix64(seed + (tensor_id + 1) * GOLDEN)
* draw j of element e (D draws per element):  z = mix64(key + (e*D + j + 1) * GOLDEN)
* normal N(0, sigma): D = 3; the twelve 16-bit fields k_i of the three draws
  give the Irwin-Hall approximation  sum_i (k_i + 0.5)/65536 - 6
  = (S - 393210) / 65536 with S = sum_i k_i  (mean 0, variance 1, support
  [-6, 6]); the value is  double(that) * sigma  (one double rounding).
* uniform U(lo, hi): D = 1; u = (z >> 40) / 2**24 in [0, 1);
  value = lo + (hi - lo) * u  in double, multiply and add rounded separately.
* the double value is rounded to float32 (nearest-even); a bfloat16 tensor
  rounds that float32 to bfloat16 (nearest-even).

Element index e is the row-major offset in the tensor's *global* layout:
activations [T][H][W][C] over the whole video (so frame t of any chunk has the
same values), weights [Cout][kt][kh][kw][Cin], bias [Cout].
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

NORMAL = 0
UNIFORM = 1

# tensor ids: one independent stream per role
TID_X, TID_W, TID_B, TID_R = 0, 1, 2, 3


def _mix64(z):
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def tensor_key(seed: int, tensor_id: int) -> np.uint64:
    s = np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    with np.errstate(over="ignore"):
        k = _mix64(s + np.uint64(tensor_id + 1) * GOLDEN)
    return k[0]


def _draw(key, idx):
    with np.errstate(over="ignore"):
        return _mix64(key + (idx + np.uint64(1)) * GOLDEN)


def values_f32(seed: int, tensor_id: int, dist: int, p0: float, p1: float, e) -> np.ndarray:
    """float32 values of elements with global indices ``e`` (any int array shape).

    dist NORMAL: p0 = mean offset (must be 0.0), p1 = sigma.
    dist UNIFORM: p0 = lo, p1 = hi.
    """
    e = np.asarray(e, dtype=np.int64)
    shape = e.shape
    e = e.reshape(-1).astype(np.uint64)
    key = tensor_key(seed, tensor_id)
    if dist == NORMAL:
        if p0 != 0.0:
            raise ValueError("normal draws are zero-mean")
        S = np.zeros(e.shape, dtype=np.int64)
        with np.errstate(over="ignore"):
            base = e * np.uint64(3)
        for j in range(3):
            z = _draw(key, base + np.uint64(j))
            for q in range(4):
                S += ((z >> np.uint64(16 * q)) & np.uint64(0xFFFF)).astype(np.int64)
        v = (S - 393210).astype(np.float64) / 65536.0
        v = v * float(p1)
    elif dist == UNIFORM:
        z = _draw(key, e)
        u = (z >> np.uint64(40)).astype(np.float64) / 16777216.0
        lo, hi = float(p0), float(p1)
        span = hi - lo
        v = lo + span * u
    else:
        raise ValueError("unknown distribution")
    return v.astype(np.float32).reshape(shape)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    rnd = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        out = (b + rnd) >> np.uint32(16)
    return out.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


@dataclass(frozen=True)
class Dist:
    """A distribution of one tensor: kind (NORMAL/UNIFORM) and its two parameters."""
    kind: int
    p0: float
    p1: float

    @staticmethod
    def normal(sigma: float) -> "Dist":
        return Dist(NORMAL, 0.0, float(sigma))

    @staticmethod
    def uniform(lo: float, hi: float) -> "Dist":
        return Dist(UNIFORM, float(lo), float(hi))


def values(seed: int, tensor_id: int, dist: Dist, e, dtype: str) -> np.ndarray:
    """Values as float64 numbers exactly equal to the stored element (f32 or bf16)."""
    f = values_f32(seed, tensor_id, dist.kind, dist.p0, dist.p1, e)
    if dtype == "f32":
        return f.astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f64(f32_to_bf16_bits(f))
    raise ValueError(dtype)


def raw(seed: int, tensor_id: int, dist: Dist, e, dtype: str) -> np.ndarray:
    """Stored representation: float32 array, or uint16 bfloat16 bit patterns."""
    f = values_f32(seed, tensor_id, dist.kind, dist.p0, dist.p1, e)
    if dtype == "f32":
        return f
    if dtype == "bf16":
        return f32_to_bf16_bits(f)
    raise ValueError(dtype)


def dense_index(shape, offset: int = 0) -> np.ndarray:
    """Global element indices of a dense row-major block starting at ``offset``."""
    n = int(np.prod(shape))
    return (np.arange(n, dtype=np.int64) + int(offset)).reshape(shape)


def fan_in_sigma(Cin: int, kt: int = 3, kh: int = 3, kw: int = 3) -> float:
    """Weight std 1/sqrt(Cin*kt*kh*kw) (fan-in scaling)."""
    return 1.0 / math.sqrt(Cin * kt * kh * kw)


# ---------------------------------------------------------------------------
# Workload recipes: shapes and distributions of the decoder-shaped layers.

@dataclass(frozen=True)
class Workload:
    name: str
    Cin: int
    Cout: int
    T: int
    H: int
    W: int
    chunks: tuple
    dtype: str
    seed: int
    x: Dist
    w: Dist
    b: Dist | None
    r: Dist | None
    kt: int = 3
    kh: int = 3
    kw: int = 3
    up2: bool = False  # the conv reads its H x W input through a nearest-2x upsample (2H x 2W outputs)

    @property
    def out_hw(self):
        return (2 * self.H, 2 * self.W) if self.up2 else (self.H, self.W)

    @property
    def flops(self) -> float:
        Ho, Wo = self.out_hw
        return 2.0 * self.Cin * self.Cout * self.kt * self.kh * self.kw * self.T * Ho * Wo


def _chunks(T, n):
    full, rest = divmod(T, n)
    return tuple([n] * full + ([rest] if rest else []))


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 16, 16, 8, 32, 32, (4, 4), "f32", 0,
                         Dist.uniform(-1.0, 1.0), Dist.normal(fan_in_sigma(16)),
                         Dist.uniform(-0.1, 0.1), None),
    "c96_residual": Workload("c96_residual", 96, 96, 24, 360, 640, _chunks(24, 4), "bf16", 1,
                             Dist.normal(1.0), Dist.normal(fan_in_sigma(96)),
                             Dist.uniform(-0.1, 0.1), Dist.normal(1.0)),
    "c192": Workload("c192", 192, 192, 24, 180, 320, _chunks(24, 4), "bf16", 2,
                     Dist.normal(1.0), Dist.normal(fan_in_sigma(192)),
                     Dist.uniform(-0.1, 0.1), None),
    "c384": Workload("c384", 384, 384, 24, 90, 160, _chunks(24, 4), "bf16", 3,
                     Dist.normal(1.0), Dist.normal(fan_in_sigma(384)),
                     Dist.uniform(-0.1, 0.1), None),
    "c384_to_192": Workload("c384_to_192", 384, 192, 24, 90, 160, _chunks(24, 4), "bf16", 4,
                            Dist.normal(1.0), Dist.normal(fan_in_sigma(384)),
                            Dist.uniform(-0.1, 0.1), None),
    "sr96": Workload("sr96", 96, 96, 361, 1440, 2560, _chunks(361, 4), "bf16", 5,
                     Dist.normal(1.0), Dist.normal(fan_in_sigma(96)),
                     Dist.uniform(-0.1, 0.1), None),
    # the decoder's neighbours of the 3x3x3 conv, at the c96 stage's size: a MemoryBlock conv
    # (kt = 2, one history frame), a TemporalGrow conv (3x1x1) and a pointwise projection (1x1x1)
    "memblock_c96": Workload("memblock_c96", 96, 96, 24, 360, 640, _chunks(24, 4), "bf16", 7,
                             Dist.normal(1.0), Dist.normal(fan_in_sigma(96, 2, 3, 3)),
                             Dist.uniform(-0.1, 0.1), Dist.normal(1.0), kt=2),
    "temporalgrow_c96": Workload("temporalgrow_c96", 96, 96, 24, 360, 640, _chunks(24, 4), "bf16", 8,
                                 Dist.normal(1.0), Dist.normal(fan_in_sigma(96, 3, 1, 1)),
                                 Dist.uniform(-0.1, 0.1), None, kh=1, kw=1),
    "pointwise_c192": Workload("pointwise_c192", 192, 192, 24, 180, 320, _chunks(24, 4), "bf16", 9,
                               Dist.normal(1.0), Dist.normal(fan_in_sigma(192, 1, 1, 1)),
                               Dist.uniform(-0.1, 0.1), None, kt=1, kh=1, kw=1),
    # the decoder's upsampling stage at the c96 stage's output size: 180x320 source frames read
    # through a nearest-2x upsample by a 96 -> 96 3x3x3 conv producing 360x640 frames
    "up2_c96": Workload("up2_c96", 96, 96, 24, 180, 320, _chunks(24, 4), "bf16", 10,
                        Dist.normal(1.0), Dist.normal(fan_in_sigma(96)), Dist.uniform(-0.1, 0.1), None, up2=True),
    "sr_head3": Workload("sr_head3", 96, 3, 361, 1440, 2560, _chunks(361, 4), "bf16", 6,
                         Dist.normal(1.0), Dist.normal(fan_in_sigma(96)),
                         Dist.uniform(-0.1, 0.1), None),
}
