"""Shared helpers of the GPU parity tests: seeded inputs, chunk loops, tolerances."""
from __future__ import annotations

import numpy as np

import synth

BF16_TOL = 2e-2   # max|y_gpu - y_oracle| <= BF16_TOL * RMS(y_oracle) over the compared set
F32_TOL = 1e-4    # max|y_gpu - y_oracle| <= F32_TOL * max|y_oracle|


def tolerance(dtype: str, ref: np.ndarray) -> float:
    if dtype == "bf16":
        return BF16_TOL * float(np.sqrt(np.mean(ref ** 2)))
    return F32_TOL * float(np.abs(ref).max())


def to_f64(raw: np.ndarray, dtype: str) -> np.ndarray:
    return synth.bf16_bits_to_f64(raw) if dtype == "bf16" else raw.astype(np.float64)


def to_device(raw: np.ndarray, dtype: str, device="cuda"):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(raw).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(raw)).to(device)


def from_device(t) -> np.ndarray:
    import torch
    return t.to(torch.float64).cpu().numpy()


def small_inputs(Cin, Cout, T, H, W, dtype, seed, bias=True, residual=False, x_dist=None, k=(3, 3, 3)):
    """Dense CPU-generated inputs (raw stored form) for sizes the oracle finishes in seconds;
    k = (kt, kh, kw) is the kernel extent."""
    e = synth.dense_index
    x_dist = x_dist or synth.Dist.normal(1.0)
    raw = {
        "x": synth.raw(seed, synth.TID_X, x_dist, e((T, H, W, Cin)), dtype),
        "w": synth.raw(seed, synth.TID_W, synth.Dist.normal(synth.fan_in_sigma(Cin, *k)),
                       e((Cout, k[0], k[1], k[2], Cin)), dtype),
    }
    if bias:
        raw["b"] = synth.raw(seed, synth.TID_B, synth.Dist.uniform(-0.1, 0.1), e((Cout,)), dtype)
    if residual:
        raw["r"] = synth.raw(seed, synth.TID_R, synth.Dist.normal(1.0), e((T, H, W, Cout)), dtype)
    return raw


def run_chunks(plan, x, w, b, r, chunks, stream=None, zero_cache_first=False):
    """Chunk loop with two ping-pong caches; returns (y, list of cache tensors after each chunk)."""
    import torch
    caches = [plan.new_cache(x.device), plan.new_cache(x.device)]
    ys, outs, s = [], [], 0
    for k, c in enumerate(chunks):
        cin = caches[k % 2] if (k > 0 or zero_cache_first) else None
        cout = caches[(k + 1) % 2]
        rc = r[s:s + c] if r is not None else None
        ys.append(plan.forward_chunk(x[s:s + c], w, b, rc, cin, cout, stream=stream))
        outs.append(cout.clone())
        s += c
    return torch.cat(ys), outs


def compositions_sample():
    return [[24], [4] * 6, [1, 23], [5, 5, 5, 5, 4], [3, 1, 4, 1, 5, 10]]

