"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Each test ties the oracle to something it does not compute itself:

* a library routine for a special case (PyTorch's CPU float64 conv3d on an
  explicitly zero-padded input: causal pad kt-1 frames in front, (k-1)/2
  spatially),
* closed forms (delta kernels reproduce / shift the input; an all-ones input
  and kernel count the taps that fall inside the video),
* invariants the pages state: the chunked form with a carried cache equals the
  whole-sequence conv ("SGLang-Diffusion advanced optimizations", section 3
  "Parallel VAE": halo-split work stays mathematically equal), the cache holds
  the *input* features of the last frames and the first chunk sees zeros
  ("SwiftVR Inference Optimization", section "ReAE: Causal Halo Exchange"),
* the worked pairing example of that section (tests/golden/causal_pairs.txt),
* causality and linearity.
"""
import itertools
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_reference(x, w, b=None, r=None):
    """PyTorch conv3d (CPU, float64) on an explicitly padded NCDHW input."""
    T, H, W, Cin = x.shape
    Cout, kt, kh, kw, _ = w.shape
    xt = torch.from_numpy(np.ascontiguousarray(x)).permute(3, 0, 1, 2)[None]
    xt = F.pad(xt, ((kw - 1) // 2, (kw - 1) // 2, (kh - 1) // 2, (kh - 1) // 2, kt - 1, 0))
    wt = torch.from_numpy(np.ascontiguousarray(w)).permute(0, 4, 1, 2, 3)
    bt = None if b is None else torch.from_numpy(np.ascontiguousarray(b))
    y = F.conv3d(xt, wt, bt)[0].permute(1, 2, 3, 0).numpy()
    if r is not None:
        y = y + r
    return y


def rand(rng, *shape):
    return rng.standard_normal(shape)


SHAPES = [
    # T, H, W, Cin, Cout, kt, kh, kw
    (6, 5, 7, 3, 4, 3, 3, 3),
    (4, 1, 1, 1, 1, 3, 3, 3),
    (5, 6, 4, 8, 2, 3, 3, 3),
    (3, 4, 5, 2, 3, 2, 3, 3),   # MemoryBlock-like temporal extent 2
    (7, 3, 3, 4, 4, 3, 1, 1),   # temporal-only 3x1x1
    (2, 7, 6, 3, 5, 1, 3, 3),   # spatial-only
    (1, 3, 3, 2, 2, 3, 3, 3),   # one frame: only the current tap sees data
]


@pytest.mark.parametrize("shape", SHAPES)
def test_whole_matches_library_conv3d(shape):
    T, H, W, Cin, Cout, kt, kh, kw = shape
    rng = np.random.default_rng(sum(shape))
    x = rand(rng, T, H, W, Cin)
    w = rand(rng, Cout, kt, kh, kw, Cin)
    b = rand(rng, Cout)
    r = rand(rng, T, H, W, Cout)
    y = oracle.conv_whole(x, w, b, r)
    ref = torch_reference(x, w, b, r)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))
    # without bias and residual
    np.testing.assert_allclose(oracle.conv_whole(x, w), torch_reference(x, w), rtol=0, atol=1e-12 * 50)


def delta_kernel(C, kt, kh, kw, dt, dh, dw):
    w = np.zeros((C, kt, kh, kw, C))
    for c in range(C):
        w[c, dt, dh, dw, c] = 1.0
    return w


def test_delta_current_center_reproduces_input():
    rng = np.random.default_rng(1)
    x = rand(rng, 6, 5, 4, 3)
    y = oracle.conv_whole(x, delta_kernel(3, 3, 3, 3, 2, 1, 1))
    assert np.array_equal(y, x)


def test_delta_oldest_tap_is_two_frames_back_with_zero_history():
    rng = np.random.default_rng(2)
    x = rand(rng, 6, 4, 4, 2)
    y = oracle.conv_whole(x, delta_kernel(2, 3, 3, 3, 0, 1, 1))
    assert np.array_equal(y[2:], x[:-2])
    assert np.all(y[:2] == 0.0)
    y1 = oracle.conv_whole(x, delta_kernel(2, 3, 3, 3, 1, 1, 1))
    assert np.array_equal(y1[1:], x[:-1])
    assert np.all(y1[:1] == 0.0)


@pytest.mark.parametrize("dh,dw", [(0, 0), (2, 2), (0, 2), (2, 0), (1, 0), (0, 1)])
def test_delta_spatial_tap_shifts_with_zero_border(dh, dw):
    rng = np.random.default_rng(3)
    T, H, W, C = 2, 5, 6, 2
    x = rand(rng, T, H, W, C)
    y = oracle.conv_whole(x, delta_kernel(C, 3, 3, 3, 2, dh, dw))
    exp = np.zeros_like(x)
    for h in range(H):
        for w in range(W):
            hs, ws = h + dh - 1, w + dw - 1
            if 0 <= hs < H and 0 <= ws < W:
                exp[:, h, w] = x[:, hs, ws]
    assert np.array_equal(y, exp)


def test_channel_routing_with_unequal_channel_counts():
    """W[co, current, centre, ci] = [ci == perm[co]] routes input channels to outputs."""
    rng = np.random.default_rng(4)
    Cin, Cout = 5, 3
    perm = [4, 0, 2]
    x = rand(rng, 3, 3, 4, Cin)
    w = np.zeros((Cout, 3, 3, 3, Cin))
    for co, ci in enumerate(perm):
        w[co, 2, 1, 1, ci] = 1.0
    y = oracle.conv_whole(x, w)
    assert np.array_equal(y, x[..., perm])


@pytest.mark.parametrize("T,H,W,Cin,Cout", [(5, 4, 6, 3, 2), (4, 1, 3, 2, 1), (3, 7, 1, 4, 2)])
def test_constant_input_counts_taps_inside_the_video(T, H, W, Cin, Cout):
    x = np.ones((T, H, W, Cin))
    w = np.ones((Cout, 3, 3, 3, Cin))
    y = oracle.conv_whole(x, w)
    for t in range(T):
        for h in range(H):
            for ww in range(W):
                nt = min(t + 1, 3)
                nh = 3 - (h == 0) - (h == H - 1)
                nw = 3 - (ww == 0) - (ww == W - 1)
                assert np.all(y[t, h, ww] == Cin * nt * nh * nw)


def test_zero_kernel_gives_bias_plus_residual():
    rng = np.random.default_rng(5)
    b = rand(rng, 4)
    r = rand(rng, 3, 2, 5, 4)
    y = oracle.conv_whole(rand(rng, 3, 2, 5, 2), np.zeros((4, 3, 3, 3, 2)), b, r)
    assert np.array_equal(y, r + b)


def test_linearity():
    rng = np.random.default_rng(6)
    x1, x2 = rand(rng, 5, 4, 5, 3), rand(rng, 5, 4, 5, 3)
    w = rand(rng, 2, 3, 3, 3, 3)
    b = rand(rng, 2)
    a, c = 0.75, -1.5
    lhs = oracle.conv_whole(a * x1 + c * x2, w, b) - b
    rhs = a * (oracle.conv_whole(x1, w, b) - b) + c * (oracle.conv_whole(x2, w, b) - b)
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)


@pytest.mark.parametrize("t0", [0, 2, 5])
def test_causality(t0):
    rng = np.random.default_rng(7)
    T = 6
    x = rand(rng, T, 3, 4, 2)
    w = rand(rng, 3, 3, 3, 3, 2)
    y0 = oracle.conv_whole(x, w)
    x2 = x.copy()
    x2[t0] += rand(rng, 3, 4, 2)
    y1 = oracle.conv_whole(x2, w)
    changed = [bool(np.any(y0[t] != y1[t])) for t in range(T)]
    assert changed == [t0 <= t <= t0 + 2 for t in range(T)]


def compositions(n):
    for cuts in itertools.product([0, 1], repeat=n - 1):
        parts, last = [], 0
        for i, c in enumerate(cuts, start=1):
            if c:
                parts.append(i - last)
                last = i
        parts.append(n - last)
        yield parts


def test_chunked_equals_whole_for_every_chunking_of_8_frames():
    rng = np.random.default_rng(8)
    T, H, W, Cin, Cout = 8, 4, 5, 3, 2
    x = rand(rng, T, H, W, Cin)
    w = rand(rng, Cout, 3, 3, 3, Cin)
    b = rand(rng, Cout)
    r = rand(rng, T, H, W, Cout)
    whole = oracle.conv_whole(x, w, b, r, nthreads=1)
    n = 0
    for parts in compositions(T):
        y, caches = oracle.conv_chunked(x, w, b, r, chunks=parts, nthreads=1)
        assert np.array_equal(y, whole), parts
        # every cache is the two input frames that precede the next chunk
        end = 0
        for p, cache in zip(parts, caches):
            end += p
            for j in range(2):
                src = end - 2 + j
                exp = x[src] if src >= 0 else np.zeros_like(x[0])
                assert np.array_equal(cache[j], exp)
        n += 1
    assert n == 128


def test_chunked_equals_whole_for_other_temporal_extents():
    rng = np.random.default_rng(9)
    for kt, kh, kw in [(2, 3, 3), (3, 1, 1), (1, 3, 3), (4, 1, 3)]:
        x = rand(rng, 7, 3, 4, 2)
        w = rand(rng, 3, kt, kh, kw, 2)
        whole = oracle.conv_whole(x, w)
        for parts in ([7], [1] * 7, [3, 4], [2, 1, 4], [1, 6]):
            y, _ = oracle.conv_chunked(x, w, chunks=parts)
            assert np.array_equal(y, whole), (kt, kh, kw, parts)


def test_single_frame_chunk_takes_one_cache_frame_from_history():
    rng = np.random.default_rng(10)
    x = rand(rng, 1, 2, 3, 2)
    cache_in = rand(rng, 2, 2, 3, 2)
    _, cache_out = oracle.conv_chunk(x, rand(rng, 2, 3, 3, 3, 2), cache_in=cache_in)
    assert np.array_equal(cache_out[0], cache_in[1])
    assert np.array_equal(cache_out[1], x[0])
    _, cache0 = oracle.conv_chunk(x, rand(rng, 2, 3, 3, 3, 2))
    assert np.all(cache0[0] == 0.0) and np.array_equal(cache0[1], x[0])


def test_points_equal_whole_at_borders_and_interior():
    rng = np.random.default_rng(11)
    T, H, W, Cin, Cout = 5, 6, 7, 3, 4
    x = rand(rng, T, H, W, Cin)
    w = rand(rng, Cout, 3, 3, 3, Cin)
    b = rand(rng, Cout)
    r = rand(rng, T, H, W, Cout)
    y = oracle.conv_whole(x, w, b, r)
    pts = [(t, h, ww) for t in (0, 1, 2, 4) for h in (0, 3, 5) for ww in (0, 2, 6)]
    xpad = np.full((T + 2, H + 2, W + 2, Cin), np.nan)  # out-of-video entries must be ignored
    xpad[2:, 1:-1, 1:-1] = x
    xwin = np.stack([xpad[t:t + 3, h:h + 3, ww:ww + 3] for t, h, ww in pts])
    rp = np.stack([r[p] for p in pts])
    yp = oracle.conv_points((T, H, W), pts, xwin, w, b, rp)
    assert np.array_equal(yp, np.stack([y[p] for p in pts]))


def test_pages_worked_pairing_example():
    """kt=2, 1x1 spatial, one channel: y = cur + 10 * prev reproduces the printed pairs."""
    vals = {"P": 3.0, "A": 5.0, "B": 7.0, "C": 11.0, "D": 13.0, "E": 17.0, "F": 19.0, "0": 0.0}
    w = np.zeros((1, 2, 1, 1, 1))
    w[0, 1, 0, 0, 0] = 1.0   # current frame (tap dt = kt-1)
    w[0, 0, 0, 0, 0] = 10.0  # previous frame (tap dt = 0)
    lines = [ln for ln in open(os.path.join(GOLDEN, "causal_pairs.txt")) if ln.strip() and not ln.startswith("#")]
    assert len(lines) == 3
    for ln in lines:
        frames, hist, pairs = (s.split() for s in ln.split("|"))
        x = np.array([vals[f] for f in frames]).reshape(-1, 1, 1, 1)
        cache_in = None if hist == ["0"] else np.array([vals[hist[0]]]).reshape(1, 1, 1, 1)
        y, cache_out = oracle.conv_chunk(x, w, cache_in=cache_in)
        exp = [vals[c] + 10.0 * vals[p] for c, p in (pp.split(",") for pp in pairs)]
        assert y.reshape(-1).tolist() == exp
        # the next chunk's history is this chunk's last input frame
        assert cache_out.reshape(-1).tolist() == [vals[frames[-1]]]


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.conv_whole(np.zeros((2, 2, 2, 2)), np.zeros((1, 3, 2, 3, 2)))  # even kh
    with pytest.raises(ValueError):
        oracle.conv_chunked(np.zeros((3, 2, 2, 1)), np.zeros((1, 3, 3, 3, 1)), chunks=[1, 1])


# ---------------------------------------------------------------- nearest-2x upsampling (the decoder's
# upsampling stage feeding a spatial convolution)

def _torch_nearest2x(x):
    """PyTorch's nearest interpolation, scale (1, 2, 2), on NCDHW (an independent library routine)."""
    xt = torch.from_numpy(np.ascontiguousarray(x)).permute(3, 0, 1, 2)[None]
    u = F.interpolate(xt, scale_factor=(1, 2, 2), mode="nearest")
    return u[0].permute(1, 2, 3, 0).numpy()


def test_upsample_matches_library_nearest_interpolation():
    rng = np.random.default_rng(11)
    x = rand(rng, 3, 5, 7, 4)
    u = oracle.upsample_nearest2x(x)
    assert u.shape == (3, 10, 14, 4)
    assert np.array_equal(u, _torch_nearest2x(x))


@pytest.mark.parametrize("T,H,W,Cin,Cout,kt", [(4, 3, 5, 3, 2, 3), (3, 2, 2, 2, 3, 2), (2, 4, 3, 1, 1, 1)])
def test_upsample_conv_matches_library_routines(T, H, W, Cin, Cout, kt):
    rng = np.random.default_rng(T * 100 + H * 10 + W)
    x, w, b = rand(rng, T, H, W, Cin), rand(rng, Cout, kt, 3, 3, Cin), rand(rng, Cout)
    r = rand(rng, T, 2 * H, 2 * W, Cout)
    y = oracle.conv_upsample2x_whole(x, w, b, r)
    ref = torch_reference(_torch_nearest2x(x), w, b, r)
    assert y.shape == (T, 2 * H, 2 * W, Cout)
    assert np.abs(y - ref).max() < 1e-11


def test_upsample_conv_of_a_constant_counts_taps_inside_the_upsampled_frame():
    # x = 1, w = 1: every output counts Cin * min(t+1, kt) * (taps inside the 2H x 2W frame)
    T, H, W, C = 3, 2, 3, 2
    y = oracle.conv_upsample2x_whole(np.ones((T, H, W, C)), np.ones((1, 3, 3, 3, C)))
    Ho, Wo = 2 * H, 2 * W
    for t in range(T):
        for h in range(Ho):
            for w_ in range(Wo):
                nh = 3 - (h == 0) - (h == Ho - 1)
                nw = 3 - (w_ == 0) - (w_ == Wo - 1)
                assert y[t, h, w_, 0] == C * min(t + 1, 3) * nh * nw
