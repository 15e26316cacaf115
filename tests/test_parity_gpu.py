"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

* small shapes compared element by element (several tiles, ragged tails, every
  kernel family: tensor-core row-aligned / flat / split-N / narrow head /
  16-channel blocks, and the fp32 CUDA-core path including the tiny fp32
  workload itself);
* the decoder-shaped workloads at full size, in the launch configuration the
  benchmark times (chunks of 4 frames with a carried cache), compared on
  sampled outputs (random positions, frame borders, chunk seams, column-block
  seams) that the oracle evaluates one by one;
* bit-identity of the GPU result across chunkings;
* tolerances: bf16  max|err| <= 2e-2 * RMS(y_oracle) over the compared set,
             fp32  max|err| <= 1e-4 * max|y_oracle|.
"""
import numpy as np
import pytest
import torch

import chunked_causal_convolution_gb300 as cc3d
import oracle
import synth
from synth import native
from tests.helpers import (compositions_sample, from_device, run_chunks, small_inputs, to_device, to_f64,
                           tolerance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


SMALL = [
    # name, dtype, Cin, Cout, T, H, W, chunks, bias, residual
    ("tiny_f32_workload", "f32", 16, 16, 8, 32, 32, [4, 4], True, False),
    ("f32_odd_shape", "f32", 3, 5, 5, 7, 9, [2, 1, 2], True, True),
    ("bf16_row_aligned_residual", "bf16", 96, 96, 5, 5, 256, [2, 3], True, True),
    ("bf16_flat", "bf16", 64, 64, 3, 7, 100, [1, 2], True, False),
    ("bf16_split_n", "bf16", 32, 384, 3, 4, 40, [3], False, True),
    ("bf16_narrow_head", "bf16", 96, 3, 3, 6, 130, [2, 1], True, True),
    ("bf16_head_strips_rows", "bf16", 64, 3, 5, 21, 260, [4, 1], True, False),
    ("bf16_head_cout1_two_passes", "bf16", 32, 1, 10, 5, 40, [10], True, True),
    ("bf16_head_cout5_cin256", "bf16", 256, 5, 7, 4, 127, [6, 1], False, True),
    ("bf16_head_cout2", "bf16", 160, 2, 3, 3, 253, [1, 2], True, False),
    ("bf16_narrow_generic", "bf16", 48, 3, 3, 5, 70, [2, 1], True, True),
    ("bf16_cb16", "bf16", 16, 32, 4, 9, 17, [1, 1, 2], True, False),
    ("bf16_two_flat_blocks", "bf16", 32, 16, 2, 3, 300, [2], True, False),
    ("bf16_c192_like", "bf16", 192, 192, 3, 8, 64, [2, 1], True, False),
    ("bf16_c96_wide_flat_window", "bf16", 96, 96, 3, 8, 100, [2, 1], True, True),
    ("bf16_c256_narrow_column_blocks", "bf16", 256, 256, 2, 3, 254, [1, 1], True, False),
    ("bf16_one_pixel", "bf16", 32, 32, 3, 1, 1, [1, 1, 1], True, True),
    # 16-channel blocks (Cin an odd multiple of 16) on SM pairs over row-aligned frames: the
    # two-frame schedule for the 4-frame chunk, the one-frame schedule for the 1-frame chunk
    ("bf16_cb16_pairs_row_aligned", "bf16", 48, 96, 5, 3, 256, [4, 1], True, True),
    # 16-channel blocks on one SM with one row group per MMA warp and 3-tap weight stages
    ("bf16_cb16_one_sm_wide_n", "bf16", 16, 192, 3, 5, 40, [2, 1], True, False),
    # a 4-channel narrow head
    ("bf16_head_cout4", "bf16", 96, 4, 4, 5, 140, [3, 1], True, True),
    # a head on frames narrower than the 8 pixels the lanes copy of the history
    ("bf16_head_narrow_frame", "bf16", 32, 3, 3, 4, 5, [2, 1], True, False),
]


# the kernel family each small case exercises
SMALL_KERNEL = {
    "tiny_f32_workload": "simt_f32", "f32_odd_shape": "simt_f32",
    "bf16_row_aligned_residual": "tc_bf16_pair", "bf16_flat": "tc_bf16", "bf16_split_n": "tc_bf16",
    "bf16_narrow_head": "tc_bf16_head", "bf16_head_strips_rows": "tc_bf16_head",
    "bf16_head_cout1_two_passes": "tc_bf16_head", "bf16_head_cout5_cin256": "tc_bf16_head",
    "bf16_head_cout2": "tc_bf16_head", "bf16_narrow_generic": "tc_bf16_narrow", "bf16_cb16": "tc_bf16",
    "bf16_two_flat_blocks": "tc_bf16", "bf16_c192_like": "tc_bf16", "bf16_one_pixel": "tc_bf16",
    "bf16_c96_wide_flat_window": "tc_bf16", "bf16_c256_narrow_column_blocks": "tc_bf16",
    "bf16_cb16_pairs_row_aligned": "tc_bf16_pair", "bf16_cb16_one_sm_wide_n": "tc_bf16",
    "bf16_head_cout4": "tc_bf16_head", "bf16_head_narrow_frame": "tc_bf16_head",
}


def _check_small(name, dtype, Cin, Cout, T, H, W, chunks, bias, residual, k=(3, 3, 3), kernel=None):
    """Element-wise parity with the oracle, history bytes, bit-identity across chunkings, and a
    second input set right after the first."""
    x_dist = synth.Dist.uniform(-1.0, 1.0) if name == "tiny_f32_workload" else None
    seed = 0 if name == "tiny_f32_workload" else 100 + len(name)
    raw = small_inputs(Cin, Cout, T, H, W, dtype, seed, bias, residual, x_dist=x_dist, k=k)
    dev = {kk: to_device(v, dtype) for kk, v in raw.items()}
    plan = cc3d.CausalConv3dPlan(Cin, Cout, H, W, *k, dtype=dtype)
    if kernel is not None:
        assert plan.kernel == kernel
    y, caches = run_chunks(plan, dev["x"], dev["w"], dev.get("b"), dev.get("r"), chunks)
    assert plan.status() == 0
    ref = oracle.conv_whole(to_f64(raw["x"], dtype), to_f64(raw["w"], dtype),
                            to_f64(raw["b"], dtype) if bias else None,
                            to_f64(raw["r"], dtype) if residual else None)
    got = from_device(y)
    err = np.abs(got - ref).max()
    assert err <= tolerance(dtype, ref), (name, err, tolerance(dtype, ref))
    # every cache_out holds the kt-1 input frames preceding the next chunk, bit for bit
    P = k[0] - 1
    xs = dev["x"]
    end = 0
    for c, cache in zip(chunks, caches):
        end += c
        assert cache.shape[0] == P
        for j in range(P):
            src = end - P + j
            exp = xs[src] if src >= 0 else torch.zeros_like(xs[0])
            assert torch.equal(cache[j], exp), (name, end, j)
    # bit-identical across chunkings
    for alt in ([T], [1] * T):
        y2, _ = run_chunks(plan, dev["x"], dev["w"], dev.get("b"), dev.get("r"), alt)
        assert torch.equal(y2, y), (name, alt)
    # a second input set right after the first: a stage consumed before its copy landed would
    # still hold the first set's data (repeated launches on equal inputs cannot show that)
    raw2 = small_inputs(Cin, Cout, T, H, W, dtype, 5000 + len(name), bias, residual, x_dist=x_dist, k=k)
    dev2 = {kk: to_device(v, dtype) for kk, v in raw2.items()}
    y3, _ = run_chunks(plan, dev2["x"], dev2["w"], dev2.get("b"), dev2.get("r"), chunks)
    assert plan.status() == 0
    ref2 = oracle.conv_whole(to_f64(raw2["x"], dtype), to_f64(raw2["w"], dtype),
                             to_f64(raw2["b"], dtype) if bias else None,
                             to_f64(raw2["r"], dtype) if residual else None)
    err2 = np.abs(from_device(y3) - ref2).max()
    assert err2 <= tolerance(dtype, ref2), (name, "second input set", err2)
    plan.close()


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes_match_oracle_elementwise(case):
    _check_small(*case, kernel=SMALL_KERNEL[case[0]])


# The decoder's neighbours of the 3x3x3 conv: MemoryBlock (kt = 2, one history frame),
# TemporalGrow (3x1x1), pointwise projections (1x1x1) and spatial-only kernels (kt = 1).
EXTENTS = [
    # name, dtype, Cin, Cout, T, H, W, chunks, bias, residual, (kt, kh, kw), kernel family
    ("bf16_memblock_kt2_pair", "bf16", 96, 96, 5, 4, 256, [2, 3], True, True, (2, 3, 3), "tc_bf16_pair"),
    ("bf16_memblock_kt2_flat", "bf16", 64, 64, 4, 6, 100, [1, 3], True, False, (2, 3, 3), "tc_bf16"),
    ("bf16_temporalgrow_stream", "bf16", 96, 96, 5, 3, 128, [3, 2], True, False, (3, 1, 1), "tc_bf16_stream"),
    ("bf16_temporalgrow_stream_res", "bf16", 32, 64, 4, 5, 70, [2, 2], False, True, (3, 1, 1), "tc_bf16_stream"),
    ("bf16_pointwise_stream", "bf16", 64, 128, 3, 4, 90, [1, 2], True, True, (1, 1, 1), "tc_bf16_stream"),
    ("bf16_kt2_1x1_stream_groups", "bf16", 64, 256, 9, 3, 50, [9], True, False, (2, 1, 1), "tc_bf16_stream"),
    ("bf16_temporalgrow_tiles", "bf16", 16, 32, 4, 5, 70, [2, 2], True, False, (3, 1, 1), "tc_bf16"),
    ("bf16_pointwise_tiles_wide", "bf16", 64, 384, 2, 3, 40, [1, 1], True, False, (1, 1, 1), "tc_bf16"),
    ("bf16_spatial_only", "bf16", 32, 32, 2, 5, 40, [1, 1], True, False, (1, 3, 3), "tc_bf16"),
    ("bf16_kt2_narrow", "bf16", 96, 3, 3, 4, 50, [2, 1], True, True, (2, 3, 3), "tc_bf16_narrow"),
    ("f32_kt2", "f32", 8, 8, 4, 5, 6, [1, 3], True, True, (2, 3, 3), "simt_f32"),
]


@pytest.mark.parametrize("case", EXTENTS, ids=[c[0] for c in EXTENTS])
def test_kernel_extents_match_oracle_elementwise(case):
    _check_small(*case[:10], k=case[10], kernel=case[11])


# ---------------------------------------------------------------- full-size workloads

def _gpu_inputs(wl, T=None, with_x=True):
    """Full tensors generated on the device from the shared counter-based generator."""
    T = T or wl.T
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    d = {}
    if with_x:
        d["x"] = native.fill_device(torch.empty((T, wl.H, wl.W, wl.Cin), dtype=dt, device="cuda"), wl.seed,
                                    synth.TID_X, wl.x)
    d["w"] = native.fill_device(torch.empty((wl.Cout, 3, 3, 3, wl.Cin), dtype=dt, device="cuda"), wl.seed,
                                synth.TID_W, wl.w)
    if wl.b is not None:
        d["b"] = native.fill_device(torch.empty((wl.Cout,), dtype=dt, device="cuda"), wl.seed, synth.TID_B, wl.b)
    if wl.r is not None:
        d["r"] = native.fill_device(torch.empty((T, wl.H, wl.W, wl.Cout), dtype=dt, device="cuda"), wl.seed,
                                    synth.TID_R, wl.r)
    return d


def _sample_points(wl, T, seams, rng, n_random):
    H, W = wl.H, wl.W
    pts = set()
    for _ in range(n_random):
        pts.add((int(rng.integers(T)), int(rng.integers(H)), int(rng.integers(W))))
    frames = sorted(f for f in ({0, 1, 2, T - 1} | set(seams) | set(s - 1 for s in seams)) if 0 <= f < T)
    cols = sorted({0, 1, W - 2, W - 1} | {c for c in (127, 128, 129, 159, 160, 161, 255, 256) if c < W})
    rows = sorted({0, 1, H - 2, H - 1} | {H // 2})
    for t in frames:
        for h in rows:
            for w in cols:
                pts.add((t, h, w))
        for _ in range(24):
            pts.add((t, int(rng.integers(H)), int(rng.integers(W))))
    return np.array(sorted(pts), dtype=np.int64)


def _windows(wl, pts):
    """Input values around each point, from the host copy of the generator (out-of-video entries
    are computed at clamped coordinates and ignored by the oracle)."""
    H, W, C = wl.H, wl.W, wl.Cin
    dt_, dh_, dw_ = np.meshgrid(np.arange(3), np.arange(3), np.arange(3), indexing="ij")
    t = np.maximum(pts[:, 0, None, None, None] + dt_ - 2, 0)
    h = np.clip(pts[:, 1, None, None, None] + dh_ - 1, 0, H - 1)
    w = np.clip(pts[:, 2, None, None, None] + dw_ - 1, 0, W - 1)
    base = ((t * H + h) * W + w) * C
    e = base[..., None] + np.arange(C)
    raw = native.values_host(wl.seed, synth.TID_X, wl.x, e, wl.dtype)
    return to_f64(raw, wl.dtype)


def _oracle_at(wl, T, pts):
    e_w = synth.dense_index((wl.Cout, 3, 3, 3, wl.Cin))
    w = to_f64(native.values_host(wl.seed, synth.TID_W, wl.w, e_w, wl.dtype), wl.dtype)
    b = None if wl.b is None else to_f64(native.values_host(wl.seed, synth.TID_B, wl.b,
                                                            np.arange(wl.Cout), wl.dtype), wl.dtype)
    r = None
    if wl.r is not None:
        e_r = (((pts[:, 0] * wl.H + pts[:, 1]) * wl.W + pts[:, 2]) * wl.Cout)[:, None] + np.arange(wl.Cout)
        r = to_f64(native.values_host(wl.seed, synth.TID_R, wl.r, e_r, wl.dtype), wl.dtype)
    return oracle.conv_points((T, wl.H, wl.W), pts, _windows(wl, pts), w, b, r)


def _gather(y, pts):
    idx = torch.from_numpy(pts).to(y.device)
    return from_device(y[idx[:, 0], idx[:, 1], idx[:, 2]])


FULL = ["c96_residual", "c192", "c384", "c384_to_192"]


def _host_tensor(wl, tid, dist, shape):
    """A tensor of the workload from the host side of the shared generator (never from the device)."""
    return to_f64(native.values_host(wl.seed, tid, dist, synth.dense_index(shape), wl.dtype), wl.dtype)


@pytest.mark.parametrize("name", ["c96_residual", "c192", "c384"])
def test_full_frame_compare_at_reduced_T(name):
    """Every output of the full-resolution layer for 8 frames (two 4-frame chunks), against the
    oracle evaluated on the whole sequence."""
    wl = synth.WORKLOADS[name]
    T = 8
    d = _gpu_inputs(wl, T=T)
    plan = cc3d.CausalConv3dPlan(wl.Cin, wl.Cout, wl.H, wl.W, dtype=wl.dtype)
    y, _ = run_chunks(plan, d["x"], d["w"], d.get("b"), d.get("r"), [4, 4])
    assert plan.status() == 0
    x = _host_tensor(wl, synth.TID_X, wl.x, (T, wl.H, wl.W, wl.Cin))
    w = _host_tensor(wl, synth.TID_W, wl.w, (wl.Cout, 3, 3, 3, wl.Cin))
    b = _host_tensor(wl, synth.TID_B, wl.b, (wl.Cout,)) if wl.b is not None else None
    r = _host_tensor(wl, synth.TID_R, wl.r, (T, wl.H, wl.W, wl.Cout)) if wl.r is not None else None
    ref = oracle.conv_whole(x, w, b, r)
    err = np.abs(from_device(y) - ref).max()
    tol = tolerance(wl.dtype, ref)
    assert err <= tol, (name, err, tol)
    y2, _ = run_chunks(plan, d["x"], d["w"], d.get("b"), d.get("r"), [T])
    assert torch.equal(y2, y)
    plan.close()


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled(name):
    wl = synth.WORKLOADS[name]
    d = _gpu_inputs(wl)
    plan = cc3d.CausalConv3dPlan(wl.Cin, wl.Cout, wl.H, wl.W, dtype=wl.dtype)
    y, _ = run_chunks(plan, d["x"], d["w"], d.get("b"), d.get("r"), list(wl.chunks))
    assert plan.status() == 0
    seams = np.cumsum(wl.chunks)[:-1].tolist()
    rng = np.random.default_rng(wl.seed)
    n_random = int(min(4096, 6e6 / (27 * wl.Cin)))
    pts = _sample_points(wl, wl.T, seams, rng, n_random)
    ref = _oracle_at(wl, wl.T, pts)
    got = _gather(y, pts)
    err = np.abs(got - ref).max()
    tol = tolerance(wl.dtype, ref)
    assert err <= tol, (name, err, tol, len(pts))
    # the same video cut differently gives the same bits
    for parts in compositions_sample():
        y2, _ = run_chunks(plan, d["x"], d["w"], d.get("b"), d.get("r"), parts)
        assert torch.equal(y2, y), (name, parts)
    plan.close()


@pytest.mark.parametrize("name", ["sr96", "sr_head3"])
def test_super_resolution_stream_sampled(name):
    """The 361-frame 1440x2560 stream in 90 chunks of 4 and a last chunk of 1, the cache carried by
    the library from chunk to chunk; outputs sampled in several chunks including the last."""
    wl = synth.WORKLOADS[name]
    d = _gpu_inputs(wl, with_x=False)
    plan = cc3d.CausalConv3dPlan(wl.Cin, wl.Cout, wl.H, wl.W, dtype=wl.dtype)
    x = torch.empty((4, wl.H, wl.W, wl.Cin), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((4, wl.H, wl.W, wl.Cout), dtype=torch.bfloat16, device="cuda")
    caches = [plan.new_cache(), plan.new_cache()]
    frame = wl.H * wl.W * wl.Cin
    check = {0, 1, 45, len(wl.chunks) - 2, len(wl.chunks) - 1}
    rng = np.random.default_rng(wl.seed)
    got_all, pts_all = [], []
    s = 0
    for k, c in enumerate(wl.chunks):
        xc, yc = x[:c], y[:c]
        native.fill_device(xc, wl.seed, synth.TID_X, wl.x, offset=s * frame)
        plan.forward_chunk(xc, d["w"], d.get("b"), None, caches[k % 2] if k else None, caches[(k + 1) % 2], yc)
        if k in check:
            pts = _sample_points(wl, c, [], rng, 160)
            got_all.append(_gather(yc, pts))
            pts[:, 0] += s
            pts_all.append(pts)
        s += c
    assert s == wl.T
    assert plan.status() == 0
    pts = np.concatenate(pts_all)
    ref = _oracle_at(wl, wl.T, pts)
    got = np.concatenate(got_all)
    err = np.abs(got - ref).max()
    assert err <= tolerance(wl.dtype, ref), (name, err, tolerance(wl.dtype, ref))
    # the final history is the video's last two input frames
    last = caches[len(wl.chunks) % 2]
    exp = torch.empty_like(last)
    native.fill_device(exp, wl.seed, synth.TID_X, wl.x, offset=(wl.T - 2) * frame)
    assert torch.equal(last, exp)
    plan.close()


# ---------------------------------------------------------------- edge cases and contract

def _tiny_bf16(T=4, H=6, W=40, C=32, residual=True, seed=7):
    raw = small_inputs(C, C, T, H, W, "bf16", seed, True, residual)
    return raw, {k: to_device(v, "bf16") for k, v in raw.items()}, cc3d.CausalConv3dPlan(C, C, H, W)


def test_empty_chunk_passes_history_through():
    raw, d, plan = _tiny_bf16()
    cin = d["x"][:2].clone()
    cout = plan.new_cache()
    cc3d.cc3d_forward_chunk(plan.handle, 0, None, d["w"], d["b"], None, cin, cout, None)
    torch.cuda.synchronize()
    assert torch.equal(cout, cin)
    cc3d.cc3d_forward_chunk(plan.handle, 0, None, d["w"], d["b"], None, None, cout, None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(cout.float()) == 0
    assert plan.status() == 0


def test_zero_history_buffer_equals_null_history():
    raw, d, plan = _tiny_bf16()
    y0, _ = run_chunks(plan, d["x"], d["w"], d["b"], d["r"], [2, 2])
    y1, _ = run_chunks(plan, d["x"], d["w"], d["b"], d["r"], [2, 2], zero_cache_first=True)
    assert torch.equal(y0, y1)


def test_single_frame_chunk_takes_history_from_cache():
    raw, d, plan = _tiny_bf16()
    _, caches = run_chunks(plan, d["x"], d["w"], d["b"], d["r"], [3, 1])
    assert torch.equal(caches[1][0], d["x"][2]) and torch.equal(caches[1][1], d["x"][3])
    _, caches = run_chunks(plan, d["x"][:1], d["w"], d["b"], d["r"][:1], [1])
    assert torch.count_nonzero(caches[0][0].float()) == 0 and torch.equal(caches[0][1], d["x"][0])


def test_optional_bias_and_residual():
    raw, d, plan = _tiny_bf16(residual=False)
    y, _ = run_chunks(plan, d["x"], d["w"], None, None, [4])
    ref = oracle.conv_whole(to_f64(raw["x"], "bf16"), to_f64(raw["w"], "bf16"))
    assert np.abs(from_device(y) - ref).max() <= tolerance("bf16", ref)


def test_rejected_calls_leave_buffers_untouched():
    raw, d, plan = _tiny_bf16()
    y = torch.full((4, 6, 40, 32), 7.0, dtype=torch.bfloat16, device="cuda")
    cout = torch.full((2, 6, 40, 32), 5.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cc3d.CC3DError) as e:
        cc3d.cc3d_forward_chunk(plan.handle, 4, d["x"], d["w"], d["b"], None, None, d["x"][2:], y)
    assert e.value.code == 4
    with pytest.raises(cc3d.CC3DError) as e:
        cc3d.cc3d_forward_chunk(plan.handle, 4, d["x"], d["w"], d["b"], y, None, cout, y)
    assert e.value.code == 4
    host = torch.zeros((4, 6, 40, 32), dtype=torch.bfloat16).pin_memory()
    with pytest.raises(cc3d.CC3DError) as e:
        cc3d.cc3d_forward_chunk(plan.handle, 4, host.data_ptr(), d["w"], d["b"], None, None, cout, y)
    assert e.value.code == 8
    torch.cuda.synchronize()
    assert torch.all(y.float() == 7.0) and torch.all(cout.float() == 5.0)


def test_reset_zeroes_a_cache():
    _, _, plan = _tiny_bf16()
    c = torch.full((2, 6, 40, 32), 3.0, dtype=torch.bfloat16, device="cuda")
    plan.reset(c)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c.float()) == 0


def test_resume_from_a_saved_history_is_bit_identical():
    raw, d, plan = _tiny_bf16(T=6)
    y_ref, caches = run_chunks(plan, d["x"], d["w"], d["b"], d["r"], [2, 2, 2])
    saved = caches[1].cpu()  # history after chunk 2 (frames 2..3)
    plan.close()
    plan2 = cc3d.CausalConv3dPlan(32, 32, 6, 40)
    cin = saved.cuda()
    cout = plan2.new_cache()
    y3 = plan2.forward_chunk(d["x"][4:], d["w"], d["b"], d["r"][4:], cin, cout)
    assert torch.equal(y3, y_ref[4:])


def test_non_default_stream():
    raw, d, plan = _tiny_bf16()
    y_ref, _ = run_chunks(plan, d["x"], d["w"], d["b"], d["r"], [4])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y_s, _ = run_chunks(plan, d["x"], d["w"], d["b"], d["r"], [4], stream=s)
    s.synchronize()
    assert torch.equal(y_s, y_ref)


# one small plan of every tensor-core kernel family: (Cin, Cout, H, W, (kt, kh, kw), family)
FAMILIES = [
    (32, 32, 6, 40, (3, 3, 3), "tc_bf16"),
    (96, 96, 3, 256, (3, 3, 3), "tc_bf16_pair"),     # two-frame schedule
    (64, 192, 4, 128, (3, 3, 3), "tc_bf16_pair"),    # one-frame schedule (192 output channels)
    (96, 3, 6, 130, (3, 3, 3), "tc_bf16_head"),
    (96, 96, 5, 70, (3, 1, 1), "tc_bf16_stream"),
    (48, 3, 5, 40, (3, 3, 3), "tc_bf16_narrow"),
]


def _family_case(Cin, Cout, H, W, k, family, T=4):
    raw = small_inputs(Cin, Cout, T, H, W, "bf16", 7, True, True, k=k)
    d = {kk: to_device(v, "bf16") for kk, v in raw.items()}
    plan = cc3d.CausalConv3dPlan(Cin, Cout, H, W, *k)
    assert plan.kernel == family
    return d, plan


@pytest.mark.parametrize("case", FAMILIES, ids=["%s_%d" % (c[-1], c[1]) for c in FAMILIES])
def test_bounded_wait_times_out_and_the_context_survives(case):
    """The loader skips its first copy (test hook), a bounded wait runs out, the kernel records a
    timeout and every role leaves; the next call on the same context is correct."""
    d, plan = _family_case(*case)
    y_ref, _ = run_chunks(plan, d["x"], d["w"], d["b"], d["r"], [4])
    plan.set_wait_budget_ns(50_000_000)
    plan.set_fault(1)
    y = torch.empty_like(y_ref)
    cout = plan.new_cache()
    plan.forward_chunk(d["x"], d["w"], d["b"], d["r"], None, cout, y)
    assert plan.status() == 7
    plan.set_fault(0)
    y2, _ = run_chunks(plan, d["x"], d["w"], d["b"], d["r"], [4])
    assert plan.status() == 0
    assert torch.equal(y2, y_ref)
    plan.close()


@pytest.mark.parametrize("case", FAMILIES, ids=["%s_%d" % (c[-1], c[1]) for c in FAMILIES])
def test_injected_host_encode_failure_launches_nothing(case):
    d, plan = _family_case(*case)
    plan.set_fault(2)
    y = torch.full((4, case[2], case[3], case[1]), 9.0, dtype=torch.bfloat16, device="cuda")
    cout = plan.new_cache()
    with pytest.raises(cc3d.CC3DError) as e:
        plan.forward_chunk(d["x"], d["w"], d["b"], d["r"], None, cout, y)
    assert e.value.code == 5
    torch.cuda.synchronize()
    assert torch.all(y.float() == 9.0)
    plan.close()


def test_bounded_wait_times_out_in_the_fused_upsample_and_the_context_survives():
    raw = small_inputs(32, 64, 4, 4, 40, "bf16", 8, True, False)
    d = {kk: to_device(v, "bf16") for kk, v in raw.items()}
    plan = cc3d.Upsample2xConvPlan(32, 64, 4, 40, 3)
    assert plan.kernel == "tc_bf16_up2"
    y_ref, _ = run_chunks(plan, d["x"], d["w"], d["b"], None, [4])
    plan.set_wait_budget_ns(50_000_000)
    plan.set_fault(1)
    y = torch.empty_like(y_ref)
    plan.forward_chunk(d["x"], d["w"], d["b"], None, None, plan.new_cache(), y)
    assert plan.status() == 7
    plan.set_fault(0)
    y2, _ = run_chunks(plan, d["x"], d["w"], d["b"], None, [4])
    assert plan.status() == 0
    assert torch.equal(y2, y_ref)
    plan.close()


# ---------------------------------------------------------------- fused nearest-2x upsampling

UP2 = [
    # name, Cin, Cout, T, H, W (source), chunks, bias, residual, kt
    ("up2_c64", 64, 64, 4, 5, 33, [2, 2], True, True, 3),
    ("up2_c96", 96, 96, 3, 4, 50, [1, 2], True, False, 3),
    ("up2_cout192_blocks", 32, 192, 3, 3, 20, [3], True, True, 3),
    ("up2_spatial_only", 32, 32, 2, 6, 70, [1, 1], True, False, 1),
    ("up2_kt2_wide_rows", 32, 64, 3, 2, 128, [2, 1], False, True, 2),
    # 16-channel blocks: one row group of four 96-channel classes, and four row groups of
    # 16-channel classes
    ("up2_cb16_c96", 16, 96, 3, 4, 40, [2, 1], True, True, 3),
    ("up2_cb16_c16", 16, 16, 3, 5, 70, [1, 2], True, False, 3),
]


@pytest.mark.parametrize("case", UP2, ids=[c[0] for c in UP2])
def test_upsample_conv_matches_oracle_and_the_materialised_upsample(case):
    name, Cin, Cout, T, H, W, chunks, bias, residual, kt = case
    seed = 300 + len(name)
    raw = small_inputs(Cin, Cout, T, H, W, "bf16", seed, bias, False, k=(kt, 3, 3))
    if residual:
        raw["r"] = synth.raw(seed, synth.TID_R, synth.Dist.normal(1.0),
                             synth.dense_index((T, 2 * H, 2 * W, Cout)), "bf16")
    dev = {kk: to_device(v, "bf16") for kk, v in raw.items()}
    plan = cc3d.Upsample2xConvPlan(Cin, Cout, H, W, kt)
    assert plan.kernel == "tc_bf16_up2"
    y, caches = run_chunks(plan, dev["x"], dev["w"], dev.get("b"), dev.get("r"), chunks)
    assert plan.status() == 0
    assert y.shape == (T, 2 * H, 2 * W, Cout)
    ref = oracle.conv_upsample2x_whole(to_f64(raw["x"], "bf16"), to_f64(raw["w"], "bf16"),
                                       to_f64(raw["b"], "bf16") if bias else None,
                                       to_f64(raw["r"], "bf16") if residual else None)
    err = np.abs(from_device(y) - ref).max()
    assert err <= tolerance("bf16", ref), (name, err)
    # the history holds the last kt-1 *source* frames
    end = 0
    for c, cache in zip(chunks, caches):
        end += c
        assert cache.shape == (kt - 1, H, W, Cin)
        for j in range(kt - 1):
            src = end - (kt - 1) + j
            exp = dev["x"][src] if src >= 0 else torch.zeros_like(dev["x"][0])
            assert torch.equal(cache[j], exp)
    for alt in ([T], [1] * T):
        y2, _ = run_chunks(plan, dev["x"], dev["w"], dev.get("b"), dev.get("r"), alt)
        assert torch.equal(y2, y), (name, alt)
    # the same products in the same order as a plain plan on the stored upsampled frames
    u = dev["x"].repeat_interleave(2, dim=1).repeat_interleave(2, dim=2)
    plain = cc3d.CausalConv3dPlan(Cin, Cout, 2 * H, 2 * W, kt, 3, 3)
    y_plain, _ = run_chunks(plain, u, dev["w"], dev.get("b"), dev.get("r"), chunks)
    assert plain.status() == 0
    assert torch.equal(y, y_plain), (name, plain.kernel, int((y != y_plain).sum()))
    plain.close()
    plan.close()


# ---------------------------------------------------------------- two-frame SM-pair schedule

TSTACK = [
    # name, Cin, Cout, T, H, W, chunks, bias, residual, kt
    ("c96_residual_like", 96, 96, 7, 5, 256, [4, 3], True, True, 3),
    ("c64_two_and_four_frame_chunks", 64, 64, 6, 3, 128, [2, 4], True, False, 3),
    ("kt2_memory_block", 96, 96, 7, 3, 128, [4, 3], True, True, 2),
    ("cout128_full_tensor_memory", 32, 128, 5, 4, 128, [5], False, True, 3),
    # 5 frames = 3 frame pairs (the last one half outside the chunk) on one row: 3 tiles, so the
    # second pair of blocks also holds a phantom tile
    ("odd_pairs_and_phantom_tile", 32, 32, 7, 1, 128, [5, 2], True, True, 3),
]


@pytest.mark.parametrize("case", TSTACK, ids=[c[0] for c in TSTACK])
def test_two_frame_pair_schedule_is_bit_identical_to_the_one_frame_schedule(case):
    """Chunks of two or more frames on SM pairs stack two output frames into N; the one-frame pair
    schedule (chosen for 1-frame chunks, or forced here through the plan's schedule knob) accumulates
    every output in the same order, so the two agree bit for bit, and both match the oracle."""
    name, Cin, Cout, T, H, W, chunks, bias, residual, kt = case
    raw = small_inputs(Cin, Cout, T, H, W, "bf16", 300 + len(name), bias, residual, k=(kt, 3, 3))
    dev = {kk: to_device(v, "bf16") for kk, v in raw.items()}
    plan = cc3d.CausalConv3dPlan(Cin, Cout, H, W, kt, 3, 3)
    assert plan.kernel == "tc_bf16_pair"
    y2, c2 = run_chunks(plan, dev["x"], dev["w"], dev.get("b"), dev.get("r"), chunks)
    assert plan.status() == 0
    plan.set_schedule("two_frame", 0)
    assert plan.describe(chunks[0], residual)["kernel"] == "tc2_bf16_kernel"
    y1, c1 = run_chunks(plan, dev["x"], dev["w"], dev.get("b"), dev.get("r"), chunks)
    assert plan.status() == 0
    plan.set_schedule("two_frame", -1)
    assert torch.equal(y2, y1), name
    for a, b in zip(c2, c1):
        assert torch.equal(a, b), name
    ref = oracle.conv_whole(to_f64(raw["x"], "bf16"), to_f64(raw["w"], "bf16"),
                            to_f64(raw["b"], "bf16") if bias else None,
                            to_f64(raw["r"], "bf16") if residual else None)
    err = np.abs(from_device(y2) - ref).max()
    assert err <= tolerance("bf16", ref), (name, err)
    # and across chunkings (1-frame chunks run the one-frame schedule)
    for alt in ([T], [1] * T, [2] * (T // 2) + [1] * (T % 2)):
        y3, _ = run_chunks(plan, dev["x"], dev["w"], dev.get("b"), dev.get("r"), alt)
        assert torch.equal(y3, y2), (name, alt)
    assert plan.status() == 0
    plan.close()


ALIGN16 = [
    # Cin, Cout, T, H, W, (kt, kh, kw), chunk, family
    (96, 96, 4, 3, 128, (3, 3, 3), 4, "tc_bf16_pair"),      # two-frame schedule
    (96, 96, 1, 3, 128, (3, 3, 3), 1, "tc_bf16_pair"),      # one-frame schedule
    (64, 64, 3, 4, 40, (3, 3, 3), 3, "tc_bf16"),            # one SM
    (32, 384, 2, 3, 20, (3, 3, 3), 2, "tc_bf16"),           # channel blocks
    (96, 96, 3, 2, 70, (3, 1, 1), 3, "tc_bf16_stream"),
]


@pytest.mark.parametrize("case", ALIGN16, ids=["%s_T%d_c%d" % (c[-1], c[2], c[1]) for c in ALIGN16])
def test_outputs_and_residual_only_16_byte_aligned(case):
    """y and the residual 16 but not 32 bytes aligned: the epilogues take their 16-byte accesses
    and the result is bit-identical to the one with 32-byte aligned buffers."""
    Cin, Cout, T, H, W, k, chunk, family = case
    raw = small_inputs(Cin, Cout, T, H, W, "bf16", 77, True, True, k=k)
    dev = {kk: to_device(v, "bf16") for kk, v in raw.items()}
    plan = cc3d.CausalConv3dPlan(Cin, Cout, H, W, *k)
    assert plan.kernel == family
    y_ref, _ = run_chunks(plan, dev["x"], dev["w"], dev["b"], dev["r"], [chunk] * (T // chunk))
    n = T * H * W * Cout
    rbuf = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
    ybuf = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
    r16 = rbuf[8:].view(T, H, W, Cout)
    y16 = ybuf[8:].view(T, H, W, Cout)
    assert r16.data_ptr() % 32 == 16 and y16.data_ptr() % 32 == 16
    r16.copy_(dev["r"])
    cache = [None, plan.new_cache(), plan.new_cache()]
    for j in range(T // chunk):
        s0 = j * chunk
        plan.forward_chunk(dev["x"][s0:s0 + chunk], dev["w"], dev["b"], r16[s0:s0 + chunk],
                           cache[j % 2 + 1] if j else None, cache[(j + 1) % 2 + 1], y16[s0:s0 + chunk])
    assert plan.status() == 0
    assert torch.equal(y16, y_ref)
    plan.close()


@pytest.mark.parametrize("shape", [(192, 192, 5, 6, 64), (384, 192, 4, 5, 40), (64, 256, 3, 7, 100)],
                         ids=["c192_like", "c384_to_192_like", "c64_to_256"])
def test_split_tail_tiles_are_bit_identical(shape):
    """A short last wave of two-row-group tiles is split into one-row-group units that both MMA
    warps compute, on half of the output channels each (at these sizes every tile is split).
    Each output keeps its MMAs and their order, so the result equals the unsplit launch bit for
    bit, and the oracle within tolerance."""
    Cin, Cout, T, H, W = shape
    raw = small_inputs(Cin, Cout, T, H, W, "bf16", 400 + Cin, True, True)
    dev = {kk: to_device(v, "bf16") for kk, v in raw.items()}
    plan = cc3d.CausalConv3dPlan(Cin, Cout, H, W)
    assert plan.kernel == "tc_bf16"
    y_split, c_split = run_chunks(plan, dev["x"], dev["w"], dev["b"], dev["r"], [T - 1, 1])
    assert plan.status() == 0
    plan.set_schedule("split_tail", 0)
    y_whole, c_whole = run_chunks(plan, dev["x"], dev["w"], dev["b"], dev["r"], [T - 1, 1])
    assert plan.status() == 0
    plan.set_schedule("split_tail", -1)
    assert torch.equal(y_split, y_whole)
    assert all(torch.equal(a, b) for a, b in zip(c_split, c_whole))
    ref = oracle.conv_whole(to_f64(raw["x"], "bf16"), to_f64(raw["w"], "bf16"), to_f64(raw["b"], "bf16"),
                            to_f64(raw["r"], "bf16"))
    assert np.abs(from_device(y_split) - ref).max() <= tolerance("bf16", ref)
    plan.close()
