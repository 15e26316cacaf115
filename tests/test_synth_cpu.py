"""CPU checks of the shared seeded input generator (no convolution arithmetic here)."""
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_matches_published_reference_outputs():
    for ln in open(os.path.join(GOLDEN, "splitmix64_reference.txt")):
        if not ln.strip() or ln.startswith("#"):
            continue
        seed, *outs = (int(v) for v in ln.split())
        s = np.array([seed], dtype=np.uint64)
        for n, exp in enumerate(outs, start=1):
            with np.errstate(over="ignore"):
                got = synth._mix64(s + np.uint64(n) * synth.GOLDEN)[0]
            assert int(got) == exp


def test_values_depend_only_on_global_index():
    d = synth.Dist.normal(1.0)
    T, H, W, C = 6, 3, 4, 5
    whole = synth.values(7, synth.TID_X, d, synth.dense_index((T, H, W, C)), "bf16")
    frame = H * W * C
    for t0, tn in [(0, 4), (4, 2), (2, 3), (5, 1)]:
        part = synth.values(7, synth.TID_X, d, synth.dense_index((tn, H, W, C), t0 * frame), "bf16")
        assert np.array_equal(part, whole[t0:t0 + tn])


def test_streams_differ_by_seed_and_tensor_id():
    e = synth.dense_index((1000,))
    d = synth.Dist.normal(1.0)
    a = synth.values_f32(1, 0, synth.NORMAL, 0.0, 1.0, e)
    assert not np.array_equal(a, synth.values_f32(2, 0, synth.NORMAL, 0.0, 1.0, e))
    assert not np.array_equal(a, synth.values_f32(1, 1, synth.NORMAL, 0.0, 1.0, e))
    assert np.array_equal(synth.values(1, 0, d, e, "f32"), a.astype(np.float64))


def test_normal_and_uniform_moments_and_support():
    e = synth.dense_index((200000,))
    z = synth.values_f32(3, 0, synth.NORMAL, 0.0, 1.0, e).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert z.min() >= -6.0 and z.max() <= 6.0
    # Irwin-Hall(12) - 6 has excess kurtosis -0.1 (a normal has 0)
    k = ((z - z.mean()) ** 4).mean() / z.var() ** 2 - 3.0
    assert abs(k + 0.1) < 0.05
    s = synth.values_f32(3, 0, synth.NORMAL, 0.0, 0.25, e).astype(np.float64)
    assert abs(s.std() - 0.25) < 0.003
    u = synth.values_f32(4, 2, synth.UNIFORM, -0.1, 0.1, e).astype(np.float64)
    assert u.min() >= -0.1 and u.max() < 0.1 and abs(u.mean()) < 0.002
    assert abs(u.std() - 0.2 / np.sqrt(12)) < 0.002


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 0.0], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(f)
    back = synth.bf16_bits_to_f64(bits)
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1); 1+3*2^-8 ties -> 1+2^-6 (even)
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 0.0]


def test_workload_recipes():
    wl = synth.WORKLOADS["c96_residual"]
    assert wl.chunks == (4,) * 6 and wl.r is not None
    assert abs(wl.flops - 2 * 96 * 96 * 27 * 24 * 360 * 640) < 1
    sr = synth.WORKLOADS["sr96"]
    assert sum(sr.chunks) == 361 and sr.chunks[-1] == 1 and len(sr.chunks) == 91
