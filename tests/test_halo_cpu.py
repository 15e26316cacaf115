"""The temporal split with the causal halo exchange (chunked_causal_convolution_gb300.halo), run as
gloo ranks on the CPU (127.0.0.1).

Each rank owns a contiguous frame range of every wave; before every causal layer it receives the
kt - 1 input frames before its range from the previous rank ("SwiftVR Inference Optimization",
section "ReAE: Causal Halo Exchange").  The layers here compute with the fp64 oracle's chunk form
(a test stand-in for the device layers), so the exchange and the wave bookkeeping are checked on
their own: every received history must be the video's frames before the range (zeros before the
video), and every rank's output must equal the whole-video oracle exactly (the oracle's chunked
form equals its whole-sequence form exactly).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (Cin, Cout, kt): a 3-frame history layer, a MemoryBlock-like 1-frame history layer, a pointwise one
LAYERS = [(3, 4, 3), (4, 2, 2), (2, 3, 1)]
H, W = 4, 5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _video(T):
    sys.path.insert(0, ROOT)
    import synth
    e = synth.dense_index
    x = synth.bf16_bits_to_f64(synth.raw(21, synth.TID_X, synth.Dist.normal(1.0), e((T, H, W, LAYERS[0][0])), "bf16"))
    ws, bs = [], []
    for j, (ci, co, kt) in enumerate(LAYERS):
        ws.append(synth.bf16_bits_to_f64(synth.raw(30 + j, synth.TID_W, synth.Dist.normal(synth.fan_in_sigma(ci, kt, 3, 3)),
                                                   e((co, kt, 3, 3, ci)), "bf16")))
        bs.append(synth.bf16_bits_to_f64(synth.raw(30 + j, synth.TID_B, synth.Dist.uniform(-0.1, 0.1), e((co,)), "bf16")))
    return x, ws, bs


class OracleLayer:
    """A layer computed by the oracle's chunk form from the history the exchange delivered."""

    def __init__(self, w, b):
        self.w, self.b = w, b
        self.P = w.shape[1] - 1

    def __call__(self, x, history):
        import oracle
        if int(x.shape[0]) == 0:  # an empty range: no output frames (the history passes through the split)
            return torch.zeros((0,) + tuple(x.shape[1:3]) + (self.w.shape[0],), dtype=torch.float64)
        y, _ = oracle.conv_chunk(x.numpy(), self.w, self.b, None,
                                 None if history is None else history.numpy(), nthreads=1)
        return torch.from_numpy(y)


def _rank_main(rank, world, port, per_wave, waves, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    from chunked_causal_convolution_gb300 import halo
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        wave_len = sum(per_wave)
        T = wave_len * waves
        x, ws, bs = _video(T)
        # the whole video through the stack, and every layer's input
        ref_in, cur = [], x
        for w, b in zip(ws, bs):
            ref_in.append(cur)
            cur = oracle.conv_whole(cur, w, b, nthreads=1)
        ref = cur
        split = halo.TimeSplit([OracleLayer(w, b) for w, b in zip(ws, bs)])
        starts = np.cumsum([0] + list(per_wave))
        errs, hist_ok = [], True
        for wv in range(waves):
            s0 = wv * wave_len + int(starts[rank])
            s1 = s0 + per_wave[rank]
            y = split.forward(torch.from_numpy(x[s0:s1]))
            errs.append(float(np.abs(y.numpy() - ref[s0:s1]).max()) if s1 > s0 else 0.0)
            for j, (hist, (_, _, kt)) in enumerate(zip(split.last_histories, LAYERS)):
                P = kt - 1
                if P == 0:
                    hist_ok &= hist is None
                    continue
                exp = np.stack([ref_in[j][t] if t >= 0 else np.zeros_like(ref_in[j][0])
                                for t in range(s0 - P, s0)])
                hist_ok &= bool(np.array_equal(hist.numpy(), exp))
        out[rank] = (max(errs), hist_ok)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,per_wave,waves", [
    (2, [3, 3], 2),       # every range longer than the history
    (3, [1, 1, 2], 2),    # ranges shorter than the 2-frame history: the boundary chains through rank 1
    (2, [2, 1], 3),       # uneven ranges over three waves
    (3, [2, 0, 2], 2),    # an empty range: rank 1 passes rank 0's boundary straight on
    (4, [1, 0, 0, 2], 2), # two empty ranges in a row, and a 1-frame range before them
])
def test_time_split_over_gloo_ranks_equals_the_whole_video(world, per_wave, waves):
    sys.path.insert(0, ROOT)
    import oracle
    oracle.build()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), per_wave, waves, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == list(range(world))
    for r, (err, hist_ok) in res.items():
        assert err == 0.0, (r, err)
        assert hist_ok, r


def test_single_rank_carries_the_history_from_wave_to_wave():
    """Without a process group the split is one rank: successive forward calls continue the
    video (the history of each layer is carried), and reset starts a new one."""
    sys.path.insert(0, ROOT)
    import oracle
    from chunked_causal_convolution_gb300 import halo
    x, ws, bs = _video(7)
    ref = x
    for w, b in zip(ws, bs):
        ref = oracle.conv_whole(ref, w, b, nthreads=1)
    split = halo.TimeSplit([OracleLayer(w, b) for w, b in zip(ws, bs)])
    ys = [split.forward(torch.from_numpy(x[a:b])).numpy() for a, b in ((0, 3), (3, 4), (4, 7))]
    assert np.array_equal(np.concatenate(ys), ref)
    split.reset()
    assert np.array_equal(split.forward(torch.from_numpy(x[:3])).numpy(), ref[:3])


def test_frame_ranges_and_end_history():
    from chunked_causal_convolution_gb300 import halo
    assert halo.frame_ranges(10, 4) == [(0, 3), (3, 6), (6, 8), (8, 10)]
    assert halo.frame_ranges(2, 3) == [(0, 1), (1, 2), (2, 2)]
    with pytest.raises(ValueError):
        halo.frame_ranges(5, 0)
    hist = torch.arange(2 * 3).reshape(2, 3)
    x = torch.arange(100, 109).reshape(3, 3)
    assert torch.equal(halo.end_history(hist, x, 2), x[1:])
    assert torch.equal(halo.end_history(hist, x[:1], 2), torch.stack([hist[1], x[0]]))


def _exchange_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from chunked_causal_convolution_gb300 import halo
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        video = torch.arange(6 * world * 4, dtype=torch.float32).reshape(6 * world, 2, 2)
        x = video[6 * rank:6 * rank + 6].clone()
        h = halo.exchange(x, 2)
        exp = video[6 * rank - 2:6 * rank] if rank else torch.zeros(2, 2, 2)
        out[rank] = bool(torch.equal(h, exp))
    finally:
        dist.destroy_process_group()


def test_single_layer_exchange_over_gloo_ranks():
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_exchange_main, args=(3, _free_port(), out), nprocs=3, join=True)
        assert dict(out) == {0: True, 1: True, 2: True}


# ---------------------------------------------------------------- height split

HS_LAYERS = [(3, 4, 3, 3), (4, 2, 2, 3), (2, 3, 1, 1)]  # (Cin, Cout, kt, kh = kw)


def _band_video(T, H, W):
    sys.path.insert(0, ROOT)
    import synth
    e = synth.dense_index
    x = synth.bf16_bits_to_f64(synth.raw(41, synth.TID_X, synth.Dist.normal(1.0), e((T, H, W, HS_LAYERS[0][0])), "bf16"))
    ws, bs = [], []
    for j, (ci, co, kt, ks) in enumerate(HS_LAYERS):
        ws.append(synth.bf16_bits_to_f64(synth.raw(50 + j, synth.TID_W, synth.Dist.normal(synth.fan_in_sigma(ci, kt, ks, ks)),
                                                   e((co, kt, ks, ks, ci)), "bf16")))
        bs.append(synth.bf16_bits_to_f64(synth.raw(50 + j, synth.TID_B, synth.Dist.uniform(-0.1, 0.1), e((co,)), "bf16")))
    return x, ws, bs


class OracleBandLayer:
    """A layer on an extended band, computed by the oracle's chunk form; keeps its history."""

    def __init__(self, w, b):
        self.w, self.b = w, b
        self.P = w.shape[1] - 1
        self.halo = (w.shape[2] - 1) // 2
        self.last_history = None

    def __call__(self, x, history):
        import oracle
        y, cache = oracle.conv_chunk(x.numpy(), self.w, self.b, None,
                                     None if history is None else history.numpy(), nthreads=1)
        self.last_history = torch.from_numpy(cache)
        return torch.from_numpy(y)


def _height_main(rank, world, port, H, chunks, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    from chunked_causal_convolution_gb300 import halo
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        T, W = sum(chunks), 5
        x, ws, bs = _band_video(T, H, W)
        ref = x
        for w, b in zip(ws, bs):
            ref = oracle.conv_whole(ref, w, b, nthreads=1)
        a, b_ = halo.row_ranges(H, world)[rank]
        split = halo.HeightSplit([OracleBandLayer(w, b) for w, b in zip(ws, bs)])
        errs, gathered_ok, s = [], True, 0
        for c in chunks:
            y = split.forward(torch.from_numpy(x[s:s + c, a:b_]))
            errs.append(float(np.abs(y.numpy() - ref[s:s + c, a:b_]).max()))
            full = split.gather(y, H)
            gathered_ok &= bool(np.array_equal(full.numpy(), ref[s:s + c]))
            s += c
        out[rank] = (max(errs), gathered_ok)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,H,chunks", [(2, 7, [4, 2]), (3, 8, [1, 3, 2])])
def test_height_split_over_gloo_ranks_equals_the_whole_frame(world, H, chunks):
    sys.path.insert(0, ROOT)
    import oracle
    oracle.build()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_height_main, args=(world, _free_port(), H, chunks, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == list(range(world))
    for r, (err, gathered_ok) in res.items():
        assert err == 0.0, (r, err)
        assert gathered_ok, r


def test_band_extent():
    from chunked_causal_convolution_gb300 import halo
    assert [halo.band_extent(8, 3, r, 1) for r in range(3)] == [(0, 4), (2, 7), (5, 8)]
    assert halo.band_extent(8, 1, 0, 1) == (0, 8)
