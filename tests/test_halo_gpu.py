"""The time-split runner with the library's layers on one GPU (a single rank: the exchange is
the hand-over of each layer's history from one wave to the next): a stack of layers run wave by
wave through halo.TimeSplit equals the plain chunk loop over the whole video bit for bit (the
library's result does not depend on where the video is cut), and each layer of that loop is within
tolerance of the oracle on the bf16 input it read."""
import numpy as np
import pytest
import torch

import chunked_causal_convolution_gb300 as cc3d
import oracle
from chunked_causal_convolution_gb300 import halo
from tests.helpers import from_device, run_chunks, small_inputs, to_device, to_f64, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_waves_through_the_time_split_equal_the_chunk_loop():
    T, H, W = 11, 5, 128
    spec = [(96, 96, 3), (96, 64, 2), (64, 3, 3)]  # SM-pair layer, MemoryBlock-like layer, narrow head
    raw = small_inputs(96, 96, T, H, W, "bf16", 600, bias=True)
    x = to_device(raw["x"], "bf16")
    layers, plans, params = [], [], []
    for j, (ci, co, kt) in enumerate(spec):
        p = small_inputs(ci, co, 1, 1, 1, "bf16", 610 + j, bias=True, k=(kt, 3, 3))
        w, b = to_device(p["w"], "bf16"), to_device(p["b"], "bf16")
        plan = cc3d.CausalConv3dPlan(ci, co, H, W, kt, 3, 3)
        plans.append(plan)
        params.append((w, b, p))
        layers.append(halo.ChunkedLayer(plan, w, b, chunk=4))
    split = halo.TimeSplit(layers)
    ys = [split.forward(x[a:b]) for a, b in ((0, 5), (5, 6), (6, 11))]
    y_split = torch.cat(ys)
    # the same stack, each layer as one chunk loop over the whole video
    cur, outs = x, []
    for plan, (w, b, _) in zip(plans, params):
        cur, _ = run_chunks(plan, cur, w, b, None, [4, 4, 3])
        outs.append(cur)
    assert all(p.status() == 0 for p in plans)
    assert torch.equal(y_split, cur)
    # every layer against the oracle on the bf16 input it read (the previous layer's stored output)
    inp = to_f64(raw["x"], "bf16")
    for j, (w, b, p) in enumerate(params):
        ref = oracle.conv_whole(inp, to_f64(p["w"], "bf16"), to_f64(p["b"], "bf16"))
        got = from_device(outs[j])
        err = np.abs(got - ref).max()
        assert err <= tolerance("bf16", ref), (j, err)
        inp = got
    for plan in plans:
        plan.close()



@pytest.mark.parametrize("world", [2, 3])
def test_bands_of_the_height_split_equal_the_whole_frame(world):
    """Every rank's layer run on its band extended by the halo rows (as halo.HeightSplit arranges
    it, with the rank's own history carried from chunk to chunk) gives, for the band's own rows,
    exactly the bits of the whole-frame chunk loop: every output's accumulation order does not
    depend on the frame's height.  The ranks run one after another on one GPU, layer by layer (the
    layer's input rows for every band come from the previous layer's output, which is what the
    exchange delivers); the exchange itself is tested over gloo ranks."""
    T, H, W, chunks = 6, 11, 128, [4, 2]
    spec = [(96, 96, 3), (96, 32, 2), (32, 3, 3)]  # SM pairs, MemoryBlock-like, narrow head
    x = to_device(small_inputs(96, 96, T, H, W, "bf16", 640, bias=False)["x"], "bf16")
    cur = x
    for j, (ci, co, kt) in enumerate(spec):
        p = small_inputs(ci, co, 1, 1, 1, "bf16", 650 + j, bias=True, k=(kt, 3, 3))
        w, b = to_device(p["w"], "bf16"), to_device(p["b"], "bf16")
        whole = cc3d.CausalConv3dPlan(ci, co, H, W, kt, 3, 3)
        ref, _ = run_chunks(whole, cur, w, b, None, chunks)
        bands = []
        for r in range(world):
            a, b_ = halo.row_ranges(H, world)[r]
            e0, e1 = halo.band_extent(H, world, r, 1)
            plan = cc3d.CausalConv3dPlan(ci, co, e1 - e0, W, kt, 3, 3)
            layer = halo.ChunkedLayer(plan, w, b)
            hist, outs, s0 = None, [], 0
            for c in chunks:
                outs.append(layer(cur[s0:s0 + c, e0:e1].contiguous(), hist))
                hist = layer.last_history
                s0 += c
            assert plan.status() == 0
            bands.append(torch.cat(outs)[:, a - e0:b_ - e0])
            plan.close()
        assert torch.equal(torch.cat(bands, 1), ref), (world, j)
        whole.close()
        cur = ref
