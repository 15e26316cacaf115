"""CUDA-graph replay of a chunk's layer sequence through the C ABI.

A chunk of the super-resolution output stage runs two layers: a 3x3x3 conv (with its own
history) feeding the 3-channel head (with another).  The sequence is captured once per cache
parity into a CUDA graph over fixed device buffers; a video is then streamed by copying each
chunk into the input buffer and replaying.  Outputs and histories must be bit-identical to the
eager chunk loop.
"""
import numpy as np
import pytest
import torch

import chunked_causal_convolution_gb300 as cc3d
import oracle
from tests.helpers import from_device, small_inputs, to_device, to_f64, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _layers():
    T, H, W, C = 8, 6, 136, 32
    a = small_inputs(C, C, T, H, W, "bf16", 71, bias=True, residual=False)
    h = small_inputs(C, 3, T, H, W, "bf16", 72, bias=True, residual=False)
    return T, H, W, C, a, h


def test_graph_replay_of_a_two_layer_chunk_is_bit_identical():
    T, H, W, C, a, h = _layers()
    Tc = 2
    x = to_device(a["x"], "bf16")
    w1, b1 = to_device(a["w"], "bf16"), to_device(a["b"], "bf16")
    w2, b2 = to_device(h["w"], "bf16"), to_device(h["b"], "bf16")
    conv = cc3d.CausalConv3dPlan(C, C, H, W)
    head = cc3d.CausalConv3dPlan(C, 3, H, W)
    assert head.kernel == "tc_bf16_head"

    # eager reference: chunk loop with ping-pong histories for both layers
    c1 = [conv.new_cache(), conv.new_cache()]
    c2 = [head.new_cache(), head.new_cache()]
    ys = []
    for k in range(T // Tc):
        xk = x[k * Tc:(k + 1) * Tc]
        mid = conv.forward_chunk(xk, w1, b1, None, c1[k % 2] if k else None, c1[(k + 1) % 2])
        ys.append(head.forward_chunk(mid, w2, b2, None, c2[k % 2] if k else None, c2[(k + 1) % 2]))
    y_eager = torch.cat(ys)
    torch.cuda.synchronize()
    assert conv.status() == 0 and head.status() == 0

    # graphs: fixed input / intermediate / output buffers, one graph per cache parity
    xs = torch.empty((Tc, H, W, C), dtype=torch.bfloat16, device="cuda")
    mid = torch.empty((Tc, H, W, C), dtype=torch.bfloat16, device="cuda")
    ys_buf = torch.empty((Tc, H, W, 3), dtype=torch.bfloat16, device="cuda")
    g1 = [conv.new_cache(), conv.new_cache()]
    g2 = [head.new_cache(), head.new_cache()]
    stream = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(stream):
        for parity in range(2):
            # warm the calls up outside the capture (first-use device queries happen there)
            conv.forward_chunk(xs, w1, b1, None, g1[parity], g1[1 - parity], mid, stream=stream)
            head.forward_chunk(mid, w2, b2, None, g2[parity], g2[1 - parity], ys_buf, stream=stream)
        stream.synchronize()
        for parity in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                conv.forward_chunk(xs, w1, b1, None, g1[parity], g1[1 - parity], mid, stream=stream)
                head.forward_chunk(mid, w2, b2, None, g2[parity], g2[1 - parity], ys_buf, stream=stream)
            graphs.append(g)
    # the first chunk starts from zero histories: reset the buffers the parity-0 graph reads
    conv.reset(g1[0])
    head.reset(g2[0])
    outs = []
    for k in range(T // Tc):
        xs.copy_(x[k * Tc:(k + 1) * Tc])
        graphs[k % 2].replay()
        outs.append(ys_buf.clone())
    torch.cuda.synchronize()
    assert conv.status() == 0 and head.status() == 0
    y_graph = torch.cat(outs)
    assert torch.equal(y_graph, y_eager)
    last = (T // Tc) % 2
    assert torch.equal(g1[last], c1[last]) and torch.equal(g2[last], c2[last])

    # and the eager result itself is the oracle's two-layer composition (bf16 intermediate)
    mid_ref = oracle.conv_whole(to_f64(a["x"], "bf16"), to_f64(a["w"], "bf16"), to_f64(a["b"], "bf16"))
    mid_gpu = torch.cat([conv.forward_chunk(x[k * Tc:(k + 1) * Tc], w1, b1, None,
                                            c1[k % 2] if k else None, c1[(k + 1) % 2]) for k in range(T // Tc)])
    assert np.abs(from_device(mid_gpu) - mid_ref).max() <= tolerance("bf16", mid_ref)
    y_ref = oracle.conv_whole(from_device(mid_gpu), to_f64(h["w"], "bf16"), to_f64(h["b"], "bf16"))
    assert np.abs(from_device(y_eager) - y_ref).max() <= tolerance("bf16", y_ref)
    conv.close()
    head.close()


@pytest.mark.parametrize("Tc", [2, 1])
def test_graph_replay_of_sm_pair_chunks_with_the_side_stream_copy(Tc):
    """SM-pair layers move part of the history on a copy engine through a side stream forked from
    and joined to the caller's stream (all of it for 1-frame chunks, one frame of it for 2-frame
    chunks).  Captured into CUDA graphs and replayed, outputs and histories are bit-identical to
    the eager chunk loop."""
    T, H, W, C = 6, 3, 128, 64
    a = small_inputs(C, C, T, H, W, "bf16", 81, bias=True, residual=True)
    x, r = to_device(a["x"], "bf16"), to_device(a["r"], "bf16")
    w, b = to_device(a["w"], "bf16"), to_device(a["b"], "bf16")
    plan = cc3d.CausalConv3dPlan(C, C, H, W)
    assert plan.kernel == "tc_bf16_pair"
    c = [plan.new_cache(), plan.new_cache()]
    ys = []
    for k in range(T // Tc):
        ys.append(plan.forward_chunk(x[k * Tc:(k + 1) * Tc], w, b, r[k * Tc:(k + 1) * Tc],
                                     c[k % 2] if k else None, c[(k + 1) % 2]))
    y_eager = torch.cat(ys)
    torch.cuda.synchronize()
    assert plan.status() == 0

    xs = torch.empty((Tc, H, W, C), dtype=torch.bfloat16, device="cuda")
    rs = torch.empty_like(xs)
    ybuf = torch.empty_like(xs)
    g = [plan.new_cache(), plan.new_cache()]
    stream = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(stream):
        for parity in range(2):
            plan.forward_chunk(xs, w, b, rs, g[parity], g[1 - parity], ybuf, stream=stream)
        stream.synchronize()
        for parity in range(2):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                plan.forward_chunk(xs, w, b, rs, g[parity], g[1 - parity], ybuf, stream=stream)
            graphs.append(gr)
    plan.reset(g[0])
    outs = []
    for k in range(T // Tc):
        xs.copy_(x[k * Tc:(k + 1) * Tc])
        rs.copy_(r[k * Tc:(k + 1) * Tc])
        graphs[k % 2].replay()
        outs.append(ybuf.clone())
    torch.cuda.synchronize()
    assert plan.status() == 0
    assert torch.equal(torch.cat(outs), y_eager)
    last = (T // Tc) % 2
    assert torch.equal(g[last], c[last])
    ref = oracle.conv_whole(to_f64(a["x"], "bf16"), to_f64(a["w"], "bf16"), to_f64(a["b"], "bf16"),
                            to_f64(a["r"], "bf16"))
    assert np.abs(from_device(y_eager) - ref).max() <= tolerance("bf16", ref)
    plan.close()


def test_graph_replay_of_a_frame_batched_layer_group_is_bit_identical():
    """A layer group (frame batches of one frame through a 3x3x3 conv and the 3-channel head) is
    captured into one CUDA graph per history parity over fixed buffers and a fixed workspace; the
    video streamed through the graphs equals the eager group calls bit for bit, outputs and both
    histories."""
    T, H, W, C, a, h = _layers()
    Tc = 4
    x = to_device(a["x"], "bf16")
    ws = [to_device(a["w"], "bf16"), to_device(h["w"], "bf16")]
    bs = [to_device(a["b"], "bf16"), to_device(h["b"], "bf16")]
    plans = [cc3d.CausalConv3dPlan(C, C, H, W), cc3d.CausalConv3dPlan(C, 3, H, W)]
    group = cc3d.LayerGroup(plans, 1)
    work = group.new_workspace(Tc)

    eager_c = [[p.new_cache(), p.new_cache()] for p in plans]
    ys = []
    for k in range(T // Tc):
        ys.append(group.forward_chunk(x[k * Tc:(k + 1) * Tc], ws, bs, [c[k % 2] for c in eager_c] if k else None,
                                      [c[(k + 1) % 2] for c in eager_c], workspace=work))
    y_eager = torch.cat(ys)
    torch.cuda.synchronize()
    assert all(p.status() == 0 for p in plans)

    xs = torch.empty((Tc, H, W, C), dtype=torch.bfloat16, device="cuda")
    yb = torch.empty((Tc, H, W, 3), dtype=torch.bfloat16, device="cuda")
    gc = [[p.new_cache(), p.new_cache()] for p in plans]
    s = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(s):
        # warm-up outside capture (the plans create their side streams on first use)
        group.forward_chunk(xs, ws, bs, None, [c[1] for c in gc], yb, workspace=work, stream=s)
    s.synchronize()
    for par in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            group.forward_chunk(xs, ws, bs, [c[par] for c in gc], [c[1 - par] for c in gc], yb, workspace=work,
                                stream=s)
        graphs.append(g)
    for p, c in zip(plans, gc):
        p.reset(c[0])  # the video's zero history, read by the first replay
    torch.cuda.synchronize()
    out = []
    for k in range(T // Tc):
        xs.copy_(x[k * Tc:(k + 1) * Tc])
        graphs[k % 2].replay()  # chunk k reads histories [k % 2] (zeros for k = 0), writes [(k + 1) % 2]
        out.append(yb.clone())
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(out), y_eager)
    for p_c, e_c in zip(gc, eager_c):
        assert torch.equal(p_c[(T // Tc) % 2], e_c[(T // Tc) % 2])
    assert all(p.status() == 0 for p in plans)
    group.close()
