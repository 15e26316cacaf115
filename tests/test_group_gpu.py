"""Layer groups run frame batch by frame batch (cc3d_group_*, "SwiftVR Inference Optimization",
section "ReAE Frame Batching"): the group's output and every layer's history after each chunk are
bit-identical to running each layer's chunk loop over the whole chunk, for every frame-batch size,
and every layer of that loop is within tolerance of the oracle applied to the bf16 input it read
(the previous layer's stored output)."""
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


STACKS = {
    # (Cin, Cout, (kt, kh, kw), up2) per layer; frames H x W of the first layer
    "pair_pointwise_head": ([(96, 96, (3, 3, 3), False), (96, 64, (1, 1, 1), False), (64, 3, (3, 3, 3), False)],
                            5, 128),
    "memblock_spatial_tiles": ([(32, 48, (2, 3, 3), False), (48, 32, (1, 3, 3), False), (32, 32, (3, 3, 3), False)],
                               6, 40),
    "upsample_then_pointwise": ([(32, 32, (3, 3, 3), True), (32, 16, (1, 1, 1), False)], 4, 24),
}


def _make(stack, H, W, seed):
    plans, params = [], []
    h, w_ = H, W
    for j, (ci, co, k, up2) in enumerate(stack):
        p = small_inputs(ci, co, 1, 1, 1, "bf16", seed + j, bias=True, k=k)
        if up2:
            plan = cc3d.Upsample2xConvPlan(ci, co, h, w_, k[0])
        else:
            plan = cc3d.CausalConv3dPlan(ci, co, h, w_, *k)
        plans.append(plan)
        params.append((to_device(p["w"], "bf16"), to_device(p["b"], "bf16"), p))
        h, w_ = plan.Ho, plan.Wo
    return plans, params


def _layer_by_layer(plans, params, x, chunks):
    """Each layer's own chunk loop over each whole chunk; histories ping-pong per layer.  Returns
    every layer's output over the whole video and the histories after each chunk."""
    caches = [[p.new_cache(), p.new_cache()] if p.kt > 1 else [None, None] for p in plans]
    outs, hists, s = [[] for _ in plans], [], 0
    for k, c in enumerate(chunks):
        cur = x[s:s + c]
        for j, (p, (w, b, _)) in enumerate(zip(plans, params)):
            cur = p.forward_chunk(cur, w, b, None, caches[j][k % 2] if k else None, caches[j][(k + 1) % 2])
            outs[j].append(cur)
        hists.append([None if c_[0] is None else c_[(k + 1) % 2].clone() for c_ in caches])
        s += c
    return [torch.cat(o) for o in outs], hists


@pytest.mark.parametrize("name", sorted(STACKS))
@pytest.mark.parametrize("frame_batch", [0, 1, 2, 3])
def test_group_equals_the_layer_by_layer_chunk_loop(name, frame_batch):
    stack, H, W = STACKS[name]
    T, chunks = 7, [4, 3]
    plans, params = _make(stack, H, W, 700 + len(name))
    raw = small_inputs(stack[0][0], stack[0][1], T, H, W, "bf16", 720 + len(name), bias=False)
    x = to_device(raw["x"], "bf16")
    outs_ref, hists_ref = _layer_by_layer(plans, params, x, chunks)
    y_ref = outs_ref[-1]
    group = cc3d.LayerGroup(plans, frame_batch)
    ws = group.new_workspace(max(chunks))
    caches = [[p.new_cache(), p.new_cache()] if p.kt > 1 else [None, None] for p in plans]
    ys, s = [], 0
    for k, c in enumerate(chunks):
        ys.append(group.forward_chunk(x[s:s + c], [q[0] for q in params], [q[1] for q in params],
                                      [c_[k % 2] if k else None for c_ in caches],
                                      [c_[(k + 1) % 2] for c_ in caches], workspace=ws))
        for j, c_ in enumerate(caches):
            if c_[0] is not None:
                assert torch.equal(c_[(k + 1) % 2], hists_ref[k][j]), (name, frame_batch, k, j)
        s += c
    assert all(p.status() == 0 for p in plans)
    y = torch.cat(ys)
    assert torch.equal(y, y_ref), (name, frame_batch, int((y != y_ref).sum()))
    # every layer against the oracle on the bf16 input it read (the previous layer's stored output)
    inp = to_f64(raw["x"], "bf16")
    for j, ((w, b, p), (ci, co, k, up2)) in enumerate(zip(params, stack)):
        conv = oracle.conv_upsample2x_whole if up2 else oracle.conv_whole
        ref = conv(inp, to_f64(p["w"], "bf16"), to_f64(p["b"], "bf16"))
        got = from_device(outs_ref[j])
        err = np.abs(got - ref).max()
        assert err <= tolerance("bf16", ref), (name, frame_batch, j, err)
        inp = got
    group.close()
    for p in plans:
        p.close()


def test_group_empty_chunk_moves_every_history():
    stack, H, W = STACKS["pair_pointwise_head"]
    plans, params = _make(stack, H, W, 790)
    group = cc3d.LayerGroup(plans, 1)
    cin = [p.new_cache() if p.kt > 1 else None for p in plans]
    for c in cin:
        if c is not None:
            c.fill_(1.5)
    cout = [p.new_cache() if p.kt > 1 else None for p in plans]
    cc3d.cc3d_group_forward_chunk(group.handle, 0, None, [q[0] for q in params], None, cin, cout, None, None, 0)
    torch.cuda.synchronize()
    for a, b in zip(cin, cout):
        if a is not None:
            assert torch.equal(a, b)
    group.close()



def _random_stacks(n=16, seed=7021):
    rng = np.random.RandomState(seed)
    out = []
    for _ in range(n):
        nl = int(rng.randint(2, 5))
        c = int(rng.choice([16, 32, 48, 64]))
        stack, used_up2 = [], False
        for _ in range(nl):
            co = int(rng.choice([16, 32, 48, 64]))
            up2 = (not used_up2) and rng.rand() < 0.2
            used_up2 |= up2
            kt = int(rng.randint(1, 4))
            k = 3 if up2 else int(rng.choice([1, 3]))
            stack.append((c, co, (kt, k, k), bool(up2)))
            c = co
        T = int(rng.randint(2, 8))
        cuts = sorted(rng.choice(np.arange(1, T), size=rng.randint(0, min(2, T - 1) + 1), replace=False))
        bounds = [0] + [int(x) for x in cuts] + [T]
        chunks = [b - a for a, b in zip(bounds, bounds[1:])]
        out.append(dict(stack=stack, H=int(rng.randint(2, 7)), W=int(rng.randint(8, 41)), T=T, chunks=chunks,
                        frame_batch=int(rng.choice([0, 1, 2, 3, 5]))))
    return out


RANDOM_STACKS = _random_stacks()


@pytest.mark.parametrize("case", RANDOM_STACKS, ids=["stack%d_fb%d" % (i, c["frame_batch"])
                                                     for i, c in enumerate(RANDOM_STACKS)])
def test_random_group_equals_the_layer_by_layer_chunk_loop(case):
    """Random stacks of 2-4 layers (any kt, 1x1 or 3x3, at most one fused upsample), random
    chunkings and frame batches: the group's output and every layer's history after each chunk
    equal those of each layer's own chunk loop, bit for bit."""
    stack, H, W, T, chunks = case["stack"], case["H"], case["W"], case["T"], case["chunks"]
    plans, params = _make(stack, H, W, 40 + len(stack) + H + W)
    raw = small_inputs(stack[0][0], stack[0][1], T, H, W, "bf16", 60 + T + W, bias=False)
    x = to_device(raw["x"], "bf16")
    outs_ref, hists_ref = _layer_by_layer(plans, params, x, chunks)
    group = cc3d.LayerGroup(plans, case["frame_batch"])
    ws = group.new_workspace(max(chunks))
    caches = [[p.new_cache(), p.new_cache()] if p.kt > 1 else [None, None] for p in plans]
    ys, s = [], 0
    for k, c in enumerate(chunks):
        ys.append(group.forward_chunk(x[s:s + c], [q[0] for q in params], [q[1] for q in params],
                                      [c_[k % 2] if k else None for c_ in caches],
                                      [c_[(k + 1) % 2] for c_ in caches], workspace=ws))
        for j, c_ in enumerate(caches):
            if c_[0] is not None:
                assert torch.equal(c_[(k + 1) % 2], hists_ref[k][j]), (case, k, j)
        s += c
    assert all(p.status() == 0 for p in plans)
    assert torch.equal(torch.cat(ys), outs_ref[-1]), case
    group.close()
    for p in plans:
        p.close()
