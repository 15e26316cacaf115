"""A seeded sweep of layer shapes drawn at random through the configurations the plans choose
between: one-SM and SM-pair tiles (flat and row-aligned frames, two-frame pairs, channel blocks,
short-last-wave splits), the narrow head and the narrow-output kernel, the streaming kernel of the
1x1 spatial extents, the fused nearest-2x upsample and the fp32 path.  Every case is compared with
the fp64 oracle element by element, and two different chunkings of the same frames give the same
bytes, outputs and final history alike (the chunked form equals the whole-sequence form:
"SGLang-Diffusion advanced optimizations", section 3 "Parallel VAE").  The cases are fixed by the
seed, so a failure names a reproducible shape."""
import numpy as np
import pytest
import torch

import chunked_causal_convolution_gb300 as cc3d
import oracle
from tests.helpers import from_device, run_chunks, small_inputs, to_device, to_f64, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _composition(rng, T):
    """A random split of T frames into chunks."""
    cuts = sorted(rng.choice(np.arange(1, T), size=rng.randint(0, min(3, T - 1) + 1), replace=False)) if T > 1 else []
    bounds = [0] + [int(c) for c in cuts] + [T]
    return [b - a for a, b in zip(bounds, bounds[1:])]


def _cases(n=96, seed=20261202):
    rng = np.random.RandomState(seed)
    cases = []
    while len(cases) < n:
        kind = rng.choice(["conv", "conv", "conv", "two_frame", "conv1x1", "conv1x1", "head", "narrow", "up2",
                           "f32"])
        T = int(rng.randint(2, 8))
        H = int(rng.randint(1, 10))
        W = int(rng.choice([int(rng.randint(1, 90)), 128, 256]))
        kt, k = 3, 3
        if kind == "two_frame":
            # SM pairs with two output frames per MMA: frames a multiple of 128 wide, at most 96
            # output channels, a history
            W = int(rng.choice([128, 256]))
        if kind == "f32":
            Cin, Cout = int(rng.choice([4, 8, 16])), int(rng.choice([3, 8, 16]))
            kt = int(rng.randint(1, 4))
            dtype = "f32"
        else:
            dtype = "bf16"
            Cin = int(rng.choice([16, 32, 48, 64, 96, 128]))
            if kind == "head":
                Cout = int(rng.randint(1, 6))
            elif kind == "two_frame":
                Cout = int(rng.choice([16, 32, 48, 64, 96]))
                kt = int(rng.randint(2, 4))
            elif kind == "narrow":
                Cout = int(rng.choice([6, 8, 12]))
                kt = int(rng.randint(1, 4))
            else:
                Cout = int(rng.choice([16, 32, 48, 64, 96, 128, 192, 256, 384]))
                kt = int(rng.randint(1, 4))
            if kind == "conv1x1":
                k = 1
        # keep the oracle to a few seconds
        while T * H * W * Cin * Cout * kt * k * k > 4e8 and W > 8 and kind != "two_frame":
            W //= 2
        bias = bool(rng.randint(2))
        residual = bool(rng.randint(2)) and kind not in ("up2",)
        chunks = [_composition(rng, T), _composition(rng, T)]
        cases.append(dict(kind=str(kind), dtype=dtype, Cin=Cin, Cout=Cout, T=T, H=H, W=W, kt=kt, k=k,
                          bias=bias, residual=residual, chunks=chunks))
    return cases


CASES = _cases()


def _id(c):
    return "%s_%s_%dto%d_k%dx%d_T%d_%dx%d%s%s" % (c["kind"], c["dtype"], c["Cin"], c["Cout"], c["kt"], c["k"], c["T"],
                                                 c["H"], c["W"], "_b" if c["bias"] else "", "_r" if c["residual"] else "")


@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_random_layer_matches_the_oracle_and_every_chunking(case):
    c = case
    kt, k = c["kt"], c["k"]
    up2 = c["kind"] == "up2"
    raw = small_inputs(c["Cin"], c["Cout"], c["T"], c["H"], c["W"], c["dtype"], 900 + len(_id(c)), c["bias"],
                       c["residual"], k=(kt, k, k))
    dev = {key: to_device(v, c["dtype"]) for key, v in raw.items()}
    if up2:
        plan = cc3d.Upsample2xConvPlan(c["Cin"], c["Cout"], c["H"], c["W"], kt, dtype=c["dtype"])
    else:
        plan = cc3d.CausalConv3dPlan(c["Cin"], c["Cout"], c["H"], c["W"], kt, k, k, dtype=c["dtype"])
    ys, caches = [], []
    for chunks in c["chunks"]:
        y, cs = run_chunks(plan, dev["x"], dev["w"], dev.get("b"), dev.get("r"), chunks)
        ys.append(y)
        caches.append(cs[-1])
    assert plan.status() == 0, (plan.kernel, c)
    assert torch.equal(ys[0], ys[1]), (plan.kernel, c)
    assert torch.equal(caches[0], caches[1]), (plan.kernel, c)
    # the final history is the last kt - 1 input frames
    P = kt - 1
    if P > 0:
        assert torch.equal(caches[0], dev["x"][c["T"] - P:]), (plan.kernel, c)
    conv = oracle.conv_upsample2x_whole if up2 else oracle.conv_whole
    ref = conv(to_f64(raw["x"], c["dtype"]), to_f64(raw["w"], c["dtype"]),
               to_f64(raw["b"], c["dtype"]) if c["bias"] else None,
               to_f64(raw["r"], c["dtype"]) if c["residual"] else None)
    err = np.abs(from_device(ys[0]) - ref).max()
    assert err <= tolerance(c["dtype"], ref), (plan.kernel, c, err)
    plan.close()


# Medium shapes with more tiles than the SMs hold at once: several tiles per block or pair, the
# one-SM kernel's split last wave, the streaming kernel's runs of units, many head strips.
MEDIUM = [
    dict(kind="conv", dtype="bf16", Cin=192, Cout=192, T=3, H=90, W=160, kt=3, k=3, bias=True, residual=True,
         chunks=[[3], [1, 2]]),                       # one SM, 171 tiles: the last 19 split
    dict(kind="two_frame", dtype="bf16", Cin=96, Cout=96, T=4, H=128, W=256, kt=3, k=3, bias=True,
         residual=True, chunks=[[4], [2, 2]]),        # two-frame pairs, two pair tiles per pair
    dict(kind="conv", dtype="bf16", Cin=128, Cout=128, T=4, H=60, W=200, kt=2, k=3, bias=False, residual=True,
         chunks=[[4], [2, 2]]),                       # flat pairs, 96 pair tiles on 76 pairs
    dict(kind="conv1x1", dtype="bf16", Cin=64, Cout=128, T=5, H=80, W=200, kt=3, k=1, bias=True,
         residual=False, chunks=[[5], [4, 1]]),       # streaming kernel, 250 units
    dict(kind="head", dtype="bf16", Cin=96, Cout=3, T=4, H=64, W=512, kt=3, k=3, bias=True, residual=False,
         chunks=[[4], [1, 3]]),                       # narrow head, many strips
    dict(kind="up2", dtype="bf16", Cin=64, Cout=64, T=3, H=48, W=80, kt=3, k=3, bias=True, residual=False,
         chunks=[[3], [2, 1]]),                       # fused upsample, 96 x 160 outputs
    # the widest layers: 512 output channels in two 256-column blocks (N = 256 MMAs), 512 inputs
    dict(kind="conv", dtype="bf16", Cin=64, Cout=512, T=4, H=3, W=40, kt=3, k=3, bias=True, residual=True,
         chunks=[[4], [3, 1]]),
    dict(kind="conv", dtype="bf16", Cin=512, Cout=64, T=4, H=4, W=40, kt=3, k=3, bias=True, residual=False,
         chunks=[[4], [1, 3]]),
    dict(kind="conv", dtype="bf16", Cin=512, Cout=512, T=3, H=2, W=24, kt=2, k=3, bias=False, residual=True,
         chunks=[[3], [2, 1]]),
]


@pytest.mark.parametrize("case", MEDIUM, ids=[_id(c) for c in MEDIUM])
def test_medium_layer_matches_the_oracle_and_every_chunking(case):
    test_random_layer_matches_the_oracle_and_every_chunking(case)
