"""Several plans in flight at once on different streams: the library keeps no state that two plans
share beyond the per-device status word, so chunk loops interleaved on two streams (each plan on
its own stream, both running concurrently on the device) give the same bytes as each loop run
alone, and the status stays clear."""
import pytest
import torch

import chunked_causal_convolution_gb300 as cc3d
from tests.helpers import run_chunks, small_inputs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


LAYERS = [
    # Cin, Cout, H, W, (kt, kh, kw), residual: two-frame pairs, flat one-SM tiles, the streaming
    # kernel and the narrow head, all with histories
    (96, 96, 6, 256, (3, 3, 3), True),
    (64, 128, 5, 70, (3, 3, 3), False),
    (64, 96, 4, 200, (3, 1, 1), False),
    (96, 3, 8, 300, (3, 3, 3), False),
]


def test_interleaved_chunk_loops_on_two_streams_equal_the_loops_alone():
    T, chunks = 6, [4, 2]
    setups = []
    for i, (ci, co, H, W, k, res) in enumerate(LAYERS):
        raw = small_inputs(ci, co, T, H, W, "bf16", 1200 + i, bias=True, residual=res, k=k)
        dev = {key: to_device(v, "bf16") for key, v in raw.items()}
        plan = cc3d.CausalConv3dPlan(ci, co, H, W, *k)
        y_alone, c_alone = run_chunks(plan, dev["x"], dev["w"], dev["b"], dev.get("r"), chunks)
        setups.append((plan, dev, y_alone, c_alone[-1]))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    state = []
    for plan, dev, _, _ in setups:
        caches = [plan.new_cache(), plan.new_cache()]
        y = torch.empty_like(setups[len(state)][2])
        state.append((caches, y))
    torch.cuda.synchronize()
    # chunk k of every layer, layers alternating between the two streams
    s0 = 0
    for k, c in enumerate(chunks):
        for i, ((plan, dev, _, _), (caches, y)) in enumerate(zip(setups, state)):
            st = streams[i % 2]
            with torch.cuda.stream(st):
                plan.forward_chunk(dev["x"][s0:s0 + c], dev["w"], dev["b"],
                                   dev["r"][s0:s0 + c] if "r" in dev else None,
                                   caches[k % 2] if k else None, caches[(k + 1) % 2], y[s0:s0 + c], stream=st)
        s0 += c
    torch.cuda.synchronize()
    for (plan, dev, y_alone, c_alone), (caches, y) in zip(setups, state):
        assert plan.status() == 0
        assert torch.equal(y, y_alone), plan.kernel
        assert torch.equal(caches[len(chunks) % 2], c_alone), plan.kernel
        plan.close()
