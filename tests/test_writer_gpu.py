"""Asynchronous chunk output through the C ABI's writer: the narrow head's 8-bit frames are copied
to pinned host slots on a copy stream and appended to a file by a worker thread while the next
chunk computes.  The file must hold exactly the frames, in order."""
import numpy as np
import pytest
import torch

import chunked_causal_convolution_gb300 as cc3d
from tests.helpers import small_inputs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_writer_streams_u8_chunks_to_a_file(tmp_path):
    Cin, Cout, T, H, W, Tc = 32, 3, 12, 10, 150, 2
    raw = small_inputs(Cin, Cout, T, H, W, "bf16", 91, bias=True, residual=False)
    x, w, b = (to_device(raw[k], "bf16") for k in ("x", "w", "b"))
    plan = cc3d.CausalConv3dPlan(Cin, Cout, H, W)
    caches = [plan.new_cache(), plan.new_cache()]
    frame = H * W * Cout
    ybuf = [torch.empty((Tc, H, W, Cout), dtype=torch.uint8, device="cuda") for _ in range(2)]
    compute = torch.cuda.Stream()
    path = tmp_path / "frames.u8"
    writer = cc3d.FrameWriter(str(path), Tc * frame)
    seqs = [-1, -1]
    with torch.cuda.stream(compute):
        for k in range(T // Tc):
            buf = k % 2
            writer.wait_copied(seqs[buf], compute)  # the buffer's previous chunk has left the device
            plan.forward_chunk_u8(x[k * Tc:(k + 1) * Tc], w, b, None, caches[k % 2] if k else None,
                                  caches[(k + 1) % 2], ybuf[buf], stream=compute)
            seqs[buf] = writer.submit(ybuf[buf], stream=compute)
    assert writer.close() == T * frame
    assert plan.status(compute) == 0
    # reference: the same chunk loop, synchronous
    ref = []
    c2 = [plan.new_cache(), plan.new_cache()]
    for k in range(T // Tc):
        ref.append(plan.forward_chunk_u8(x[k * Tc:(k + 1) * Tc], w, b, None, c2[k % 2] if k else None,
                                         c2[(k + 1) % 2]).cpu().numpy())
    data = np.fromfile(path, dtype=np.uint8)
    assert data.size == T * frame
    assert np.array_equal(data, np.concatenate(ref).reshape(-1))
    plan.close()
