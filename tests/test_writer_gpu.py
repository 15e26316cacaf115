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


def test_writer_drops_the_chunks_queued_behind_a_failed_write(tmp_path):
    """A write that fails (here: the file is a FIFO whose reader has gone) makes the writer drop
    the chunks queued behind it instead of writing them, so the output never holds a gap followed
    by later chunks.  A second reader opens the FIFO after the failure and before the next queued
    chunk's copy lands: it must receive nothing."""
    import os
    import time
    n = 16384
    chunks = [torch.full((n,), 10 + k, dtype=torch.uint8, device="cuda") for k in range(3)]
    path = str(tmp_path / "frames.fifo")
    os.mkfifo(path)
    r1 = os.open(path, os.O_RDONLY | os.O_NONBLOCK)
    writer = cc3d.FrameWriter(path, n)
    compute, aux = torch.cuda.Stream(), torch.cuda.Stream()
    r2 = None
    try:
        writer.submit(chunks[0], stream=compute)
        got, t0 = b"", time.time()
        while len(got) < n and time.time() - t0 < 10:
            try:
                got += os.read(r1, n - len(got))
            except BlockingIOError:
                time.sleep(0.01)
        assert got == bytes([10]) * n
        os.close(r1)  # no reader: the next write fails
        with torch.cuda.stream(compute):
            torch.cuda._sleep(600_000_000)     # chunk 1's copy lands after this
            seq1 = writer.submit(chunks[1], stream=compute)
            torch.cuda._sleep(3_000_000_000)   # chunk 2's copy lands after this
            writer.submit(chunks[2], stream=compute)
        writer.wait_copied(seq1, aux)
        aux.synchronize()
        time.sleep(0.3)                        # the worker's write of chunk 1 has failed by now
        r2 = os.open(path, os.O_RDONLY | os.O_NONBLOCK)
        with pytest.raises(cc3d.CC3DError) as e:
            writer.close()
        assert e.value.code == 9
        try:
            late = os.read(r2, 2 * n)
        except BlockingIOError:
            late = b""
        assert late == b"", len(late)
    finally:
        writer.close()
        if r2 is not None:
            os.close(r2)
        torch.cuda.synchronize()
