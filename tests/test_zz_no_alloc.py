"""The layer group's allocation-free entry point, cc3d_group_forward_chunk_static.

Some callers cannot allocate device memory: a plugin inside a host framework whose allocator owns
the GPU's memory and only hands over input and output buffers, or a processing loop that must not
allocate once it runs (cudaMalloc and cudaFree can synchronise the device).  For them the library
runs a layer group with a fixed device array of its own as the workspace.  Called through the C ABI
twice in a row (two chunks of one video, the second continuing the first's histories), it must
give what cc3d_group_forward_chunk gives with a workspace the caller allocated, within the bf16
tolerance of the parity tests; and a chunk that needs more than the array holds is refused before
anything is launched.  This file is collected last, so that a run stopping at its first failure
has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import chunked_causal_convolution_gb300 as cc3d
from tests.helpers import from_device, small_inputs, to_device, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _arr(items):
    return (ctypes.c_void_p * len(items))(*[None if t is None else t.data_ptr() for t in items])


def test_static_scratch_group_matches_the_workspace_group_on_two_calls_in_a_row():
    lib = cc3d.load_library()
    H, W = 6, 130
    spec = [(96, 96, (3, 3, 3)), (96, 64, (1, 1, 1)), (64, 3, (3, 3, 3))]
    plans, ws_, bs_ = [], [], []
    for j, (ci, co, k) in enumerate(spec):
        p = small_inputs(ci, co, 1, 1, 1, "bf16", 900 + j, bias=True, k=k)
        plans.append(cc3d.CausalConv3dPlan(ci, co, H, W, *k))
        ws_.append(to_device(p["w"], "bf16"))
        bs_.append(to_device(p["b"], "bf16"))
    x = to_device(small_inputs(96, 96, 7, H, W, "bf16", 910, bias=False)["x"], "bf16")
    group = cc3d.LayerGroup(plans, 2)
    chunks = [4, 3]
    assert group.workspace_bytes(4) <= 64 * 1024 * 1024  # the chunk fits the fixed array

    def run(static):
        caches = [[p.new_cache(), p.new_cache()] if p.kt > 1 else [None, None] for p in plans]
        ys, s = [], 0
        stream = torch.cuda.current_stream()
        for k, c in enumerate(chunks):
            y = torch.empty((c, H, W, 3), dtype=torch.bfloat16, device="cuda")
            cin = [c_[k % 2] if k else None for c_ in caches]
            cout = [c_[(k + 1) % 2] for c_ in caches]
            if static:
                rc = lib.cc3d_group_forward_chunk_static(group.handle, c, x[s:s + c].data_ptr(), _arr(ws_), _arr(bs_),
                                                         _arr(cin), _arr(cout), y.data_ptr(), stream.cuda_stream)
                assert rc == 0, cc3d.cc3d_status_string(rc)
            else:
                group.forward_chunk(x[s:s + c], ws_, bs_, cin, cout, y)
            ys.append(y)
            s += c
        assert all(p.status() == 0 for p in plans)
        return torch.cat(ys), [c_[len(chunks) % 2] for c_ in caches if c_[0] is not None]

    y_ws, h_ws = run(static=False)
    for _ in range(2):  # the array keeps the previous call's contents; results must not depend on them
        y_st, h_st = run(static=True)
        ref = from_device(y_ws)
        assert np.abs(from_device(y_st) - ref).max() <= tolerance("bf16", ref)
        for a, b in zip(h_st, h_ws):
            r = from_device(b)
            assert np.abs(from_device(a) - r).max() <= tolerance("bf16", r)
    group.close()
    for p in plans:
        p.close()


def test_static_scratch_refuses_a_chunk_larger_than_the_array():
    lib = cc3d.load_library()
    H, W = 360, 640
    plans = [cc3d.CausalConv3dPlan(96, 96, H, W), cc3d.CausalConv3dPlan(96, 3, H, W)]
    group = cc3d.LayerGroup(plans, 0)  # the whole 4-frame chunk: 177 MB of intermediates
    assert group.workspace_bytes(4) > 64 * 1024 * 1024
    x = torch.zeros((4, H, W, 96), dtype=torch.bfloat16, device="cuda")
    y = torch.full((4, H, W, 3), 7.0, dtype=torch.bfloat16, device="cuda")
    w = [torch.zeros((96, 3, 3, 3, 96), dtype=torch.bfloat16, device="cuda"),
         torch.zeros((3, 3, 3, 3, 96), dtype=torch.bfloat16, device="cuda")]
    cout = [p.new_cache() for p in plans]
    rc = lib.cc3d_group_forward_chunk_static(group.handle, 4, x.data_ptr(), _arr(w), None, None, _arr(cout),
                                             y.data_ptr(), None)
    assert rc == 10 and cc3d.STATUS_NAMES[rc] == "CC3D_ERR_SCRATCH_TOO_SMALL"
    torch.cuda.synchronize()
    assert torch.all(y.float() == 7.0)
    group.close()
    for p in plans:
        p.close()
