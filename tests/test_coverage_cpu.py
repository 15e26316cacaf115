"""Which compiled kernels the GPU parity cases reach, worked out on the host with
cc3d_plan_describe.

Every template instantiation of the tensor-core kernels that some supported layer can launch is
listed. The test checks that the GPU parity cases (tests/test_parity_gpu.py,
tests/test_graph_gpu.py and the full-size workloads) launch each one.  A change that makes a new
instantiation reachable fails here until a GPU case covers it.
"""
import itertools

import pytest

import chunked_causal_convolution_gb300 as cc3d
import synth
from chunked_causal_convolution_gb300 import build as lib_build
from tests import test_parity_gpu as tp
from tests.helpers import compositions_sample

# Reachable kernel instantiations that no GPU parity case launches yet: none.  (The 16-channel-block
# SM-pair, one-SM and fused-upsample instantiations and the 4-channel head have their own cases.)
KNOWN_GAPS = set()


def instantiation(d, Cout):
    """The compiled kernel a chunk launches: kernel name and template arguments."""
    k = d["kernel"]
    if k == "tc_bf16_kernel":
        # row groups per MMA warp (the launch's template argument)
        sub = d["row_groups"]
        subi = sub // 2 if (d["mma_warps"] == 2 and not d["split_n"] and not d["up2"]) else sub
        return (k, d["channel_block"], subi, d["tap_rows_per_weight_stage"])
    if k in ("tc2_bf16_kernel", "tc2s_bf16_kernel"):
        return (k, d["channel_block"], d["tap_rows_per_weight_stage"])
    if k == "head_bf16_kernel":
        return (k, Cout)
    return (k,)


def reached(plan_args, chunkings, residual, up2=False):
    try:
        plan = cc3d.Upsample2xConvPlan(*plan_args) if up2 else cc3d.CausalConv3dPlan(*plan_args)
    except cc3d.CC3DError:
        return set()
    Cout = plan_args[1]
    out = set()
    try:
        for c in {c for ch in chunkings for c in ch}:
            try:
                out.add(instantiation(plan.describe(c, residual), Cout))
            except cc3d.CC3DError:
                pass
    finally:
        plan.close()
    return out


def covered_by_gpu_cases():
    cov = set()

    def small(name, dtype, Cin, Cout, T, H, W, chunks, bias, residual, k=(3, 3, 3)):
        if dtype == "bf16":
            cov.update(reached((Cin, Cout, H, W) + tuple(k), [chunks, [T], [1] * T], residual))

    for c in tp.SMALL:
        small(*c)
    for c in tp.EXTENTS:
        small(*c[:10], k=c[10])
    for name, Cin, Cout, T, H, W, chunks, bias, residual, kt in tp.TSTACK:
        cov.update(reached((Cin, Cout, H, W, kt, 3, 3), [chunks, [T], [1] * T], residual))
    for name, Cin, Cout, T, H, W, chunks, bias, residual, kt in tp.UP2:
        cov.update(reached((Cin, Cout, H, W, kt), [chunks, [T], [1] * T], residual, up2=True))
    for Cin, Cout, H, W, k, family in tp.FAMILIES:
        cov.update(reached((Cin, Cout, H, W) + tuple(k), [[4]], True))
    for name in ("c96_residual", "c192", "c384", "c384_to_192", "sr96", "sr_head3"):
        wl = synth.WORKLOADS[name]
        cov.update(reached((wl.Cin, wl.Cout, wl.H, wl.W), [list(wl.chunks), [4, 4], [8]] + compositions_sample(),
                           wl.r is not None))
    return cov


def reachable():
    out = set()
    for Cin, Cout, W, kt, ks, T in itertools.product((16, 32, 48, 96), (1, 2, 3, 4, 5, 16, 32, 96, 192, 512),
                                                     (17, 128, 256), (1, 2, 3), (1, 3), (1, 2, 3)):
        out |= reached((Cin, Cout, 4, W, kt, ks, ks), [[T]], True)
    for Cin, Cout, W, kt, T in itertools.product((16, 32, 48, 96), (16, 64, 96, 192), (17, 128), (1, 3), (1, 2)):
        out |= reached((Cin, Cout, 8, W, kt), [[T]], True, up2=True)
    return out


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return cc3d.load_library()


def test_gpu_parity_cases_launch_every_reachable_kernel_but_the_listed_gaps(lib):
    cov = covered_by_gpu_cases()
    reach = reachable()
    assert cov <= reach | cov  # the cases only use supported shapes
    missing = reach - cov
    assert missing <= KNOWN_GAPS, sorted(missing - KNOWN_GAPS)
    # the gaps are real: reachable, and not covered
    assert KNOWN_GAPS <= reach and not (KNOWN_GAPS & cov), (sorted(KNOWN_GAPS - reach), sorted(KNOWN_GAPS & cov))


def test_the_measured_workloads_launch_the_kernels_they_are_reported_for(lib):
    cov = set()
    for name in ("c96_residual", "c192", "c384", "c384_to_192"):
        wl = synth.WORKLOADS[name]
        cov |= reached((wl.Cin, wl.Cout, wl.H, wl.W), [[4]], wl.r is not None)
    assert ("tc2s_bf16_kernel", 32, 3) in cov and ("tc2_bf16_kernel", 32, 1) in cov
