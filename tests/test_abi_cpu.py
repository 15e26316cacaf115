"""C-ABI checks that need no GPU: the library loads, exports every declared symbol, and
rejects bad arguments before touching any buffer (argument checks run on the host)."""
import ctypes
import os
import re

import pytest

import chunked_causal_convolution_gb300 as cc3d
from chunked_causal_convolution_gb300 import build as lib_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "cc3d.h")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return cc3d.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cc3d_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("cc3d_plan_create", "cc3d_forward_chunk", "cc3d_reset", "cc3d_destroy", "cc3d_get_status"):
        assert n in names
    assert set(names) == set(cc3d.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(10):
        s = cc3d.cc3d_status_string(code)
        assert s and s != "unknown status"
    assert cc3d.cc3d_status_string(99) == "unknown status"


@pytest.mark.parametrize("args,code", [
    ((0, 16, 8, 8, 3, 3, 3, cc3d.CC3D_BF16), 1),
    ((16, 16, 8, 0, 3, 3, 3, cc3d.CC3D_BF16), 1),
    ((16, 16, 8, 8, 3, 2, 3, cc3d.CC3D_BF16), 1),    # even spatial extent
    ((16, 16, 8, 8, 3, 3, 3, 7), 1),                 # unknown dtype
    ((24, 16, 8, 8, 3, 3, 3, cc3d.CC3D_BF16), 2),    # Cin not a multiple of 16
    ((32, 24, 8, 8, 3, 3, 3, cc3d.CC3D_BF16), 2),    # Cout >= 16 not a multiple of 16
    ((32, 32, 8, 8, 3, 5, 5, cc3d.CC3D_BF16), 2),    # bf16: 3x3 or 1x1 spatial kernels only
    ((32, 32, 8, 8, 3, 3, 1, cc3d.CC3D_BF16), 2),    # bf16: square spatial kernels only
    ((32, 32, 8, 8, 4, 3, 3, cc3d.CC3D_BF16), 2),    # bf16: temporal extent at most 3
    ((32, 1024, 8, 8, 3, 3, 3, cc3d.CC3D_BF16), 2),  # beyond tensor-memory budget
    ((4, 4, 8, 8, 5, 3, 3, cc3d.CC3D_F32), 2),       # fp32 temporal extent limit
])
def test_plan_create_rejects(lib, args, code):
    h = ctypes.c_void_p(123)
    rc = lib.cc3d_plan_create(*args, ctypes.byref(h))
    assert rc == code
    assert h.value is None  # *out is cleared on error


@pytest.mark.parametrize("args,kernel,launches", [
    ((96, 96, 360, 640, 3, 3, 3, cc3d.CC3D_BF16), "tc_bf16_pair", 1),
    ((192, 192, 180, 320, 3, 3, 3, cc3d.CC3D_BF16), "tc_bf16", 1),
    ((384, 384, 90, 160, 3, 3, 3, cc3d.CC3D_BF16), "tc_bf16", 1),
    ((96, 3, 1440, 2560, 3, 3, 3, cc3d.CC3D_BF16), "tc_bf16_head", 1),
    ((96, 96, 360, 640, 2, 3, 3, cc3d.CC3D_BF16), "tc_bf16_pair", 1),    # MemoryBlock, 1-frame history
    ((96, 96, 360, 640, 3, 1, 1, cc3d.CC3D_BF16), "tc_bf16_stream", 1),  # TemporalGrow
    ((192, 192, 180, 320, 1, 1, 1, cc3d.CC3D_BF16), "tc_bf16_stream", 1), # pointwise projection
    ((16, 32, 64, 64, 3, 1, 1, cc3d.CC3D_BF16), "tc_bf16", 1),           # 16-channel blocks: tiles
    ((64, 384, 64, 64, 1, 1, 1, cc3d.CC3D_BF16), "tc_bf16", 1),          # N > 256: tiles
    ((96, 3, 64, 64, 2, 3, 3, cc3d.CC3D_BF16), "tc_bf16_narrow", 1),     # the narrow head kernel is 3x3x3 only
    ((48, 3, 64, 64, 3, 3, 3, cc3d.CC3D_BF16), "tc_bf16_narrow", 1),   # Cin not a multiple of 32
    ((512, 3, 64, 64, 3, 3, 3, cc3d.CC3D_BF16), "tc_bf16_narrow", 1),  # too wide to stage a row
    ((96, 8, 64, 64, 3, 3, 3, cc3d.CC3D_BF16), "tc_bf16_narrow", 1),   # 9 taps x 8 channels exceed N = 48
    ((16, 16, 32, 32, 3, 3, 3, cc3d.CC3D_F32), "simt_f32", 2),
    ((3, 5, 7, 9, 2, 1, 3, cc3d.CC3D_F32), "simt_f32", 2),
])
def test_plan_create_accepts(lib, args, kernel, launches):
    p = cc3d.cc3d_plan_create(*args)
    try:
        assert cc3d.cc3d_plan_kernel(p) == kernel
        assert cc3d.cc3d_plan_launches_per_chunk(p) == launches
    finally:
        cc3d.cc3d_destroy(p)


def test_destroy_null_is_safe(lib):
    lib.cc3d_destroy(None)


def test_forward_rejects_before_any_device_work(lib):
    p = cc3d.cc3d_plan_create(32, 32, 4, 8, 3, 3, 3, cc3d.CC3D_BF16)
    try:
        # x 2 KB, w 54 KB, y 2 KB, caches 4 KB each: disjoint spans in one host buffer
        buf = (ctypes.c_uint8 * (1 << 17))()
        base = (ctypes.addressof(buf) + 255) & ~255
        x, w, y, c0, c1 = base, base + 4096, base + 65536, base + 69632, base + 77824
        f = lib.cc3d_forward_chunk
        assert f(None, 1, x, w, None, None, None, c1, y, None) == 1          # null plan
        assert f(p, -1, x, w, None, None, None, c1, y, None) == 1            # negative T
        assert f(p, 1, None, w, None, None, None, c1, y, None) == 1          # missing x
        assert f(p, 1, x, w, None, None, None, None, y, None) == 1           # missing cache_out
        assert f(p, 1 << 29, x, w, None, None, None, c1, y, None) == 2       # 2^34 positions in one chunk
        assert f(p, 1, x + 8, w, None, None, None, c1, y, None) == 3         # misaligned
        assert f(p, 1, x, w, None, None, None, c1, x, None) == 4             # y overlaps x
        assert f(p, 1, x, w, None, None, c0, c0, y, None) == 4               # cache_out overlaps cache_in
        assert f(p, 1, x, w, None, None, None, x, y, None) == 4              # cache_out overlaps x
        # host memory is not device memory (no GPU here: the check itself fails closed)
        assert f(p, 1, x, w, None, None, None, c1, y, None) == 8
        assert lib.cc3d_reset(p, base + 8, None) == 3
        assert lib.cc3d_reset(None, base, None) == 1
        assert lib.cc3d_debug_set_fault(p, 9) == 1
        assert lib.cc3d_debug_set_wait_budget_ns(p, 0) == 1
    finally:
        cc3d.cc3d_destroy(p)


def test_binding_raises_loudly_without_the_library(monkeypatch, tmp_path):
    import importlib
    mod = importlib.import_module("chunked_causal_convolution_gb300")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        mod.cc3d_plan_create(16, 16, 8, 8)


def test_u8_output_is_for_narrow_head_plans_only(lib):
    # checked before any argument or device work: a wide plan is refused outright
    p = cc3d.cc3d_plan_create(32, 32, 4, 8, 3, 3, 3, cc3d.CC3D_BF16)
    try:
        assert lib.cc3d_forward_chunk_u8(p, 1, None, None, None, None, None, None, None, None) == 2
    finally:
        cc3d.cc3d_destroy(p)
    p = cc3d.cc3d_plan_create(96, 3, 16, 200, 3, 3, 3, cc3d.CC3D_BF16)
    try:
        assert cc3d.cc3d_plan_kernel(p) == "tc_bf16_head"
        assert lib.cc3d_forward_chunk_u8(p, 1, None, None, None, None, None, None, None, None) == 1  # missing x
    finally:
        cc3d.cc3d_destroy(p)


def test_writer_argument_and_file_errors_need_no_device(lib, tmp_path):
    import ctypes
    h = ctypes.c_void_p(123)
    assert lib.cc3d_writer_create(None, 1024, ctypes.byref(h)) == 1 and h.value is None
    assert lib.cc3d_writer_create(str(tmp_path / "a.bin").encode(), 0, ctypes.byref(h)) == 1
    # a path that cannot be opened fails before any CUDA work
    assert lib.cc3d_writer_create(str(tmp_path / "missing_dir" / "a.bin").encode(), 1024, ctypes.byref(h)) == 9
    assert h.value is None
    assert lib.cc3d_writer_submit(None, None, 0, None, None) == 1
    assert lib.cc3d_writer_wait_copied(None, 0, None) == 1
    assert lib.cc3d_writer_close(None, None) == 1


@pytest.mark.parametrize("C", [16, 32, 48, 64, 96, 128, 192, 256, 384, 512])
def test_every_supported_bf16_shape_gets_a_configuration(lib, C):
    # channel counts the tensor-core kernels accept, against flat and row-aligned frame widths
    for Cout in (3, C, 2 * C if 2 * C <= 512 else C // 2):
        for W in (1, 17, 100, 128, 200, 254, 256, 300, 640, 2560):
            for H in (1, 8, 1440):
                p = cc3d.cc3d_plan_create(C, Cout, H, W, 3, 3, 3, cc3d.CC3D_BF16)
                cc3d.cc3d_destroy(p)
        for k in ((2, 3, 3), (3, 1, 1), (1, 1, 1)):
            p = cc3d.cc3d_plan_create(C, C, 64, 100, *k, cc3d.CC3D_BF16)
            cc3d.cc3d_destroy(p)
        p = cc3d.cc3d_plan_create_upsample2x(C, C, 32, 100, 3, cc3d.CC3D_BF16)
        cc3d.cc3d_destroy(p)


# The launch configuration each decoder layer's chunk gets (host-only): the kernel, its stage
# rings and its tile count, as measured and described in the design notes.  A change to the
# selection logic shows up here before any GPU run.
@pytest.mark.parametrize("plan_args,T,expect", [
    (dict(Cin=96, Cout=96, H=360, W=640), 4,
     dict(kernel="tc2s_bf16_kernel", pair=1, two_frame=1, NT=96, row_aligned=1, tap_rows_per_weight_stage=3,
          window_stages=3, weight_stages=2, acc_stages=1, smem_bytes=213376, tiles=1800,
          history_frames_on_copy_engine=1)),
    (dict(Cin=96, Cout=96, H=360, W=640), 1,
     dict(kernel="tc2_bf16_kernel", pair=1, two_frame=0, acc_stages=2, tiles=900, history_frames_on_copy_engine=2)),
    (dict(Cin=192, Cout=192, H=180, W=320), 4,
     dict(kernel="tc2_bf16_kernel", row_aligned=0, NT=192, tap_rows_per_weight_stage=1, weight_stages=6,
          tiles=912, history_frames_on_copy_engine=2)),
    (dict(Cin=192, Cout=192, H=180, W=320), 3,
     dict(kernel="tc_bf16_kernel", pair=0, weight_stages=3, history_frames_on_copy_engine=0)),
    (dict(Cin=384, Cout=384, H=90, W=160), 4, dict(kernel="tc2_bf16_kernel", cout_blocks=2, NT=192, tiles=456)),
    (dict(Cin=384, Cout=192, H=90, W=160), 4, dict(kernel="tc2_bf16_kernel", cout_blocks=1, tiles=228)),
    (dict(Cin=96, Cout=96, H=1440, W=2560), 4, dict(kernel="tc2s_bf16_kernel", tiles=28800)),
    (dict(Cin=96, Cout=96, H=360, W=640, kt=2), 4,
     dict(kernel="tc2s_bf16_kernel", two_frame=1, history_frames_on_copy_engine=1)),
    (dict(Cin=96, Cout=3, H=1440, W=2560), 4, dict(kernel="head_bf16_kernel", column_strips=21)),
    (dict(Cin=96, Cout=96, H=360, W=640, kt=3, kh=1, kw=1), 4,
     dict(kernel="stream_bf16_kernel", position_blocks=1800)),
    (dict(Cin=16, Cout=16, H=32, W=32, dtype="f32"), 4, dict(kernel="simt_f32_kernel", launches=2)),
])
def test_describe_reports_the_measured_configurations(lib, plan_args, T, expect):
    plan = cc3d.CausalConv3dPlan(**plan_args)
    try:
        got = plan.describe(T)
    finally:
        plan.close()
    assert {k: got.get(k) for k in expect} == expect


def test_describe_of_the_fused_upsample_plan(lib):
    plan = cc3d.Upsample2xConvPlan(96, 96, 180, 320)
    try:
        got = plan.describe(4)
    finally:
        plan.close()
    assert got["kernel"] == "tc_bf16_kernel" and got["up2"] == 1 and got["pair"] == 0


@pytest.mark.parametrize("C", [16, 32, 64, 96, 192, 384])
def test_every_tensor_core_configuration_fits_the_sm(lib, C):
    # shared memory within the 227 KB a block may take (static barriers included), tensor memory
    # within 512 columns, at least double-buffered rings, and the two-frame schedule only where
    # the epilogue can hold two 96-column row groups
    for Cout in (C, C // 2 if C >= 32 else C):
        for H, W in ((8, 100), (360, 640), (90, 160), (1440, 2560), (5, 254)):
            for kt in (2, 3):
                plan = cc3d.CausalConv3dPlan(C, Cout, H, W, kt)
                try:
                    for T in (1, 2, 3, 4, 5):
                        d = plan.describe(T, has_residual=(T % 2 == 0))
                        assert d["kernel"] in ("tc_bf16_kernel", "tc2_bf16_kernel", "tc2s_bf16_kernel")
                        assert d["smem_bytes"] + 1024 <= 227 * 1024, d
                        assert d["tmem_cols"] <= 512 and d["tmem_cols"] & (d["tmem_cols"] - 1) == 0, d
                        assert 2 <= d["window_stages"] <= 8 and 2 <= d["weight_stages"] <= 8, d
                        assert d["tiles"] >= 1
                        if d["two_frame"]:
                            assert d["pair"] == 1 and d["NT"] <= 96 and T >= 2, d
                finally:
                    plan.close()


def test_describe_rejects_bad_arguments(lib):
    plan = cc3d.cc3d_plan_create(96, 96, 360, 640, 3, 3, 3, cc3d.CC3D_BF16)
    try:
        buf = ctypes.create_string_buffer(16)
        assert lib.cc3d_plan_describe(plan, 4, 1, buf, len(buf)) == 1  # line longer than the buffer
        assert buf.value == b""
        big = ctypes.create_string_buffer(1024)
        assert lib.cc3d_plan_describe(plan, 0, 1, big, len(big)) == 1
        assert lib.cc3d_plan_describe(None, 4, 1, big, len(big)) == 1
        assert lib.cc3d_plan_describe(plan, 4, 1, None, 0) == 1
        assert lib.cc3d_plan_describe(plan, 4, 1, big, len(big)) == 0
        assert big.value.startswith(b"kernel=tc2s_bf16_kernel ")
    finally:
        cc3d.cc3d_destroy(plan)


def test_plan_methods_check_tensor_sizes_before_the_call(lib):
    # the C ABI sees bare pointers: the plan object rejects a tensor whose element count or dtype
    # does not match the plan before any pointer reaches the library
    import torch
    bf = torch.bfloat16
    T, H, W, C = 2, 4, 8, 32
    plan = cc3d.CausalConv3dPlan(C, C, H, W)
    x = torch.zeros((T, H, W, C), dtype=bf)
    w = torch.zeros((C, 3, 3, 3, C), dtype=bf)
    y = torch.zeros((T, H, W, C), dtype=bf)
    cache = torch.zeros((2, H, W, C), dtype=bf)
    bad = [
        dict(x=torch.zeros((T, H, W, C // 2), dtype=bf)),
        dict(w=torch.zeros((C, 2, 3, 3, C), dtype=bf)),
        dict(b=torch.zeros((C + 1,), dtype=bf)),
        dict(residual=torch.zeros((T + 1, H, W, C), dtype=bf)),
        dict(cache_in=torch.zeros((1, H, W, C), dtype=bf)),
        dict(cache_out=torch.zeros((2, H, W + 1, C), dtype=bf)),
        dict(y=torch.zeros((T, H, W, C), dtype=torch.float32)),
        dict(w=torch.zeros((C, 3, 3, 3, C), dtype=torch.float32)),
    ]
    for kw in bad:
        args = dict(x=x, w=w, b=None, residual=None, cache_in=None, cache_out=cache, y=y)
        args.update(kw)
        with pytest.raises(ValueError, match=next(iter(kw))):
            plan.forward_chunk(**args)
    with pytest.raises(ValueError, match="cache"):
        plan.reset(torch.zeros((3, H, W, C), dtype=bf))
    with pytest.raises(ValueError, match="y has dtype"):
        plan.forward_chunk_u8(x, w, None, None, None, cache, y)
    # matching sizes pass the check and stop at the device-memory check of the binding
    with pytest.raises(ValueError, match="CUDA"):
        plan.forward_chunk(x, w, None, None, None, cache, y)
    plan.close()
    # the fused upsample: outputs and residual are 2H x 2W, the history holds source frames
    up = cc3d.Upsample2xConvPlan(C, C, H, W)
    with pytest.raises(ValueError, match="residual"):
        up.forward_chunk(x, w, None, torch.zeros((T, H, W, C), dtype=bf), None, cache,
                         torch.zeros((T, 2 * H, 2 * W, C), dtype=bf))
    with pytest.raises(ValueError, match="CUDA"):
        up.forward_chunk(x, w, None, torch.zeros((T, 2 * H, 2 * W, C), dtype=bf), None, cache,
                         torch.zeros((T, 2 * H, 2 * W, C), dtype=bf))
    up.close()


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "cc3d.h"

int main(void)
{
    cc3d_plan_t plan = NULL;
    char line[1024];
    cc3d_status s = cc3d_plan_create(96, 96, 360, 640, 3, 3, 3, CC3D_BF16, &plan);
    if (s != CC3D_OK) { printf("create: %s\n", cc3d_status_string(s)); return 1; }
    s = cc3d_plan_describe(plan, 4, 1, line, sizeof line);
    if (s != CC3D_OK) { printf("describe: %s\n", cc3d_status_string(s)); return 2; }
    printf("%s\n%s\n", cc3d_plan_kernel(plan), line);
    /* argument checks run on the host before any device work */
    s = cc3d_forward_chunk(plan, 4, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL);
    printf("forward without buffers: %d\n", (int)s);
    cc3d_destroy(plan);
    cc3d_destroy(NULL);
    return 0;
}
"""


def test_a_plain_c_program_compiles_links_and_calls_the_library(lib, tmp_path):
    # the boundary is a C ABI: the header compiles as strict C99 on its own, and a C program links
    # libcc3d.so and calls its host-only entry points with no Python or PyTorch involved
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_cc3d.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_cc3d"
    libdir = os.path.dirname(cc3d.library_path())
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.dirname(HEADER),
                    str(src), "-o", str(exe), "-L", libdir, "-lcc3d", "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout.splitlines()
    assert out[0] == "tc_bf16_pair"
    assert out[1].startswith("kernel=tc2s_bf16_kernel ")
    assert out[2] == "forward without buffers: 1"


def test_schedule_knobs_are_validated_and_plan_local(lib):
    p = cc3d.cc3d_plan_create(96, 96, 360, 640, 3, 3, 3, cc3d.CC3D_BF16)
    q = cc3d.cc3d_plan_create(96, 96, 360, 640, 3, 3, 3, cc3d.CC3D_BF16)
    try:
        f = lib.cc3d_debug_set_schedule
        assert f(None, 0, 1) == 1                              # null plan
        assert f(p, -1, 0) == 1 and f(p, 12, 0) == 1           # unknown knobs
        for knob, bad in ((0, 2), (1, -2), (4, 3), (5, 3), (5, 8), (6, 3), (7, 2), (8, 1), (9, 9), (10, 4), (11, 24),
                          (11, 64)):
            assert f(p, knob, bad) == 1, (knob, bad)
        assert cc3d.cc3d_plan_describe(p, 4)["kernel"] == "tc2s_bf16_kernel"
        cc3d.cc3d_debug_set_schedule(p, "channel_block", 16)
        assert cc3d.cc3d_plan_describe(p, 4)["channel_block"] == 16
        cc3d.cc3d_debug_set_schedule(p, "channel_block", -1)
        assert cc3d.cc3d_plan_describe(p, 4)["channel_block"] == 32
        cc3d.cc3d_debug_set_schedule(p, "two_frame", 0)
        assert cc3d.cc3d_plan_describe(p, 4)["kernel"] == "tc2_bf16_kernel"
        cc3d.cc3d_debug_set_schedule(p, "pair", 0)
        assert cc3d.cc3d_plan_describe(p, 4)["kernel"] == "tc_bf16_kernel"
        # another plan of the same shape keeps its defaults
        assert cc3d.cc3d_plan_describe(q, 4)["kernel"] == "tc2s_bf16_kernel"
        cc3d.cc3d_debug_set_schedule(p, "pair", -1)
        cc3d.cc3d_debug_set_schedule(p, "two_frame", -1)
        assert cc3d.cc3d_plan_describe(p, 4) == cc3d.cc3d_plan_describe(q, 4)
        # a combination with no configuration is refused when the chunk is described (or run)
        # (SM pairs hold at most two 128-row groups per block)
        cc3d.cc3d_debug_set_schedule(p, "row_groups", 4)
        with pytest.raises(cc3d.CC3DError) as e:
            cc3d.cc3d_plan_describe(p, 1)
        assert e.value.code == 2
    finally:
        cc3d.cc3d_destroy(p)
        cc3d.cc3d_destroy(q)


def test_launch_configuration_ignores_the_environment(lib):
    """The library reads no environment variable: a process that carries old tuning variables
    gets the measured configuration."""
    import subprocess
    import sys
    code = ("import json, chunked_causal_convolution_gb300 as c;"
            "p = c.cc3d_plan_create(96, 96, 360, 640); print(json.dumps(c.cc3d_plan_describe(p, 4)))")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root)
    plain = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    env.update({"CC3D_TC_PAIR": "0", "CC3D_TC_TSTACK": "0", "CC3D_TC_NA": "5", "CC3D_TC_RB": "1",
                "CC3D_TC_SUB": "1"})
    tuned = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    assert plain.stdout == tuned.stdout and "tc2s_bf16_kernel" in plain.stdout
    src = os.path.join(root, "chunked_causal_convolution_gb300", "csrc")
    for name in os.listdir(src):
        assert "getenv" not in open(os.path.join(src, name)).read(), name


def test_binding_refuses_a_tensor_of_another_device(monkeypatch):
    """A CUDA tensor on another device than the current one is refused before any pointer reaches
    the library (the C ABI compares the pointer's device with the current one as well)."""
    import torch

    class FakeCudaTensor:
        is_cuda = True
        device = torch.device("cuda", 1)

        def is_contiguous(self):
            return True

        def data_ptr(self):
            return 0x10000

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(ValueError, match="current device"):
        cc3d._addr(FakeCudaTensor())
    FakeCudaTensor.device = torch.device("cuda", 0)
    assert cc3d._addr(FakeCudaTensor()) == 0x10000


def test_group_create_checks_the_layer_chain(lib):
    a = cc3d.cc3d_plan_create(96, 64, 36, 64, 3, 3, 3, cc3d.CC3D_BF16)
    b = cc3d.cc3d_plan_create(64, 32, 36, 64, 1, 1, 1, cc3d.CC3D_BF16)
    c = cc3d.cc3d_plan_create(96, 32, 36, 64, 3, 3, 3, cc3d.CC3D_BF16)   # Cin does not follow a
    d = cc3d.cc3d_plan_create(64, 32, 18, 32, 3, 3, 3, cc3d.CC3D_BF16)   # frame size does not follow a
    u = cc3d.cc3d_plan_create_upsample2x(32, 16, 36, 64, 3, cc3d.CC3D_BF16)  # reads b's output, doubles it
    v = cc3d.cc3d_plan_create(16, 3, 72, 128, 3, 3, 3, cc3d.CC3D_BF16)
    try:
        arr = lambda *ps: (ctypes.c_void_p * len(ps))(*ps)  # noqa: E731
        g = ctypes.c_void_p(1)
        assert lib.cc3d_group_create(0, arr(a), 1, ctypes.byref(g)) == 1 and g.value is None
        assert lib.cc3d_group_create(1, arr(a), -1, ctypes.byref(g)) == 1
        assert lib.cc3d_group_create(2, arr(a, c), 1, ctypes.byref(g)) == 1
        assert lib.cc3d_group_create(2, arr(a, d), 1, ctypes.byref(g)) == 1
        assert lib.cc3d_group_create(2, arr(a, None), 1, ctypes.byref(g)) == 1
        h = cc3d.cc3d_group_create([a, b, u, v], 2)
        cc3d.cc3d_group_destroy(h)
    finally:
        for p in (a, b, c, d, u, v):
            cc3d.cc3d_destroy(p)


def test_group_workspace_sizes(lib):
    """Two buffers for the intermediate batches (each one batch of the largest output it holds),
    plus one more history per causal layer when a chunk takes several batches; 256-byte sections."""
    H, W = 360, 640
    px = H * W
    a = cc3d.cc3d_plan_create(96, 96, H, W, 3, 3, 3, cc3d.CC3D_BF16)
    b = cc3d.cc3d_plan_create(96, 192, H, W, 1, 1, 1, cc3d.CC3D_BF16)
    c = cc3d.cc3d_plan_create(192, 3, H, W, 3, 3, 3, cc3d.CC3D_BF16)
    try:
        g1 = cc3d.cc3d_group_create([a, b, c], 1)
        g0 = cc3d.cc3d_group_create([a, b, c], 0)
        gs = cc3d.cc3d_group_create([a], 1)
        # frame batch 1, 4-frame chunks: buffer 0 holds a's 96-channel frame, buffer 1 b's
        # 192-channel frame; histories of a (2 x 96 channels) and c (2 x 192 channels)
        exp1 = px * 96 * 2 + px * 192 * 2 + 2 * px * 96 * 2 + 2 * px * 192 * 2
        assert cc3d.cc3d_group_workspace_bytes(g1, 4) == exp1
        assert cc3d.cc3d_group_workspace_bytes(g1, 1) == px * 96 * 2 + px * 192 * 2  # one batch: no extra history
        # whole chunk: both intermediates of all 4 frames, no extra history
        assert cc3d.cc3d_group_workspace_bytes(g0, 4) == 4 * (px * 96 * 2 + px * 192 * 2)
        assert cc3d.cc3d_group_workspace_bytes(g0, 0) == 0
        # a single layer needs only its second history
        assert cc3d.cc3d_group_workspace_bytes(gs, 4) == 2 * px * 96 * 2
        assert cc3d.cc3d_group_workspace_bytes(gs, 1) == 0
        # odd sizes are rounded up to 256-byte sections
        o1 = cc3d.cc3d_plan_create(16, 16, 3, 5, 1, 1, 1, cc3d.CC3D_BF16)
        o2 = cc3d.cc3d_plan_create(16, 16, 3, 5, 1, 1, 1, cc3d.CC3D_BF16)
        go = cc3d.cc3d_group_create([o1, o2], 1)
        assert cc3d.cc3d_group_workspace_bytes(go, 3) == 512  # 15 * 16 * 2 = 480 -> 512
        for h in (g1, g0, gs, go):
            cc3d.cc3d_group_destroy(h)
        for p in (o1, o2):
            cc3d.cc3d_destroy(p)
    finally:
        for p in (a, b, c):
            cc3d.cc3d_destroy(p)


def test_group_forward_rejects_before_any_device_work(lib):
    a = cc3d.cc3d_plan_create(32, 32, 4, 8, 3, 3, 3, cc3d.CC3D_BF16)
    b = cc3d.cc3d_plan_create(32, 16, 4, 8, 1, 1, 1, cc3d.CC3D_BF16)
    g = cc3d.cc3d_group_create([a, b], 1)
    try:
        need = cc3d.cc3d_group_workspace_bytes(g, 2)
        buf = (ctypes.c_uint8 * (1 << 20))()
        base = (ctypes.addressof(buf) + 255) & ~255
        x, y, w0, w1, c0, c1, ws = (base, base + 8192, base + 16384, base + 81920, base + 98304, base + 106496,
                                    base + 131072)
        W = (ctypes.c_void_p * 2)(w0, w1)
        CO = (ctypes.c_void_p * 2)(c1, None)
        f = lib.cc3d_group_forward_chunk
        assert f(None, 2, x, W, None, None, CO, y, ws, need, None) == 1          # null group
        assert f(g, -1, x, W, None, None, CO, y, ws, need, None) == 1            # negative T
        assert f(g, 2, x, None, None, None, CO, y, ws, need, None) == 1          # no weights
        assert f(g, 2, x, W, None, None, None, y, ws, need, None) == 1           # no histories
        assert f(g, 2, x, W, None, None, CO, y, ws, need - 1, None) == 1         # workspace too small
        assert f(g, 2, x, W, None, None, CO, y, None, need, None) == 1           # no workspace
        assert f(g, 2, x, W, None, None, CO, y, ws + 16, need, None) == 3        # workspace misaligned
        assert f(g, 2, x, W, None, None, CO, y, x, need, None) == 4              # workspace over x
        assert f(g, 2, x, W, None, None, CO, y, w0, need, None) == 4             # workspace over a weight
        # host memory: refused by the check of the first launch, nothing launched
        assert f(g, 2, x, W, None, None, CO, y, ws, need, None) == 8
    finally:
        cc3d.cc3d_group_destroy(g)
        cc3d.cc3d_destroy(a)
        cc3d.cc3d_destroy(b)


def test_frame_batching_holds_one_batch_of_intermediates(lib):
    """The decoder tail at the c96 stage (two 96-channel 3x3x3 convs and the 3-channel head) on the
    pages' 24-frame chunks: batches of one frame hold two intermediate frames and one more history
    per layer, the whole chunk at once holds both 24-frame intermediates."""
    H, W = 360, 640
    plans = [cc3d.CausalConv3dPlan(96, 96, H, W), cc3d.CausalConv3dPlan(96, 96, H, W),
             cc3d.CausalConv3dPlan(96, 3, H, W)]
    frame = H * W * 96 * 2
    whole = cc3d.LayerGroup(plans, 0).workspace_bytes(24)
    one = cc3d.LayerGroup(plans, 1).workspace_bytes(24)
    two = cc3d.LayerGroup(plans, 2).workspace_bytes(24)
    assert whole == 2 * 24 * frame
    assert one == 2 * frame + 3 * 2 * frame
    assert two == 2 * 2 * frame + 3 * 2 * frame
    assert whole / one == 6.0
