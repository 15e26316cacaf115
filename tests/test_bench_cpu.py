"""Host logic of bench.py that needs no GPU: the roofline's traffic record is used only for the
kernel source and workload it was captured on, clock samples are summarised with their throttle
reasons, the peaks come from the measured file, and the workload's FLOP count is the metric's."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_traffic_record_is_used_only_for_its_kernel_source_and_workload(monkeypatch):
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: rec["kernel_source_sha"])
    assert bench.traffic_per_launch(rec["workload"]) == float(rec["dram_bytes_per_launch"])
    assert bench.traffic_per_launch("c192") is None
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "0" * 16)
    assert bench.traffic_per_launch(rec["workload"]) is None


def test_traffic_record_is_a_plausible_capture():
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"]
    # DRAM traffic well above the algorithmic bytes would mean re-reads; far below, a wrong capture
    ratio = rec["dram_bytes_per_launch"] / rec["algorithmic_bytes_per_launch"]
    assert 0.5 < ratio < 1.5, ratio


def test_kernel_source_hash_covers_the_tensor_core_kernels():
    names = {os.path.basename(p) for p in bench.KERNEL_SOURCES}
    assert {"cc3d_tc.cu", "cc3d_tc2.cu", "cc3d_tc2s.cu", "cc3d_tc_common.cuh", "cc3d_ptx.cuh"} <= names
    assert len(bench.kernel_source_sha()) == 16


def test_clock_summary_reports_median_max_and_active_reasons():
    s = bench.ClockSampler(0)
    s.lines = [
        "2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1965, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    out = s.summary()
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    s.lines = ["1500, 2070, 1000, 0x8, Active, Not Active, Active, Not Active"]
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s.lines = []
    assert s.summary()["samples"] == 0 and s.summary()["sm_mhz"] is None


def test_peaks_come_from_the_measured_file_when_present():
    p, kind = bench.peaks()
    if os.path.exists(bench.PEAKS_FILE):
        assert kind == "measured"
        with open(bench.PEAKS_FILE) as f:
            assert p["bf16_tflops"] == json.load(f)["bf16_tflops"]
    else:
        assert kind == "fallback" and p == bench.FALLBACK_PEAKS


@pytest.mark.parametrize("name", ["c96_residual", "c192", "c384", "c384_to_192", "memblock_c96", "up2_c96"])
def test_workload_config_states_the_flop_count_and_the_l2_rule(name):
    wl = synth.WORKLOADS[name]
    cfg = bench.workload_config(wl)
    Ho, Wo = wl.out_hw
    assert cfg["flop_per_step"] == 2 * wl.Cin * wl.Cout * wl.kt * wl.kh * wl.kw * wl.T * Ho * Wo
    assert cfg["workload"].startswith(name + ": causal conv3d")
    assert "larger than L2" in cfg["l2"]
    # inputs larger than L2 is what lets the bench skip the flush
    assert wl.T * wl.H * wl.W * wl.Cin * 2 > 129e6


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the fp64 oracle on the host cores) prints exactly one JSON line
    with the keys of the bench contract, on the headline workload, with no GPU."""
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "3", "--ref-rows", "2"], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] >= 3 and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("c96_residual")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
