"""Benchmark of the chunked causal 3-D convolution on GB300.

One step = one pass of the whole hot path over one decoder layer's worth of
frames: the chunk loop (chunks of 4 frames, the 2-frame temporal cache carried
from chunk to chunk in two ping-pong buffers), each chunk one launch of the
tensor-core kernel (implicit-GEMM conv + bias + residual epilogue + cache
update).  Inputs are resident in HBM before the timed region and larger than
L2.  Prints one JSON line (rank 0).

The same line carries, under "configs", the other decoder stages of the target
(c192, c384, c384_to_192: the same 6 x 4-frame step, warm-up and timing, each
with its clocks) and "sr_stream": the 4x super-resolution stage (the 96 -> 96
conv, then the 96 -> 3 head on its output) over all 361 frames of 1440 x 2560
in 90 chunks of 4 and one of 1.  Its "e2e" object adds the box's own pinned-copy
floor for the step's host<->device bytes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--no-configs] [--sr-passes P]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (host cores), printing the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal conv3d TFLOP/s"
UNIT = "TFLOP/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "tc_bf16_kernel_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "chunked_causal_convolution_gb300", "csrc", f)
                  for f in ("cc3d_tc.cu", "cc3d_tc2.cu", "cc3d_tc2s.cu", "cc3d_tc_common.cuh", "cc3d_ptx.cuh")]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_per_launch(workload):
    """DRAM bytes per launch from the committed ncu capture, if it was taken on this kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("kernel_source_sha") == kernel_source_sha() and t.get("workload") == workload:
            return float(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_config(wl):
    Ho, Wo = wl.out_hw
    frame = ("H=%d W=%d" % (wl.H, wl.W) if not wl.up2 else
             "input H=%d W=%d read through a nearest-2x upsample, output H=%d W=%d" % (wl.H, wl.W, Ho, Wo))
    return {
        "workload": "%s: causal conv3d Cin=%d Cout=%d k=%dx%dx%d, T=%d frames in chunks %s with a %d-frame "
                    "cache, %s, batch 1, bias%s" % (
                        wl.name, wl.Cin, wl.Cout, wl.kt, wl.kh, wl.kw, wl.T,
                        "x".join(str(c) for c in sorted(set(wl.chunks))), wl.kt - 1,
                        frame, " + residual" if wl.r is not None else ""),
        "Cin": wl.Cin, "Cout": wl.Cout, "T": wl.T, "H": wl.H, "W": wl.W, "chunks": list(wl.chunks),
        "flop_per_step": wl.flops,
        "l2": "inputs larger than L2 (%.2f GB per activation tensor vs 129 MB L2), no flush" % (
            wl.T * wl.H * wl.W * wl.Cin * 2 / 1e9),
    }


# ---------------------------------------------------------------- ranks

def max_over_ranks(x, dist=None, device="cpu"):
    """The largest value of x over all ranks (the job's time is its slowest rank's); x itself
    when there is one rank.  device is where the reduction tensor lives (cuda for NCCL, cpu for
    gloo)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle sample

def oracle_sample(wl, rows, nthreads=None):
    """Time the oracle's chunk form on one output frame (first `rows` rows) of the workload, from its
    2-frame history: returns (metric FLOPs of the outputs computed, seconds, threads).  For an
    upsampling layer the oracle upsamples rows/2 source rows and convolves the result."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    import synth
    from synth import native

    t0 = wl.T // 2
    H, W, C = (rows // 2 if wl.up2 else rows), wl.W, wl.Cin

    def gen(tid, dist, shape, frame0):
        # rows 0..rows-1 of frames frame0.. of the global video
        f, h = np.meshgrid(np.arange(shape[0]), np.arange(shape[1]), indexing="ij")
        base = ((frame0 + f) * wl.H + h) * wl.W * shape[3]
        e = base[..., None, None] + (np.arange(shape[2])[:, None] * shape[3] + np.arange(shape[3]))[None, None]
        parts = np.array_split(e.reshape(-1), 16)
        with ThreadPoolExecutor(16) as ex:
            vals = list(ex.map(lambda p: native.values_host(wl.seed, tid, dist, p, wl.dtype), parts))
        raw = np.concatenate(vals).reshape(shape)
        return synth.bf16_bits_to_f64(raw) if wl.dtype == "bf16" else raw.astype(np.float64)

    P = wl.kt - 1
    hist = gen(synth.TID_X, wl.x, (P, H, W, C), t0 - P) if P > 0 else None
    x = gen(synth.TID_X, wl.x, (1, H, W, C), t0)
    w = synth.bf16_bits_to_f64(native.values_host(wl.seed, synth.TID_W, wl.w,
                                                  synth.dense_index((wl.Cout, wl.kt, wl.kh, wl.kw, C)), wl.dtype))
    b = synth.bf16_bits_to_f64(native.values_host(wl.seed, synth.TID_B, wl.b, np.arange(wl.Cout), wl.dtype))
    r = gen(synth.TID_R, wl.r, (1, H, W, wl.Cout), t0) if wl.r is not None and not wl.up2 else None
    n = nthreads or oracle.default_threads()
    ts = time.perf_counter()
    if wl.up2:
        x = oracle.upsample_nearest2x(x)
        hist = oracle.upsample_nearest2x(hist) if hist is not None else None
    oracle.conv_chunk(x, w, b, r, hist, nthreads=n)
    dt = time.perf_counter() - ts
    flops = 2.0 * wl.Cin * wl.Cout * wl.kt * wl.kh * wl.kw * x.shape[1] * x.shape[2]
    return flops, dt, n


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(wl, rows)
    times, flops, n = [], 0.0, 1
    for _ in range(args.steps):
        flops, dt, n = oracle_sample(wl, rows)
        times.append(dt)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    sample = ("fp64 oracle chunk form: %d of %d rows of one output frame (frame %d) of %s from its 2-frame "
              "history, per step" % (rows, wl.H, wl.T // 2, wl.name))
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def _dominant_bound(wl, c_full, frame_in, frame_out, has_res, p):
    """Bound of a full-chunk launch of the layer, its FLOPs and algorithmic bytes: tensor cores
    unless its arithmetic intensity (history in and out included) is below the ridge."""
    flop_per_launch = wl.flops / wl.T * c_full
    bytes_per_launch = (c_full * frame_in + c_full * frame_out * (2 if has_res else 1)
                        + 2 * (wl.kt - 1) * frame_in)
    ridge = float(p["bf16_tflops"]) * 1e12 / (float(p["hbm_gbs"]) * 1e9)
    return flop_per_launch, bytes_per_launch, flop_per_launch / bytes_per_launch < ridge


def measure_layer(wl, args, dev, dist, local, world, keep=False):
    """One layer's bench step (its chunk loop, histories ping-ponged) on resident inputs: W warm-up
    steps, then K timed steps with CUDA events on the launching stream, a per-launch event pair
    around every chunk, and the SM clocks sampled meanwhile.  Returns the measurements (and, with
    keep, the tensors and plan for the end-to-end leg)."""
    import torch

    import chunked_causal_convolution_gb300 as cc3d
    import synth
    from synth import native

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    dt = torch.bfloat16
    T, H, W = wl.T, wl.H, wl.W
    Ho, Wo = wl.out_hw  # output frames (2H x 2W for an upsampling layer)
    x = native.fill_device(torch.empty((T, H, W, wl.Cin), dtype=dt, device=dev), wl.seed, synth.TID_X, wl.x)
    wt = native.fill_device(torch.empty((wl.Cout, wl.kt, wl.kh, wl.kw, wl.Cin), dtype=dt, device=dev), wl.seed,
                            synth.TID_W, wl.w)
    b = native.fill_device(torch.empty((wl.Cout,), dtype=dt, device=dev), wl.seed, synth.TID_B, wl.b)
    r = None
    if wl.r is not None:
        r = native.fill_device(torch.empty((T, Ho, Wo, wl.Cout), dtype=dt, device=dev), wl.seed, synth.TID_R, wl.r)
    y = torch.empty((T, Ho, Wo, wl.Cout), dtype=dt, device=dev)
    if wl.up2:
        plan = cc3d.Upsample2xConvPlan(wl.Cin, wl.Cout, H, W, wl.kt, dtype="bf16")
    else:
        plan = cc3d.CausalConv3dPlan(wl.Cin, wl.Cout, H, W, wl.kt, wl.kh, wl.kw, dtype="bf16")
    caches = [plan.new_cache(dev), plan.new_cache(dev)]
    stream = torch.cuda.Stream(device=dev)
    bounds = []
    s = 0
    for c in wl.chunks:
        bounds.append((s, c))
        s += c
    # N > 1 ranks: the video is split along time, rank i owning frames [i*T, (i+1)*T); before its
    # chunk loop every rank receives the kt - 1 input frames before its range from rank i - 1 (the
    # causal halo exchange, NCCL point-to-point; zeros on rank 0) and its first chunk reads them
    halo_hist = plan.new_cache(dev) if (dist is not None and wl.kt > 1) else None

    def step(ev_pairs=None):
        first_hist = None
        if halo_hist is not None:
            from chunked_causal_convolution_gb300 import halo
            first_hist = halo.exchange(x, wl.kt - 1, out=halo_hist)
        for k, (s0, c) in enumerate(bounds):
            if ev_pairs is not None:
                ev_pairs[k][0].record(stream)
            cc3d.cc3d_forward_chunk(plan.handle, c, x[s0:s0 + c], wt, b, r[s0:s0 + c] if r is not None else None,
                                    caches[k % 2] if k else first_hist, caches[(k + 1) % 2], y[s0:s0 + c], stream)
            if ev_pairs is not None:
                ev_pairs[k][1].record(stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    st = plan.status(stream)
    if st != 0:
        raise RuntimeError("%s: device status after warm-up: %s" % (wl.name, cc3d.cc3d_status_string(st)))

    # ---- timed region: K steps, events on the launching stream
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launch_evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in bounds] for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clocks:
        time.sleep(0.25)
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(args.steps):
                step(launch_evs[i])
            end.record(stream)
        stream.synchronize()
        time.sleep(0.25)
    barrier()
    ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    st = plan.status(stream)
    if st != 0:
        raise RuntimeError("%s: device status after timing: %s" % (wl.name, cc3d.cc3d_status_string(st)))
    ms_per_step = ms / args.steps
    value = wl.flops * world * args.steps / (ms / 1e3) / 1e12
    # per-step durations (first launch start to last launch end of each step) and algorithmic bytes
    step_ms = sorted(row[0][0].elapsed_time(row[-1][1]) for row in launch_evs)
    step_stats = {"min": step_ms[0], "mean": sum(step_ms) / len(step_ms),
                  "p99": step_ms[min(len(step_ms) - 1, int(round(0.99 * (len(step_ms) - 1))))]}
    frame_in, frame_out = H * W * wl.Cin * 2, Ho * Wo * wl.Cout * 2
    bytes_per_step = 0
    for k, (_, c) in enumerate(bounds):
        bytes_per_step += c * frame_in + c * frame_out * (2 if r is not None else 1)  # x, y (+ residual)
        bytes_per_step += ((wl.kt - 1) * frame_in if k else 0) + (wl.kt - 1) * frame_in  # history read, written
    p, src = peaks()
    hbm_gbs = bytes_per_step * world / (ms_per_step / 1e3) / 1e9
    # per-launch durations of the dominant (only) kernel
    launch_ms = [a.elapsed_time(bb) for row in launch_evs for (a, bb) in row]
    c_full = max(wl.chunks)
    full = [ms_ for ms_, (_, c) in zip(launch_ms, bounds * args.steps) if c == c_full]
    avg_launch_ms = sum(full) / len(full)
    flop_per_launch, bytes_per_launch, hbm_bound = _dominant_bound(wl, c_full, frame_in, frame_out, r is not None, p)
    if hbm_bound:
        achieved = bytes_per_launch / (avg_launch_ms / 1e3) / 1e9
        peak = float(p["hbm_gbs"])
    else:
        achieved = flop_per_launch / (avg_launch_ms / 1e3) / 1e12
        peak = float(p["bf16_tflops"])
    peak_note = "%s MEASURED_PEAKS %s" % (src, "hbm_gbs (copy bandwidth)" if hbm_bound else
                                           "bf16_tflops (burst, kernel timed alone)")
    out = {
        "value": value, "ms_per_step": ms_per_step, "kernel": plan.kernel,
        "time_split": (None if halo_hist is None else
                       "%d ranks, each %d frames; the %d-frame input history exchanged point-to-point before "
                       "each step's chunk loop" % (world, T, wl.kt - 1)),
        "dominant_kernel": plan.describe(c_full, r is not None).get("kernel"),
        "output_frames_per_s": wl.T * world * args.steps / (ms / 1e3),
        "pct_of_dense_bf16_peak": {"measured_burst": 100 * value / world / float(p["bf16_tflops"]),
                                   "measured_sustained": 100 * value / world / float(p["bf16_tflops_sustained"]),
                                   "spec_2250": 100 * value / world / 2250.0},
        "roofline": {"bound": "hbm" if hbm_bound else "tensor", "achieved": achieved, "peak": peak,
                     "unit": "GB/s" if hbm_bound else "TFLOP/s", "frac": achieved / peak,
                     "traffic": traffic_per_launch(wl.name), "peak_source": peak_note, "kernel": plan.kernel,
                     "flop_per_launch": flop_per_launch, "algorithmic_bytes_per_launch": bytes_per_launch,
                     "avg_launch_ms": avg_launch_ms},
        "avg_launch_ms": avg_launch_ms,
        "clocks": clocks.summary(),
        "step_ms": step_stats,
        "hbm": {"achieved_gbs": hbm_gbs, "peak_gbs": float(p["hbm_gbs"]),
                "frac": hbm_gbs / world / float(p["hbm_gbs"]), "algorithmic_bytes_per_step": bytes_per_step},
        "gpu_launches": args.steps * len(bounds) * plan.launches_per_chunk,
    }
    if keep:
        out["_ctx"] = dict(x=x, wt=wt, b=b, r=r, y=y, plan=plan, caches=caches, stream=stream, bounds=bounds)
    else:
        plan.close()
        del x, wt, b, r, y, caches
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def measure_sr_stream(args, dev, local):
    """The 4x super-resolution output stage as a stream: the 96 -> 96 3x3x3 conv and the 96 -> 3
    head after it, over all 361 frames of 1440 x 2560 in 90 chunks of 4 and a last chunk of 1, both
    histories carried by the library from chunk to chunk, the head reading the conv's output.
    Inputs: a ring of two 4-frame chunks (the video's frames 0-3 and 4-7, generated on the device
    before the timed region) that chunk k reads in turn (k mod 2), so the 255 GB video never has
    to be resident; the work per chunk is the same.  One untimed pass, then `args.sr_passes`
    timed passes back to back (CUDA events around each pass and around every launch)."""
    import torch

    import chunked_causal_convolution_gb300 as cc3d
    import synth
    from synth import native

    conv_wl, head_wl = synth.WORKLOADS["sr96"], synth.WORKLOADS["sr_head3"]
    H, W, C = conv_wl.H, conv_wl.W, conv_wl.Cin
    dt = torch.bfloat16
    frame = H * W * C
    ring = [native.fill_device(torch.empty((4, H, W, C), dtype=dt, device=dev), conv_wl.seed, synth.TID_X, conv_wl.x,
                               offset=4 * j * frame) for j in range(2)]
    w1 = native.fill_device(torch.empty((96, 3, 3, 3, C), dtype=dt, device=dev), conv_wl.seed, synth.TID_W, conv_wl.w)
    b1 = native.fill_device(torch.empty((96,), dtype=dt, device=dev), conv_wl.seed, synth.TID_B, conv_wl.b)
    w2 = native.fill_device(torch.empty((3, 3, 3, 3, C), dtype=dt, device=dev), head_wl.seed, synth.TID_W, head_wl.w)
    b2 = native.fill_device(torch.empty((3,), dtype=dt, device=dev), head_wl.seed, synth.TID_B, head_wl.b)
    conv = cc3d.CausalConv3dPlan(C, 96, H, W)
    head = cc3d.CausalConv3dPlan(96, 3, H, W)
    c1 = [conv.new_cache(dev), conv.new_cache(dev)]
    c2 = [head.new_cache(dev), head.new_cache(dev)]
    y1 = torch.empty((4, H, W, 96), dtype=dt, device=dev)
    y2 = torch.empty((4, H, W, 3), dtype=dt, device=dev)
    stream = torch.cuda.Stream(device=dev)
    chunks = list(conv_wl.chunks)

    def one_pass(evs=None):
        for k, c in enumerate(chunks):
            if evs is not None:
                evs[k][0].record(stream)
            cc3d.cc3d_forward_chunk(conv.handle, c, ring[k % 2][:c], w1, b1, None, c1[k % 2] if k else None,
                                    c1[(k + 1) % 2], y1[:c], stream)
            if evs is not None:
                evs[k][1].record(stream)
            cc3d.cc3d_forward_chunk(head.handle, c, y1[:c], w2, b2, None, c2[k % 2] if k else None,
                                    c2[(k + 1) % 2], y2[:c], stream)
            if evs is not None:
                evs[k][2].record(stream)

    with torch.cuda.stream(stream):
        one_pass()
    for plan in (conv, head):
        st = plan.status(stream)
        if st != 0:
            raise RuntimeError("sr stream: device status after warm-up: %s" % cc3d.cc3d_status_string(st))
    passes = max(1, args.sr_passes)
    evs = [[tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in chunks] for _ in range(passes)]
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.25)
        with torch.cuda.stream(stream):
            for i in range(passes):
                one_pass(evs[i])
        stream.synchronize()
        time.sleep(0.25)
    for plan in (conv, head):
        st = plan.status(stream)
        if st != 0:
            raise RuntimeError("sr stream: device status after timing: %s" % cc3d.cc3d_status_string(st))
    pass_ms = [e[0][0].elapsed_time(e[-1][2]) for e in evs]
    conv_ms = [e[k][0].elapsed_time(e[k][1]) for e in evs for k, c in enumerate(chunks) if c == 4]
    head_ms = [e[k][1].elapsed_time(e[k][2]) for e in evs for k, c in enumerate(chunks) if c == 4]
    p, src = peaks()
    flops_conv, flops_head = conv_wl.flops, head_wl.flops
    total_s = sum(pass_ms) / 1e3
    conv_launch = sum(conv_ms) / len(conv_ms)
    head_launch = sum(head_ms) / len(head_ms)
    conv_tflops = flops_conv / conv_wl.T * 4 / (conv_launch / 1e3) / 1e12
    # the head's algorithmic bytes per 4-frame launch: x read, 2-frame history read and written, y
    head_bytes = 4 * H * W * C * 2 + 2 * 2 * H * W * C * 2 + 4 * H * W * 3 * 2
    head_gbs = head_bytes / (head_launch / 1e3) / 1e9
    out = {
        "workload": "sr_stream: 4x super-resolution output stage, causal conv3d 96->96 3x3x3 (bias) then the "
                    "96->3 3x3x3 head (bias) on its output, 361 frames of 1440x2560 in 90 chunks of 4 + 1 of 1, "
                    "both 2-frame histories carried through the library, batch 1",
        "inputs": "ring of two 4-frame input chunks (frames 0-3 and 4-7 of the seeded video, generated on the "
                  "device before the timed region), chunk k reads ring[k mod 2]; 2.83 GB per chunk (larger than L2)",
        "passes": passes, "ms_per_pass": total_s * 1e3 / passes,
        "value": (flops_conv + flops_head) * passes / total_s / 1e12, "unit": UNIT,
        "output_frames_per_s": conv_wl.T * passes / total_s,
        "flop_per_pass": flops_conv + flops_head,
        # a pass lasts about half a second under the power cap: the sustained peak is the
        # denominator (the burst fraction beside it)
        "conv": {"kernel": conv.describe(4, False).get("kernel"), "avg_launch_ms": conv_launch,
                 "tflops": conv_tflops, "frac": conv_tflops / float(p["bf16_tflops_sustained"]),
                 "peak": float(p["bf16_tflops_sustained"]),
                 "peak_source": src + " MEASURED_PEAKS bf16_tflops_sustained (kernel inside a long step)",
                 "frac_of_burst": conv_tflops / float(p["bf16_tflops"])},
        "head": {"kernel": head.describe(4, False).get("kernel"), "avg_launch_ms": head_launch,
                 "algorithmic_bytes_per_launch": head_bytes, "achieved_gbs": head_gbs,
                 "frac_of_hbm": head_gbs / float(p["hbm_gbs"]), "peak_gbs": float(p["hbm_gbs"]),
                 "peak_source": src + " MEASURED_PEAKS hbm_gbs (copy bandwidth)"},
        "clocks": clocks.summary(),
        "gpu_launches": passes * 2 * len(chunks),
    }
    conv.close()
    head.close()
    del ring, y1, y2, c1, c2
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def copy_bound(xh, rh, yh, x, r, y, dev, reps=3):
    """The box's own pinned-copy floor for the end-to-end step's bytes: the step's host->device
    bytes (x, then the residual) on one stream and its device->host bytes (y) on another, each as
    whole-tensor cudaMemcpyAsync calls, both directions at once; also each direction alone.  Best of
    `reps` (milliseconds)."""
    import torch

    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(h2d, d2h):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_in)
            s_out.wait_event(e0)
            if h2d:
                with torch.cuda.stream(s_in):
                    x.copy_(xh, non_blocking=True)
                    if rh is not None:
                        r.copy_(rh, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    yh.copy_(y, non_blocking=True)
            s_in.wait_stream(s_out)
            e1.record(s_in)
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1)
            best = t if best is None else min(best, t)
        return best

    return {"both_ms": timed(True, True), "h2d_only_ms": timed(True, False), "d2h_only_ms": timed(False, True)}


def run_ours(args, wl):
    import torch

    import chunked_causal_convolution_gb300 as cc3d
    import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()
    __graft_entry__.build()

    dev = torch.device("cuda", local)
    dt = torch.bfloat16
    m = measure_layer(wl, args, dev, dist, local, world, keep=True)
    ctx = m.pop("_ctx")
    x, wt, b, r, y, plan, caches, stream, bounds = (ctx[k] for k in ("x", "wt", "b", "r", "y", "plan", "caches",
                                                                    "stream", "bounds"))

    # ---- end to end: pinned host inputs -> device -> chunk loop -> host result, every step.
    # Steps are double-buffered on the device: step i's inputs (x, residual) go in as whole-tensor
    # copies on one copy stream while step i - 1's output goes out on another and the compute
    # stream runs the chunk loop of whichever step has its inputs; events order the reuse of every
    # buffer.  (Chunk-sized copies in both directions were measured to serialise on some boxes,
    # which put the step at the sum of the two directions instead of the larger one.)  The timed
    # region spans the first copy in to the last copy out.
    xh = x.cpu().pin_memory()
    rh = r.cpu().pin_memory() if r is not None else None
    yh = torch.empty(y.shape, dtype=dt).pin_memory()
    xb = [x, torch.empty_like(x)]
    rb = [r, torch.empty_like(r)] if r is not None else None
    yb = [y, torch.empty_like(y)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # step's inputs copied in
    ev_used = [torch.cuda.Event() for _ in range(2)]  # step's chunk loop done (inputs free, output ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # step's output copied out (output buffer free)
    e2e_count = [0]

    def e2e_step():
        j = e2e_count[0] % 2
        e2e_count[0] += 1
        s_in.wait_event(ev_used[j])
        with torch.cuda.stream(s_in):
            xb[j].copy_(xh, non_blocking=True)
            if rh is not None:
                rb[j].copy_(rh, non_blocking=True)
        ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])
        for k, (s0, c) in enumerate(bounds):
            cc3d.cc3d_forward_chunk(plan.handle, c, xb[j][s0:s0 + c], wt, b, rb[j][s0:s0 + c] if rb is not None else None,
                                    caches[k % 2] if k else None, caches[(k + 1) % 2], yb[j][s0:s0 + c], stream)
        ev_used[j].record(stream)
        s_out.wait_event(ev_used[j])
        with torch.cuda.stream(s_out):
            yh.copy_(yb[j], non_blocking=True)
        ev_out[j].record(s_out)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(args.steps):
        e2e_step()
    s_out.wait_stream(s_in)
    s_out.wait_stream(stream)
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    if not torch.equal(yh.to(dev), yb[(e2e_count[0] - 1) % 2]) or not torch.equal(yb[0], yb[1]):
        raise RuntimeError("end-to-end result differs from the device-resident result")
    h2d = x.numel() * 2 + (r.numel() * 2 if r is not None else 0)
    d2h = y.numel() * 2
    cb = copy_bound(xh, rh, yh, x, r, y, dev)
    e2e_step_ms = e2e_ms / args.steps
    plan.close()
    del x, r, y, xb, rb, yb, caches, ctx, xh, rh, yh
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # ---- the other decoder stages of the same target, each its own 6 x 4-frame step, and the
    # super-resolution stage as a 361-frame stream
    configs = {}
    if not args.no_configs:
        for name in ("c192", "c384", "c384_to_192"):
            if name == wl.name:
                continue
            mc = measure_layer(synth.WORKLOADS[name], args, dev, dist, local, world)
            configs[name] = {k: mc[k] for k in ("value", "ms_per_step", "output_frames_per_s", "avg_launch_ms",
                                                "kernel", "dominant_kernel", "clocks", "gpu_launches")}
            configs[name]["roofline"] = {k: mc["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac")}
            configs[name]["config"] = workload_config(synth.WORKLOADS[name])
        if world == 1:
            configs["sr_stream"] = measure_sr_stream(args, dev, local)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # whole output frames of the workload, repeated until about 10 s of CPU work
        flops, secs, reps = 0.0, 0.0, 0
        while secs < 10.0 and reps < 8:
            f, dt_, n = oracle_sample(wl, wl.H)
            flops, secs, reps = flops + f, secs + dt_, reps + 1
        cpu = {"value": flops / secs / 1e12, "unit": UNIT, "cores": n, "kind": "oracle",
               "sample": "fp64 oracle chunk form: one whole output frame (frame %d, %dx%d) of %s from its "
                         "2-frame history, %d times (%.1f s)" % (wl.T // 2, wl.out_hw[0], wl.out_hw[1], wl.name, reps, secs)}

    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    out = {
        "metric": METRIC, "value": m["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded counter-based generator, on device)",
        "config": workload_config(wl),
        "output_frames_per_s": m["output_frames_per_s"],
        "pct_of_dense_bf16_peak": m["pct_of_dense_bf16_peak"],
        "roofline": m["roofline"],
        "cpu_baseline": cpu,
        "e2e": {"value": wl.flops * world * args.steps / (e2e_ms / 1e3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_step_ms,
                "copy_bound_ms": cb["both_ms"], "frac_of_copy_bound": cb["both_ms"] / e2e_step_ms,
                "copy_bound": dict(cb, how="the step's H2D bytes (x, residual) and D2H bytes (y) as whole-tensor "
                                           "pinned cudaMemcpyAsync calls, the two directions on two streams at "
                                           "once; best of 3")},
        "gpu_launches": m["gpu_launches"],
        "clocks": m["clocks"],
        "step_ms": m["step_ms"],
        "hbm": m["hbm"],
        "configs": configs,
    }
    print(json.dumps(out), flush=True)
    return 0


def run_single_chunk(args, wl):
    """Profiling case: `n` launches of one 4-frame chunk of the workload (no JSON line)."""
    import torch

    import __graft_entry__
    import chunked_causal_convolution_gb300 as cc3d
    import synth
    from synth import native

    __graft_entry__.build()
    dt = torch.bfloat16
    T = min(4, wl.T)
    x = native.fill_device(torch.empty((T, wl.H, wl.W, wl.Cin), dtype=dt, device="cuda"), wl.seed, synth.TID_X,
                           wl.x)
    w = native.fill_device(torch.empty((wl.Cout, wl.kt, wl.kh, wl.kw, wl.Cin), dtype=dt, device="cuda"), wl.seed,
                           synth.TID_W, wl.w)
    b = native.fill_device(torch.empty((wl.Cout,), dtype=dt, device="cuda"), wl.seed, synth.TID_B, wl.b)
    Ho, Wo = wl.out_hw
    r = None
    if wl.r is not None:
        r = native.fill_device(torch.empty((T, Ho, Wo, wl.Cout), dtype=dt, device="cuda"), wl.seed,
                               synth.TID_R, wl.r)
    if wl.up2:
        plan = cc3d.Upsample2xConvPlan(wl.Cin, wl.Cout, wl.H, wl.W, wl.kt)
    else:
        plan = cc3d.CausalConv3dPlan(wl.Cin, wl.Cout, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    cin, cout = plan.new_cache(), plan.new_cache()
    y = torch.empty((T, Ho, Wo, wl.Cout), dtype=dt, device="cuda")
    for _ in range(args.single_chunk):
        plan.forward_chunk(x, w, b, r, cin, cout, y)
    st = plan.status()
    if st != 0:
        raise RuntimeError("device status %s" % cc3d.cc3d_status_string(st))
    log("ran %d launches of one %d-frame chunk of %s" % (args.single_chunk, T, wl.name))
    return 0


def run_output_pipeline(args, wl):
    """Auxiliary measurement (one JSON line, not the bench line): a chunk loop of the narrow head
    with 8-bit frames out, as compute only, with synchronous output (D2H, then the write, then the
    next chunk) and with the asynchronous chunk writer of the C ABI."""
    import torch

    import __graft_entry__
    import chunked_causal_convolution_gb300 as cc3d
    import synth
    from synth import native

    __graft_entry__.build()
    n, Tc, H, W, dt = args.output_chunks, 4, wl.H, wl.W, torch.bfloat16
    x = native.fill_device(torch.empty((Tc, H, W, wl.Cin), dtype=dt, device="cuda"), wl.seed, synth.TID_X, wl.x)
    w = native.fill_device(torch.empty((wl.Cout, wl.kt, wl.kh, wl.kw, wl.Cin), dtype=dt, device="cuda"), wl.seed,
                           synth.TID_W, wl.w)
    b = native.fill_device(torch.empty((wl.Cout,), dtype=dt, device="cuda"), wl.seed, synth.TID_B, wl.b)
    plan = cc3d.CausalConv3dPlan(wl.Cin, wl.Cout, H, W, wl.kt, wl.kh, wl.kw)
    caches = [plan.new_cache(), plan.new_cache()]
    ybuf = [torch.empty((Tc, H, W, wl.Cout), dtype=torch.uint8, device="cuda") for _ in range(2)]
    nbytes = ybuf[0].numel()
    s = torch.cuda.Stream()

    def chunk(k, buf):
        # the same 4-frame input every chunk: the histories still ping-pong as in a stream
        plan.forward_chunk_u8(x, w, b, None, caches[k % 2], caches[(k + 1) % 2], ybuf[buf], stream=s)

    with torch.cuda.stream(s):
        for k in range(3):
            chunk(k, 0)
    s.synchronize()
    out = {"measurement": "chunk output path", "workload": wl.name, "chunk_frames": Tc, "chunks": n,
           "bytes_per_chunk": nbytes, "path": args.output_path}
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        for k in range(n):
            chunk(k, k % 2)
    s.synchronize()
    out["compute_only_ms_per_chunk"] = (time.perf_counter() - t0) * 1e3 / n
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    with open(args.output_path, "wb") as f:
        t0 = time.perf_counter()
        with torch.cuda.stream(s):
            for k in range(n):
                chunk(k, 0)
                host.copy_(ybuf[0].view(-1), non_blocking=True)
                s.synchronize()
                f.write(host.numpy().tobytes())
    out["synchronous_ms_per_chunk"] = (time.perf_counter() - t0) * 1e3 / n
    writer = cc3d.FrameWriter(args.output_path, nbytes)
    seqs = [-1, -1]
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        for k in range(n):
            buf = k % 2
            writer.wait_copied(seqs[buf], s)
            chunk(k, buf)
            seqs[buf] = writer.submit(ybuf[buf], stream=s)
    out["bytes_written"] = writer.close()
    s.synchronize()
    out["asynchronous_ms_per_chunk"] = (time.perf_counter() - t0) * 1e3 / n
    out["status"] = plan.status(s)
    print(json.dumps(out), flush=True)
    return 0 if out["status"] == 0 else 1


def run_graph_timing(args, wl):
    """Auxiliary measurement (one JSON line, not the bench line): the bench step (the workload's
    chunk loop) launched eagerly and replayed from one captured CUDA graph."""
    import torch

    import __graft_entry__
    import chunked_causal_convolution_gb300 as cc3d
    import synth
    from synth import native

    __graft_entry__.build()
    dt = torch.bfloat16
    x = native.fill_device(torch.empty((wl.T, wl.H, wl.W, wl.Cin), dtype=dt, device="cuda"), wl.seed, synth.TID_X,
                           wl.x)
    w = native.fill_device(torch.empty((wl.Cout, wl.kt, wl.kh, wl.kw, wl.Cin), dtype=dt, device="cuda"), wl.seed,
                           synth.TID_W, wl.w)
    b = native.fill_device(torch.empty((wl.Cout,), dtype=dt, device="cuda"), wl.seed, synth.TID_B, wl.b)
    r = (native.fill_device(torch.empty((wl.T, wl.H, wl.W, wl.Cout), dtype=dt, device="cuda"), wl.seed,
                            synth.TID_R, wl.r) if wl.r is not None else None)
    y = torch.empty((wl.T, wl.H, wl.W, wl.Cout), dtype=dt, device="cuda")
    plan = cc3d.CausalConv3dPlan(wl.Cin, wl.Cout, wl.H, wl.W, wl.kt, wl.kh, wl.kw)
    caches = [plan.new_cache(), plan.new_cache()]
    s = torch.cuda.Stream()
    bounds, t = [], 0
    for c in wl.chunks:
        bounds.append((t, c))
        t += c

    def step():
        for k, (s0, c) in enumerate(bounds):
            cc3d.cc3d_forward_chunk(plan.handle, c, x[s0:s0 + c], w, b, r[s0:s0 + c] if r is not None else None,
                                    caches[k % 2] if k else None, caches[(k + 1) % 2], y[s0:s0 + c], s)

    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            step()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    out = {"measurement": "eager vs graph replay", "workload": wl.name, "steps": args.steps}
    for mode in ("eager", "graph", "eager", "graph"):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(args.steps):
                if mode == "eager":
                    step()
                else:
                    g.replay()
            e1.record(s)
        s.synchronize()
        out.setdefault(mode + "_ms_per_step", []).append(e0.elapsed_time(e1) / args.steps)
    out["status"] = plan.status(s)
    print(json.dumps(out), flush=True)
    return 0 if out["status"] == 0 else 1


def run_layer_group(args, wl):
    """Auxiliary measurement (one JSON line, not the bench line): the decoder's last three layers at
    the c96 stage (two 96 -> 96 3x3x3 convs and the 96 -> 3 head, 360 x 640) over one 24-frame
    chunk (the pages' chunk length) per step, run as a frame-batched layer group with batches of
    1, 2 and 4 frames and as the whole chunk at once: time per chunk and the device memory the
    step holds (inputs, outputs, histories and workspace; the peak of the caching allocator)."""
    import torch

    import __graft_entry__
    import chunked_causal_convolution_gb300 as cc3d
    import synth
    from synth import native

    __graft_entry__.build()
    dt, T, H, W = torch.bfloat16, 24, 360, 640
    base = synth.WORKLOADS["c96_residual"]
    spec = [(96, 96), (96, 96), (96, 3)]
    out = {"measurement": "frame-batched layer group", "layers": "96->96 3x3x3, 96->96 3x3x3, 96->3 3x3x3 at "
           "360x640, bias", "chunk_frames": T, "steps": args.steps, "runs": {}}
    for fb in (0, 1, 2, 4):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats()
        before = torch.cuda.memory_allocated()
        plans = [cc3d.CausalConv3dPlan(ci, co, H, W) for ci, co in spec]
        ws_ = [native.fill_device(torch.empty((co, 3, 3, 3, ci), dtype=dt, device="cuda"), base.seed + j,
                                  synth.TID_W, synth.Dist.normal(synth.fan_in_sigma(ci))) for j, (ci, co) in enumerate(spec)]
        bs_ = [native.fill_device(torch.empty((co,), dtype=dt, device="cuda"), base.seed + j, synth.TID_B,
                                  base.b) for j, (ci, co) in enumerate(spec)]
        x = native.fill_device(torch.empty((T, H, W, 96), dtype=dt, device="cuda"), base.seed, synth.TID_X, base.x)
        y = torch.empty((T, H, W, 3), dtype=dt, device="cuda")
        caches = [[p.new_cache(), p.new_cache()] for p in plans]
        group = cc3d.LayerGroup(plans, fb)
        ws = group.new_workspace(T)
        s = torch.cuda.Stream()

        def step(k):
            group.forward_chunk(x, ws_, bs_, [c[k % 2] for c in caches] if k else None,
                                [c[(k + 1) % 2] for c in caches], y, ws, stream=s)

        with torch.cuda.stream(s):
            for k in range(args.warmup):
                step(k)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for k in range(args.steps):
                step(k + 1)
            e1.record(s)
        s.synchronize()
        st = [p.status(s) for p in plans]
        out["runs"]["whole_chunk" if fb == 0 else "batch_%d" % fb] = {
            "ms_per_chunk": e0.elapsed_time(e1) / args.steps, "workspace_bytes": group.workspace_bytes(T),
            "peak_bytes": torch.cuda.max_memory_allocated() - before, "status": st}
        group.close()
        for p in plans:
            p.close()
        del x, y, caches, ws, ws_, bs_
    print(json.dumps(out), flush=True)
    return 0


def run_upsample_compare(args, wl):
    """Auxiliary measurement (one JSON line, not the bench line): the chunk loop of an upsampling
    layer with the nearest-2x upsample fused into the conv, against the unfused pipeline that
    writes each chunk's upsampled frames to memory (a torch broadcast copy) and runs the plain
    conv plan on them.  The outputs of the two must be bit-identical."""
    import torch

    import __graft_entry__
    import chunked_causal_convolution_gb300 as cc3d
    import synth
    from synth import native

    if not wl.up2:
        raise SystemExit("--upsample-compare wants an upsampling workload")
    __graft_entry__.build()
    dt = torch.bfloat16
    Ho, Wo = wl.out_hw
    x = native.fill_device(torch.empty((wl.T, wl.H, wl.W, wl.Cin), dtype=dt, device="cuda"), wl.seed, synth.TID_X,
                           wl.x)
    w = native.fill_device(torch.empty((wl.Cout, wl.kt, wl.kh, wl.kw, wl.Cin), dtype=dt, device="cuda"), wl.seed,
                           synth.TID_W, wl.w)
    b = native.fill_device(torch.empty((wl.Cout,), dtype=dt, device="cuda"), wl.seed, synth.TID_B, wl.b)
    fused = cc3d.Upsample2xConvPlan(wl.Cin, wl.Cout, wl.H, wl.W, wl.kt)
    plain = cc3d.CausalConv3dPlan(wl.Cin, wl.Cout, Ho, Wo, wl.kt, 3, 3)
    fc = [fused.new_cache(), fused.new_cache()]
    pc = [plain.new_cache(), plain.new_cache()]
    cmax = max(wl.chunks)
    xu = torch.empty((cmax, Ho, Wo, wl.Cin), dtype=dt, device="cuda")
    y_fused = torch.empty((wl.T, Ho, Wo, wl.Cout), dtype=dt, device="cuda")
    y_plain = torch.empty_like(y_fused)
    s = torch.cuda.Stream()
    bounds, t = [], 0
    for c in wl.chunks:
        bounds.append((t, c))
        t += c

    def step_fused():
        for k, (s0, c) in enumerate(bounds):
            cc3d.cc3d_forward_chunk(fused.handle, c, x[s0:s0 + c], w, b, None, fc[k % 2] if k else None,
                                    fc[(k + 1) % 2], y_fused[s0:s0 + c], s)

    def step_plain():
        for k, (s0, c) in enumerate(bounds):
            # one broadcast copy: every source position written to its 2 x 2 output block
            xu[:c].view(c, wl.H, 2, wl.W, 2, wl.Cin).copy_(
                x[s0:s0 + c, :, None, :, None, :].expand(c, wl.H, 2, wl.W, 2, wl.Cin))
            cc3d.cc3d_forward_chunk(plain.handle, c, xu[:c], w, b, None, pc[k % 2] if k else None,
                                    pc[(k + 1) % 2], y_plain[s0:s0 + c], s)

    out = {"measurement": "fused nearest-2x upsample vs upsample written to memory + plain conv",
           "workload": wl.name, "steps": args.steps, "fused_kernel": fused.kernel, "plain_kernel": plain.kernel,
           "flop_per_step": wl.flops}
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            step_fused()
            step_plain()
    s.synchronize()
    for mode, fn in (("fused", step_fused), ("unfused", step_plain), ("fused", step_fused), ("unfused", step_plain)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(args.steps):
                fn()
            e1.record(s)
        s.synchronize()
        out.setdefault(mode + "_ms_per_step", []).append(e0.elapsed_time(e1) / args.steps)
    out["fused_tflops"] = wl.flops / (min(out["fused_ms_per_step"]) / 1e3) / 1e12
    out["unfused_tflops"] = wl.flops / (min(out["unfused_ms_per_step"]) / 1e3) / 1e12
    out["status"] = [fused.status(s), plain.status(s)]
    out["bit_identical"] = bool(torch.equal(y_fused, y_plain))
    print(json.dumps(out), flush=True)
    return 0 if out["status"] == [0, 0] and out["bit_identical"] else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c96_residual")
    ap.add_argument("--ref-rows", type=int, default=90, help="rows of the oracle sample frame")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the headline workload (not the other decoder stages and the SR stream)")
    ap.add_argument("--sr-passes", type=int, default=2, help="timed passes over the 361-frame SR stream")
    ap.add_argument("--single-chunk", type=int, default=0,
                    help="profiling case: run this many launches of one 4-frame chunk and exit")
    ap.add_argument("--output-path", default=None,
                    help="auxiliary: time the chunk output path of a narrow head writing 8-bit frames here")
    ap.add_argument("--output-chunks", type=int, default=16)
    ap.add_argument("--graph-timing", action="store_true",
                    help="auxiliary: time the step eagerly and replayed from a CUDA graph")
    ap.add_argument("--layer-group", action="store_true",
                    help="auxiliary: time a frame-batched layer group of the decoder's last layers")
    ap.add_argument("--upsample-compare", action="store_true",
                    help="auxiliary: time an upsampling workload fused and with the upsample written to memory")
    args = ap.parse_args()
    if args.warmup < 3:
        log("warm-up raised to 3 steps")
        args.warmup = 3
    import synth
    wl = synth.WORKLOADS[args.workload]
    if args.single_chunk:
        return run_single_chunk(args, wl)  # one 4-frame chunk: fits for every workload
    if args.output_path:
        return run_output_pipeline(args, wl)  # one 4-frame input chunk
    if args.layer_group:
        return run_layer_group(args, wl)
    if wl.T * wl.H * wl.W * max(wl.Cin, wl.Cout) * 2 > 32e9:
        log("%s does not fit resident on one device; it is covered by the streaming parity test" % wl.name)
        return 2
    if args.graph_timing:
        return run_graph_timing(args, wl)
    if args.upsample_compare:
        return run_upsample_compare(args, wl)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
