#!/usr/bin/env python3
"""Benchmark of the direct-stencil convolution library on one GB300.

A step is one pass of the whole path over one batch of each benchmark
configuration: the six convolutions of the five workloads (depthwise 3x3
fp32 NCHW; the MobileNetV2-style bf16 channels-last depthwise layer at stride
1 and at stride 2; the 7x7 bf16 channels-last depthwise layer; the
multiplier-4 4x4 fp16 NCHW layer; the grouped 4->8 9x9 stride-2 bf16
channels-last layer), each bound once, launched through the C ABI and written
into its preallocated output.

Metric: achieved HBM GB/s with algorithmic bytes = x + w + bias + y, each
moved once, summed over the step's convolutions, plus output pixels per
second (Gpix/s = N*OH*OW / s).  Timing: warm-up steps, then exactly K steps
replayed from CUDA graphs of back-to-back launches, bracketed by a barrier and
a device synchronise, timed with CUDA events on the launching stream; max
over ranks.  L2: every step reads and writes one of several input/output sets
whose total exceeds 3x the L2 size, so no step finds its data in L2.  The
MobileNetV2 pair alone is reported as a sub-entry (``mbv2_step``), every
workload alone under ``per_config`` (with the fp64 oracle timed on the host
cores on the same workload), and the roofline of the kernel that takes the
largest share of the step.

``--impl reference`` times the CPU fp64 oracle (the only reference this
method has) on a bounded sample of the same step instead.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The six convolutions of the five benchmark workloads: one step.
STEP_WORKLOADS = ("dw3x3_f32_nchw", "mbv2_dw3x3_s1_bf16_cl", "mbv2_dw3x3_s2_bf16_cl",
                  "dw7x7_bf16_cl", "dw4x4_m4_f16_nchw", "grp4x8_9x9_s2_bf16_cl")
# The MobileNetV2 layer at both strides, reported as its own sub-step.
MBV2_STEP = ("mbv2_dw3x3_s1_bf16_cl", "mbv2_dw3x3_s2_bf16_cl")
STEP_NAME = ("dw3x3 f32 NCHW 1x32x56x56 + MobileNetV2 dw3x3 bf16 CL 32x144x56x56 s1 + s2 + "
             "dw7x7 bf16 CL 128x96x56x56 + dw4x4 m4 f16 NCHW 16x64x112x112 pad 1/2 + "
             "grouped 4->8 9x9 s2 bf16 CL 8x256x128x128")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
# FP32 FMA lanes: 152 SMs x 128 lanes x 2070 MHz (max SM clock).
SMS, FMA_LANES, MAX_MHZ = 152, 128, 2070.0
DERIVED_FMA_PEAK = SMS * FMA_LANES * MAX_MHZ * 1e6


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload breakdown")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--case", default=None,
                    help="profiling helper: run this workload --reps times and exit (no timing)")
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--schedule", default=None, help="force a schedule for --case")
    return ap.parse_args()


def run_case(args):
    """Run one workload a few times through the C ABI, for ncu captures.
    ``<workload>.backward_input`` / ``.backward_weight`` run that backward
    pass instead."""
    import torch
    import grouped_convolution_gb300 as gc
    from grouped_convolution_gb300.inputs import WORKLOADS, make_inputs
    gc.build()
    if ".backward_" in args.case:
        base, part = args.case.split(".backward_")
        c = BackwardCase(base, 1, "cuda", part)
        for i in range(args.reps):
            c.run(i)
        torch.cuda.synchronize()
        print(json.dumps({"case": args.case, "reps": args.reps}))
        return
    wl = WORKLOADS[args.case]
    x, w, b = make_inputs(wl, device="cuda")
    d = gc.bind(x, w, b, wl.stride, wl.pad_before, wl.pad_after, wl.dilation, wl.groups,
                wl.transposed, wl.output_padding)
    if args.schedule:
        d.schedule = gc.SCHEDULES[args.schedule]
    y = gc.empty_output(d, x)
    for _ in range(args.reps):
        gc.run(d, x, w, b, y)
    torch.cuda.synchronize()
    print(json.dumps({"case": args.case, "reps": args.reps, "shape": list(y.shape),
                      "schedule": gc.conv_select_schedule(d, x, w, b, y)}))


# ------------------------------------------------------------------ helpers

def dist_setup(n_gpus):
    import torch
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def algorithmic(desc, elem):
    """Bytes (x + w + bias + y, each once), FMAs and output pixels of one conv.
    A transposed convolution's FMAs are its input's scatter: every input
    element meets Cout_g * KH * KW weights (before the crop)."""
    x = desc.N * desc.C_in * desc.H * desc.W
    w = desc.C_out * desc.Cin_g * desc.KH * desc.KW
    b = desc.C_out if desc.has_bias else 0
    y = desc.N * desc.C_out * desc.OH * desc.OW
    if desc.transposed:
        fma = x * desc.Cout_g * desc.KH * desc.KW
    else:
        fma = y * desc.Cin_g * desc.KH * desc.KW
    return (x + w + b + y) * elem, fma, desc.N * desc.OH * desc.OW


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while it runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# Source files that define each schedule's kernel; the recorded DRAM traffic
# of a kernel is void once any of them changes.
KERNEL_SOURCES = {
    "dw_row8": ["k_row8.cuh", "k_row8.cu", "stencil_math.cuh", "device_common.cuh", "tma.cuh",
                "launch.cuh"],
    "dw_flat": ["k_flat.cu", "device_common.cuh", "launch.cuh"],
    "dw_small": ["k_small.cu", "device_common.cuh", "launch.cuh"],
    "dw_tc": ["k_dwtc.cu", "tc_common.cuh", "device_common.cuh", "tma.cuh", "tma.cu", "launch.cuh"],
    "dw_tcl": ["k_dwtcl.cu", "tc_common.cuh", "device_common.cuh", "tma.cuh", "tma.cu", "launch.cuh"],
    "dw_mult": ["k_mult.cuh", "k_mult.cu", "device_common.cuh", "tma.cuh", "launch.cuh"],
    "grp_plane": ["k_grp.cuh", "k_grp_impl.cuh", "k_grp.cu", "device_common.cuh", "launch.cuh"],
    "grp_reduce": ["k_reduce.cu", "device_common.cuh", "launch.cuh"],
    "grp_tc": ["k_tc.cu", "k_tcs.cu", "tc_common.cuh", "device_common.cuh", "tma.cuh", "tma.cu", "launch.cuh"],
    "dw_line": ["k_line.cu", "stencil_math.cuh", "device_common.cuh", "launch.cuh"],
}


def kernel_source_sha(schedule):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES.get(schedule, []):
        path = os.path.join(ROOT, "grouped_convolution_gb300", "csrc", name)
        try:
            with open(path, "rb") as f:
                h.update(f.read())
        except OSError:
            return None
    return h.hexdigest()[:16]


def recorded_traffic(schedule, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source has not changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get(f"{workload}@{schedule}") or table.get(workload)
    if not ent or ent.get("schedule") != schedule or \
            ent.get("source_sha") != kernel_source_sha(schedule):
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------- our GPU path

class ConvCase:
    """One workload bound once, with R rotating input/output sets."""

    def __init__(self, name, sets, device, schedule=None):
        import torch
        import grouped_convolution_gb300 as gc
        from grouped_convolution_gb300.inputs import WORKLOADS, make_inputs
        self.gc = gc
        self.wl = WORKLOADS[name]
        x, w, b = make_inputs(self.wl)
        self.x_host = x
        self.w = w.to(device)
        self.b = b.to(device) if b is not None else None
        wl = self.wl
        self.desc = gc.bind(x, w, b, wl.stride, wl.pad_before, wl.pad_after, wl.dilation,
                            wl.groups, wl.transposed, wl.output_padding)
        if schedule is not None:
            self.desc.schedule = gc.SCHEDULES[schedule]
        xd = x.to(device)
        self.xs = [xd] + [xd.clone() for _ in range(sets - 1)]
        self.ys = [gc.empty_output(self.desc, xd) for _ in range(sets)]
        self.elem = x.element_size()
        self.bytes, self.fma, self.pix = algorithmic(self.desc, self.elem)
        self.schedule = gc.conv_select_schedule(self.desc, self.xs[0], self.w, self.b, self.ys[0])

    def footprint(self):
        return sum(t.numel() * t.element_size() for t in self.xs + self.ys)

    def run(self, i, stream=None):
        k = i % len(self.xs)
        self.gc.run(self.desc, self.xs[k], self.w, self.b, self.ys[k], stream)


class BackwardCase:
    """The backward of one forward workload: ``part`` "input" (dx from gy and
    w) or "weight" (dw and db from x and gy, with the fp32 workspace), bound
    once, with R rotating sets of its streamed tensors."""

    def __init__(self, name, sets, device, part):
        import torch
        import grouped_convolution_gb300 as gc
        from grouped_convolution_gb300.inputs import WORKLOADS, make_grad, make_inputs
        self.gc = gc
        self.part = part
        self.wl = wl = WORKLOADS[name]
        x, w, _ = make_inputs(wl)
        self.desc = d = gc.conv_bind(x, w, None, wl.stride, wl.pad_before, wl.pad_after,
                                     wl.dilation, wl.groups)
        ysz, _ = gc.out_shape_and_stride(d)
        gy = make_grad(wl, ysz)
        self.w = w.to(device)
        elem = x.element_size()
        n_x, n_y, n_w = x.numel(), gy.numel(), w.numel()
        self.pix = d.N * d.OH * d.OW
        taps = d.Cin_g * d.KH * d.KW
        self.fma = n_y * taps
        xd, gyd = x.to(device), gy.to(device)
        if part == "input":
            sizes, strides = gc.grad_input_shape_and_stride(d)
            self.gys = [gyd] + [gyd.clone() for _ in range(sets - 1)]
            self.dxs = [torch.empty_strided(sizes, strides, dtype=x.dtype, device=device)
                        for _ in range(sets)]
            self.bytes = (n_y + n_w + n_x) * elem
            self.streamed = self.gys + self.dxs
        else:
            self.xs = [xd] + [xd.clone() for _ in range(sets - 1)]
            self.gys = [gyd] + [gyd.clone() for _ in range(sets - 1)]
            self.dw = torch.empty(tuple(w.shape), dtype=x.dtype, device=device)
            self.db = torch.empty(d.C_out, dtype=x.dtype, device=device)
            self.ws_bytes = gc.conv_backward_weight_workspace_size(d)
            self.ws = torch.empty((self.ws_bytes + 15) // 16 * 4, dtype=torch.float32,
                                  device=device)
            self.bytes = (n_x + n_y + n_w + d.C_out) * elem
            self.streamed = self.xs + self.gys
        self.elem = elem
        self.schedule = f"backward_{part}"

    def footprint(self):
        return sum(t.numel() * t.element_size() for t in self.streamed)

    def run(self, i, stream=None):
        k = i % len(self.gys)
        if self.part == "input":
            self.gc.conv_backward_input(self.desc, self.gys[k], self.w, self.dxs[k], stream)
        else:
            self.gc.conv_backward_weight(self.desc, self.xs[k], self.gys[k], self.dw, self.db,
                                         self.ws, self.ws_bytes, stream)


def sets_needed(bytes_per_set, l2_bytes):
    return max(2, math.ceil(3 * l2_bytes / max(bytes_per_set, 1)) + 1)


def time_graph(cases, steps, warmup, world, chunk=200):
    """Time exactly `steps` steps (each runs every case once) replayed from
    CUDA graphs.  Returns total milliseconds (max over ranks) and the number
    of kernel launches inside the timed region."""
    import torch
    gc = cases[0].gc
    stream = torch.cuda.Stream()
    chunk = max(1, min(chunk, steps))

    def capture(n, offset):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    for c in cases:
                        c.run(offset + i, stream)
        return g

    torch.cuda.synchronize()
    g_full = capture(chunk, 0)
    rem = steps % chunk
    g_rem = capture(rem, 0) if rem else None
    # warm-up: eager launches, then whole graphs
    with torch.cuda.stream(stream):
        for i in range(warmup):
            for c in cases:
                c.run(i, stream)
    g_full.replay()
    torch.cuda.synchronize()
    launches_before = gc.conv_launch_count()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps // chunk):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(end)
    # Graph replays do not pass through the library; count the kernels they hold.
    per_step = sum(1 for _ in cases)
    launches = steps * per_step
    assert gc.conv_launch_count() == launches_before
    return max_over_ranks(ms, world), launches


def time_e2e(cases, steps, world, lanes=3):
    """Same metric through the public API with host buffers: every step copies
    each distinct input from pinned host memory, runs the convolutions and
    reads every result back to pinned host memory.  Steps rotate over `lanes`
    streams, each with its own device and pinned output buffers, so step i's
    input copies overlap step i-1's kernels and step i-2's read-backs (the
    copy engines and the SMs work at once, as a streaming user would run
    them).  Convolutions of one workload id (the MobileNetV2 layer at both
    strides) read the same input, copied once."""
    import torch
    gc = cases[0].gc
    streams = [torch.cuda.Stream() for _ in range(lanes)]
    host_x, slot = [], []
    for c in cases:
        for k, (wid, _) in enumerate(host_x):
            if wid == c.wl.wid:
                slot.append(k)
                break
        else:
            slot.append(len(host_x))
            host_x.append((c.wl.wid, c.x_host.pin_memory()))
    host_x = [h for _, h in host_x]
    dev_x = [[cases[slot.index(k)].xs[0] if lane == 0 else cases[slot.index(k)].xs[0].clone()
              for k in range(len(host_x))] for lane in range(lanes)]
    dev_y = [[gc.empty_output(c.desc, c.xs[0]) for c in cases] for _ in range(lanes)]
    # Pinned host outputs with the device outputs' own strides (channels-last
    # stays channels-last), so each read-back is one plain copy.
    outs = [[torch.empty_strided(c.ys[0].shape, c.ys[0].stride(), dtype=c.ys[0].dtype,
                                 pin_memory=True) for c in cases]
            for _ in range(lanes)]
    h2d = sum(h.numel() * h.element_size() for h in host_x)
    d2h = sum(o.numel() * o.element_size() for o in outs[0])
    main = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def step(i):
        k = i % lanes
        with torch.cuda.stream(streams[k]):
            for dx, hx in zip(dev_x[k], host_x):
                dx.copy_(hx, non_blocking=True)
            for c, s_, y, o in zip(cases, slot, dev_y[k], outs[k]):
                c.gc.run(c.desc, dev_x[k][s_], c.w, c.b, y, streams[k])
                o.copy_(y, non_blocking=True)

    for i in range(2 * lanes):  # warm-up
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    start.record(main)
    for st in streams:
        st.wait_event(start)
    for i in range(steps):
        step(i)
    for st in streams:
        main.wait_stream(st)
    end.record(main)
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(start.elapsed_time(end), world), h2d, d2h


def measure_fma_peak(dev, reps=5):
    """The chip's fp32 FMA rate, measured: the library's probe kernel (every
    SM full of independent FMA chains) timed with CUDA events, best of
    `reps` launches after one warm-up.  FMAs per second."""
    import torch
    import grouped_convolution_gb300 as gc
    sink = torch.zeros(152 * 64, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    gc.conv_probe_fma_rate(64, sink, stream)
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = gc.conv_probe_fma_rate(4096, sink, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        rate = n / (e0.elapsed_time(e1) * 1e-3)
        best = rate if best is None else max(best, rate)
    return best


# Schedules whose multiply-adds run on the tensor cores: the FP32 FMA pipe is
# not their bound.
TENSOR_CORE_SCHEDULES = ("grp_tc", "dw_tc", "dw_tcl")


def roofline_of(c, us, hbm_peak, fma_peak):
    """Roofline of one kernel: the bound is the resource whose peak time is
    the larger (HBM for the algorithmic bytes, the FP32 FMA pipe for the
    algorithmic FMAs); a tensor-core schedule is held to HBM and the bf16
    tensor peak is not its limit at these shapes."""
    t = us * 1e-6
    t_hbm = c.bytes / (hbm_peak * 1e9)
    t_fma = c.fma / fma_peak
    if c.schedule in TENSOR_CORE_SCHEDULES or t_hbm >= t_fma:
        ach = c.bytes / t / 1e9
        return {"bound": "hbm", "achieved": round(ach, 2), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(ach / hbm_peak, 4)}
    ach = 2 * c.fma / t / 1e12
    peak = 2 * fma_peak / 1e12
    return {"bound": "alu", "achieved": round(ach, 3), "peak": round(peak, 3),
            "unit": "TFLOP/s", "frac": round(ach / peak, 4),
            "note": "fp32 FMA pipe, 2 flops per FMA; peak = the probe's measured FMA rate"}


def run_ours(args):
    import torch
    import grouped_convolution_gb300 as gc
    rank, world = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    gc.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    fma_peak = measure_fma_peak(dev)

    # Step cases share one rotation depth sized from their joint footprint.
    probe = [ConvCase(n, 1, dev) for n in STEP_WORKLOADS]
    per_set = sum(p.footprint() for p in probe)
    R = sets_needed(per_set, l2)
    del probe
    torch.cuda.empty_cache()
    cases = [ConvCase(n, R, dev) for n in STEP_WORKLOADS]

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    total_ms, launches = time_graph(cases, args.steps, args.warmup, world)
    mb_cases = [c for c in cases if c.wl.name in MBV2_STEP]
    mb_ms, _ = time_graph(mb_cases, args.steps, args.warmup, world)
    clocks = sampler.stop()

    step_bytes = sum(c.bytes for c in cases)
    step_pix = sum(c.pix for c in cases)
    ms_per_step = total_ms / args.steps
    value = step_bytes * args.steps * world / (total_ms * 1e-3) / 1e9
    gpix = step_pix * args.steps * world / (total_ms * 1e-3) / 1e9
    mb_bytes = sum(c.bytes for c in mb_cases)
    mb_value = mb_bytes * args.steps * world / (mb_ms * 1e-3) / 1e9

    e2e_steps = max(1, min(args.steps, 30))
    e2e_ms, h2d, d2h = time_e2e(cases, e2e_steps, world)
    e2e_value = step_bytes * e2e_steps * world / (e2e_ms * 1e-3) / 1e9
    del cases, mb_cases
    torch.cuda.empty_cache()

    # Every workload alone (its own rotation depth): the per-kernel times
    # behind the roofline, and the per-config record.
    configs = per_config(args, world, l2, hbm_peak, fma_peak, dev)
    share = {n: configs[n]["us"] for n in STEP_WORKLOADS}
    dom_name = max(share, key=share.get)
    dom = configs[dom_name]
    roof = dict(dom["roofline"])
    roof.update({"kernel": f"{dom['schedule']} ({dom_name})", "peak_kind": peak_kind,
                 "traffic": recorded_traffic(dom["schedule"], dom_name),
                 "algorithmic_bytes": dom["bytes"], "algorithmic_fma": dom["fma"],
                 "launch_us": dom["us"],
                 "share_of_kernel_time": round(share[dom_name] / sum(share.values()), 4)})
    if roof["bound"] == "alu":
        roof["peak_kind"] = "measured (FMA probe)"
    result = {
        "metric": "direct-stencil conv HBM GB/s (algorithmic bytes x+w+b+y once) and Gpix/s",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32/bf16/f16 in/out (per workload), fp32 accumulate",
        "data": "synthetic (seeded)",
        "config": {"workload": STEP_NAME,
                   "convs_per_step": list(STEP_WORKLOADS),
                   "schedules": {n: configs[n]["schedule"] for n in STEP_WORKLOADS},
                   "l2": f"{R} rotating input/output sets, {R * per_set / 2**20:.0f} MiB "
                         f"> 3x L2 ({l2 / 2**20:.0f} MiB)",
                   "parallelism": f"replicas x{world}"},
        "gpix_per_s": round(gpix, 3),
        "frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "frac_of_measured_hbm": round(value / world / hbm_peak, 4),
        "mbv2_step": {"convs": list(MBV2_STEP), "GB_s": round(mb_value, 2),
                      "us_per_step": round(mb_ms / args.steps * 1e3, 3),
                      "frac_of_measured_hbm": round(mb_value / world / hbm_peak, 4)},
        "fma_peak": {"measured_tfma_s": round(fma_peak / 1e12, 3),
                     "derived_tfma_s": round(DERIVED_FMA_PEAK / 1e12, 3),
                     "derived_from": "152 SMs x 128 FP32 lanes x 2070 MHz"},
        "per_kernel_us": share,
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if not args.no_configs:
        result["per_config"] = configs
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        base = cpu_baseline(configs, budget_s=2.5)
        result["cpu_baseline"] = base
        if not args.no_configs:
            for n, b in base.pop("per_config").items():
                configs[n]["cpu_baseline"] = b
        else:
            base.pop("per_config")
    if rank == 0:
        line = json.dumps(result)
        print(line, flush=True)
        if args.out:
            with open(args.out, "a") as f:
                f.write(line + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def per_config(args, world, l2, hbm_peak, fma_peak, dev):
    """Every workload alone: GB/s, Gpix/s, HBM fraction, FMA-pipe fraction
    and the kernel's roofline.  With --no-configs only the step's workloads."""
    import torch
    from grouped_convolution_gb300.inputs import WORKLOADS
    out = {}
    steps = max(20, min(args.steps, 2000))

    def measure(name, schedule=None):
        one = ConvCase(name, 1, dev, schedule)
        R = sets_needed(one.footprint(), l2)
        del one
        torch.cuda.empty_cache()
        c = ConvCase(name, R, dev, schedule)
        ms, _ = time_graph([c], steps, max(3, min(args.warmup, 50)), world)
        t = ms / steps * 1e-3
        gbs = c.bytes / t / 1e9
        res = {"schedule": c.schedule, "us": round(t * 1e6, 3),
               "GB_s": round(gbs, 1), "Gpix_s": round(c.pix / t / 1e9, 3),
               "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
               "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
               "TFMA_s": round(c.fma / t / 1e12, 3),
               "frac_of_fma_peak_measured": round(c.fma / t / fma_peak, 4),
               "frac_of_fma_peak_2070mhz": round(c.fma / t / DERIVED_FMA_PEAK, 4),
               "roofline": roofline_of(c, t * 1e6, hbm_peak, fma_peak),
               "bytes": c.bytes, "fma": c.fma, "rotating_sets": R}
        del c
        torch.cuda.empty_cache()
        return res

    def measure_bwd(name, part):
        one = BackwardCase(name, 1, dev, part)
        R = sets_needed(one.footprint(), l2)
        del one
        torch.cuda.empty_cache()
        c = BackwardCase(name, R, dev, part)
        ms, _ = time_graph([c], steps, max(3, min(args.warmup, 50)), world)
        t = ms / steps * 1e-3
        gbs = c.bytes / t / 1e9
        res = {"pass": part, "us": round(t * 1e6, 3), "GB_s": round(gbs, 1),
               "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
               "TFMA_s": round(c.fma / t / 1e12, 3),
               "frac_of_fma_peak_measured": round(c.fma / t / fma_peak, 4),
               "bytes": c.bytes, "fma": c.fma, "launches_per_call": 1 if part == "input" else 2}
        del c
        torch.cuda.empty_cache()
        return res

    names = list(WORKLOADS) if not args.no_configs else list(STEP_WORKLOADS)
    for name in names:
        out[name] = measure(name)
        # A call the picker sends to the tensor cores is also timed on the
        # direct stencil (no tensor cores) that would take it otherwise.
        if out[name]["schedule"] == "grp_tc" and not args.no_configs:
            st = measure(name, "grp_plane")
            out[name]["direct_stencil"] = {k: st[k] for k in (
                "schedule", "us", "GB_s", "frac_of_measured_hbm", "TFMA_s",
                "frac_of_fma_peak_measured", "roofline")}
        # The channels-last 7x7 layer stays on the FMA-pipe stencil (dw_row8);
        # it is also timed on its tensor-core form (dw_tcl).
        if name == "dw7x7_bf16_cl" and not args.no_configs:
            st = measure(name, "dw_tcl")
            out[name]["tensor_cores"] = {k: st[k] for k in (
                "schedule", "us", "GB_s", "frac_of_measured_hbm", "TFMA_s", "roofline")}
    if args.no_configs:
        return out
    # The backward of the MobileNetV2 layers: dx (a transposed convolution of
    # the output gradient) and dw + db (two launches: slice partials, then
    # the fixed-order sum).
    for name in MBV2_STEP:
        for part in ("input", "weight"):
            out[f"{name}.backward_{part}"] = measure_bwd(name, part)
    return out


# ------------------------------------------------------------- CPU oracle

class OracleSample:
    """The fp64 oracle on one workload, restricted to its first n images
    (inputs widened to fp64 outside the timed region)."""

    def __init__(self, name):
        import oracle
        from grouped_convolution_gb300.inputs import WORKLOADS, make_inputs
        self.oracle = oracle
        self.wl = wl = WORKLOADS[name]
        x, w, b = make_inputs(wl)
        self.elem = x.element_size()
        self.x = x.double().contiguous()
        self.w = w.double()
        self.b = b.double() if b is not None else None
        self.n_max = x.shape[0]

    def bytes_for(self, n_img):
        wl, o = self.wl, self.oracle
        oh = o.out_size(wl.H, wl.KH, wl.stride[0], wl.pad_before[0], wl.pad_after[0])
        ow = o.out_size(wl.W, wl.KW, wl.stride[1], wl.pad_before[1], wl.pad_after[1])
        return (n_img * wl.C_in * wl.H * wl.W + wl.C_out * wl.cin_g * wl.KH * wl.KW +
                (wl.C_out if wl.bias else 0) + n_img * wl.C_out * oh * ow) * self.elem

    def one_pass(self, n_img):
        wl = self.wl
        t0 = time.perf_counter()
        self.oracle.conv2d(self.x[:n_img], self.w, self.b, wl.stride, wl.pad_before,
                           wl.pad_after, wl.groups)
        return time.perf_counter() - t0

    def timed(self, budget_s):
        """Whole passes over as many images as fit about `budget_s`: returns
        (GB/s, images, passes, seconds)."""
        t1 = self.one_pass(1)
        n_img = max(1, min(self.n_max, int(budget_s / max(t1, 1e-4))))
        self.one_pass(n_img)                    # untimed first pass at this size
        t, reps = 0.0, 0
        while reps < 1 or (t < budget_s and reps < 200):
            t += self.one_pass(n_img)
            reps += 1
        return self.bytes_for(n_img) * reps / t / 1e9, n_img, reps, t


def cpu_baseline(configs, budget_s=2.5):
    """The oracle on every workload of the step, on the host cores: per
    workload GB/s on a bounded sample, the step aggregate (sum of the samples'
    bytes over the sum of their times, per image of each workload), and the
    first workload once more on one thread."""
    import oracle
    per, tot_b, tot_t = {}, 0.0, 0.0
    cores = oracle.num_threads()
    for name in STEP_WORKLOADS:
        smp = OracleSample(name)
        gbs, n_img, reps, t = smp.timed(budget_s)
        per[name] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                     "sample": f"first {n_img} of {smp.n_max} images, {reps} passes, "
                               f"{t:.2f} s",
                     "gpu_over_oracle": round(configs[name]["GB_s"] / gbs, 1)}
        # whole-step aggregate: each workload's full bytes at its sampled rate
        tot_b += smp.bytes_for(smp.n_max)
        tot_t += smp.bytes_for(smp.n_max) / (gbs * 1e9)
        if name == STEP_WORKLOADS[0]:
            oracle.set_num_threads(1)
            try:
                g1, n1, r1, t1 = smp.timed(budget_s / 2)
            finally:
                oracle.set_num_threads(cores)
            per[name]["single_thread"] = {"value": round(g1, 4), "unit": "GB/s", "cores": 1,
                                          "sample": f"first {n1} images, {r1} passes, "
                                                    f"{t1:.2f} s"}
    return {"value": round(tot_b / tot_t / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"fp64 oracle on each of the step's {len(STEP_WORKLOADS)} convolutions "
                      f"(about {budget_s:.1f} s of whole passes each over its first images), "
                      "combined as the full step's bytes over its time at the sampled rates",
            "per_config": per}


def run_reference(args):
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return
    samples = [OracleSample(n) for n in STEP_WORKLOADS]
    budget = 150.0
    per_step_budget = budget / max(1, args.steps + args.warmup)
    # images per workload: the same fraction of every workload's batch
    full = sum(s.one_pass(1) * s.n_max for s in samples)   # one step at full size, estimated
    frac = min(1.0, per_step_budget / max(full, 1e-6))
    n_img = [max(1, min(s.n_max, int(round(frac * s.n_max)))) for s in samples]
    for _ in range(args.warmup):
        for s, n in zip(samples, n_img):
            s.one_pass(n)
    t = 0.0
    for _ in range(args.steps):
        for s, n in zip(samples, n_img):
            t += s.one_pass(n)
    step_bytes = sum(s.bytes_for(n) for s, n in zip(samples, n_img))
    gbs = step_bytes * args.steps / t / 1e9
    cores = samples[0].oracle.num_threads()
    line = {
        "impl": "reference",
        "metric": "direct-stencil conv HBM GB/s (algorithmic bytes x+w+b+y once) and Gpix/s",
        "value": round(gbs, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": STEP_NAME, "convs_per_step": list(STEP_WORKLOADS),
                   "sample_images_per_step": dict(zip(STEP_WORKLOADS, n_img))},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": "first " + ", ".join(f"{n} of {s.n_max}" for s, n in
                                                        zip(samples, n_img)) +
                                   " images of the step's convolutions per step"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(json.dumps(line) + "\n")


if __name__ == "__main__":
    a = parse()
    if a.case:
        run_case(a)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
