#!/usr/bin/env python3
"""Benchmark of the direct-stencil convolution library on one GB300.

A step is one pass of the whole path over one batch: the MobileNetV2-style
depthwise layer (N=32, C=144, 56x56, bf16 channels-last, 3x3, padding 1/1,
bias) at stride 1 and at stride 2, each bound, launched through the C ABI and
written into its preallocated output.

Metric: achieved HBM GB/s with algorithmic bytes = x + w + bias + y, each
moved once, plus output pixels per second (Gpix/s = N*OH*OW / s).  Timing:
warm-up steps, then exactly K steps replayed from CUDA graphs of back-to-back
launches, bracketed by a barrier and a device synchronise, timed with CUDA
events on the launching stream; max over ranks.  L2: every step reads and
writes one of several input/output sets whose total exceeds 3x the L2 size,
so no step finds its data in L2.

``--impl reference`` times the CPU fp64 oracle (the only reference this
method has) on a bounded sample of the same workload instead.
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

STEP_WORKLOADS = ("mbv2_dw3x3_s1_bf16_cl", "mbv2_dw3x3_s2_bf16_cl")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
# FP32 FMA lanes: 152 SMs x 128 lanes x 2070 MHz (max SM clock).
SMS, FMA_LANES, MAX_MHZ = 152, 128, 2070.0


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
    "dw_mult": ["k_mult.cuh", "k_mult.cu", "device_common.cuh", "tma.cuh", "launch.cuh"],
    "grp_plane": ["k_grp.cuh", "k_grp_impl.cuh", "k_grp.cu", "device_common.cuh", "launch.cuh"],
    "grp_reduce": ["k_reduce.cu", "device_common.cuh", "launch.cuh"],
    "grp_tc": ["k_tc.cu", "device_common.cuh", "tma.cuh", "launch.cuh"],
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
    its input from pinned host memory, runs the convolutions and reads the
    results back to pinned host memory.  Steps rotate over `lanes` streams,
    each with its own device and pinned output buffers, so step i's input
    copy overlaps step i-1's kernels and step i-2's read-back (the copy
    engines and the SMs work at once, as a streaming user would run them)."""
    import torch
    gc = cases[0].gc
    host_x = cases[0].x_host.pin_memory()
    streams = [torch.cuda.Stream() for _ in range(lanes)]
    dev_x = [cases[0].xs[0]] + [cases[0].xs[0].clone() for _ in range(lanes - 1)]
    dev_y = [[gc.empty_output(c.desc, dev_x[0]) for c in cases] for _ in range(lanes)]
    # Pinned host outputs with the device outputs' own strides (channels-last
    # stays channels-last), so each read-back is one plain copy.
    outs = [[torch.empty_strided(c.ys[0].shape, c.ys[0].stride(), dtype=c.ys[0].dtype,
                                 pin_memory=True) for c in cases]
            for _ in range(lanes)]
    h2d = host_x.numel() * host_x.element_size()
    d2h = sum(o.numel() * o.element_size() for o in outs[0])
    main = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def step(i):
        k = i % lanes
        with torch.cuda.stream(streams[k]):
            dev_x[k].copy_(host_x, non_blocking=True)
            for c, y, o in zip(cases, dev_y[k], outs[k]):
                c.gc.run(c.desc, dev_x[k], c.w, c.b, y, streams[k])
                o.copy_(y, non_blocking=True)

    for i in range(3 * lanes):  # warm-up
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
    clocks = sampler.stop()

    # Per-kernel average launch time, each kernel alone over the same protocol.
    per_kernel = {}
    for c in cases:
        ms, _ = time_graph([c], args.steps, args.warmup, world)
        per_kernel[c.wl.name] = ms / args.steps

    step_bytes = sum(c.bytes for c in cases)
    step_pix = sum(c.pix for c in cases)
    ms_per_step = total_ms / args.steps
    value = step_bytes * args.steps * world / (total_ms * 1e-3) / 1e9
    gpix = step_pix * args.steps * world / (total_ms * 1e-3) / 1e9

    dom = cases[0]
    dom_ms = per_kernel[dom.wl.name]
    achieved = dom.bytes / (dom_ms * 1e-3) / 1e9
    traffic = recorded_traffic(dom.schedule, dom.wl.name)

    e2e_steps = max(1, min(args.steps, 50))
    e2e_ms, h2d, d2h = time_e2e(cases, e2e_steps, world)
    e2e_value = step_bytes * e2e_steps * world / (e2e_ms * 1e-3) / 1e9

    result = {
        "metric": "direct-stencil conv HBM GB/s (algorithmic bytes x+w+b+y once) and Gpix/s",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in/out, fp32 accumulate", "data": "synthetic (seeded)",
        "config": {"workload": "MobileNetV2 depthwise 3x3 bf16 channels-last N=32 C=144 "
                               "56x56 pad 1/1 bias, stride 1 + stride 2",
                   "convs_per_step": [c.wl.name for c in cases],
                   "schedules": {c.wl.name: c.schedule for c in cases},
                   "l2": f"{R} rotating input/output sets, {R * per_set / 2**20:.0f} MiB "
                         f"> 3x L2 ({l2 / 2**20:.0f} MiB)",
                   "parallelism": f"replicas x{world}"},
        "gpix_per_s": round(gpix, 3),
        "frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "frac_of_measured_hbm": round(value / world / hbm_peak, 4),
        "per_kernel_us": {k: round(v * 1e3, 3) for k, v in per_kernel.items()},
        "roofline": {"bound": "hbm", "kernel": f"{dom.schedule} ({dom.wl.name})",
                     "achieved": round(achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                     "traffic": traffic, "algorithmic_bytes": dom.bytes},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if not args.no_configs:
        result["per_config"] = per_config(args, world, l2, hbm_peak, dev)
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(budget_s=15.0)
    if rank == 0:
        line = json.dumps(result)
        print(line, flush=True)
        if args.out:
            with open(args.out, "a") as f:
                f.write(line + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def per_config(args, world, l2, hbm_peak, dev):
    """Every workload alone: GB/s, Gpix/s, HBM fraction and FMA-pipe fraction."""
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
        fma_peak = SMS * FMA_LANES * MAX_MHZ * 1e6
        res = {"schedule": c.schedule, "us": round(t * 1e6, 3),
               "GB_s": round(gbs, 1), "Gpix_s": round(c.pix / t / 1e9, 3),
               "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
               "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
               "TFMA_s": round(c.fma / t / 1e12, 3),
               "frac_of_fma_peak_2070mhz": round(c.fma / t / fma_peak, 4),
               "bytes": c.bytes, "fma": c.fma}
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
        fma_peak = SMS * FMA_LANES * MAX_MHZ * 1e6
        res = {"pass": part, "us": round(t * 1e6, 3), "GB_s": round(gbs, 1),
               "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
               "TFMA_s": round(c.fma / t / 1e12, 3),
               "frac_of_fma_peak_2070mhz": round(c.fma / t / fma_peak, 4),
               "bytes": c.bytes, "fma": c.fma, "launches_per_call": 1 if part == "input" else 2}
        del c
        torch.cuda.empty_cache()
        return res

    for name in WORKLOADS:
        out[name] = measure(name)
        # A call the picker sends to the tensor cores is also timed on the
        # direct stencil (no tensor cores) that would take it otherwise.
        if out[name]["schedule"] == "grp_tc":
            st = measure(name, "grp_plane")
            out[name]["direct_stencil"] = {k: st[k] for k in (
                "schedule", "us", "GB_s", "frac_of_measured_hbm", "TFMA_s",
                "frac_of_fma_peak_2070mhz")}
    # The backward of the step's layers: dx (a transposed convolution of the
    # output gradient) and dw + db (two launches: slice partials, then the
    # fixed-order sum).
    for name in STEP_WORKLOADS:
        for part in ("input", "weight"):
            out[f"{name}.backward_{part}"] = measure_bwd(name, part)
    return out


# ------------------------------------------------------------- CPU oracle

def oracle_step_sample(budget_s, max_steps=None):
    """Time the fp64 oracle on the step's workloads, restricted to the first
    n images, with n grown until one pass takes a measurable time."""
    import oracle
    from grouped_convolution_gb300.inputs import WORKLOADS, make_inputs
    wls = [WORKLOADS[n] for n in STEP_WORKLOADS]
    x, w, b = make_inputs(wls[0])
    xs = x.double().contiguous()   # widening, outside the timed region
    ws, bs = w.double(), b.double()
    elem = x.element_size()

    def bytes_for(n_img):
        total = 0
        for wl in wls:
            oh = oracle.out_size(wl.H, wl.KH, wl.stride[0], wl.pad_before[0], wl.pad_after[0])
            ow = oracle.out_size(wl.W, wl.KW, wl.stride[1], wl.pad_before[1], wl.pad_after[1])
            total += (n_img * wl.C_in * wl.H * wl.W + wl.C_out * wl.cin_g * wl.KH * wl.KW +
                      wl.C_out + n_img * wl.C_out * oh * ow) * elem
        return total

    def one_pass(n_img):
        t0 = time.perf_counter()
        for wl in wls:
            oracle.conv2d(xs[:n_img], ws, bs, wl.stride, wl.pad_before, wl.pad_after, wl.groups)
        return time.perf_counter() - t0

    return oracle, wls, one_pass, bytes_for, xs.shape[0]


def cpu_baseline(budget_s=15.0):
    oracle, wls, one_pass, bytes_for, n_max = oracle_step_sample(budget_s)
    n_img = n_max
    t1 = one_pass(n_img)
    reps = max(1, int(budget_s / max(t1, 1e-3)))
    t = 0.0
    for _ in range(reps):
        t += one_pass(n_img)
    gbs = bytes_for(n_img) * reps / t / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle, both convolutions of the step over all {n_img} images, "
                      f"{reps} passes, {t:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return
    oracle, wls, one_pass, bytes_for, n_max = oracle_step_sample(0)
    t1 = one_pass(1)
    budget = 150.0
    per_step_budget = budget / max(1, args.steps + args.warmup)
    n_img = max(1, min(n_max, int(per_step_budget / max(t1, 1e-4))))
    for _ in range(args.warmup):
        one_pass(n_img)
    t = 0.0
    for _ in range(args.steps):
        t += one_pass(n_img)
    gbs = bytes_for(n_img) * args.steps / t / 1e9
    line = {
        "impl": "reference",
        "metric": "direct-stencil conv HBM GB/s (algorithmic bytes x+w+b+y once) and Gpix/s",
        "value": round(gbs, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": "MobileNetV2 depthwise 3x3 bf16 channels-last N=32 C=144 "
                               "56x56 pad 1/1 bias, stride 1 + stride 2",
                   "sample_images_per_step": n_img},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"first {n_img} of {n_max} images per step, both strides"},
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
