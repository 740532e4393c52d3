"""Multi-process paths of bench.py on CPU (gloo, world size 2).

The library itself has no multi-GPU path (replicas only); what runs on more
than one rank is bench.py's launcher logic: process-group setup, barriers,
max-over-ranks timing, and the reference arm's rank-0-only output under
torchrun.  These run here with the gloo backend on 127.0.0.1.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w = bench.dist_setup(world)
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    worst = bench.max_over_ranks(1.5 + rank, w)   # each rank reports its own time
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "max": worst}, f)
    dist.destroy_process_group()


def test_rank_helpers_over_gloo(tmp_path):
    """Every rank sees the slowest rank's time (the bench reports the max)."""
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [g["rank"] for g in got] == [0, 1]
    assert all(g["world"] == 2 and g["max"] == 2.5 for g in got)


def test_reference_arm_under_torchrun_prints_once():
    """Under torchrun the reference arm runs on rank 0 only: one JSON line,
    every rank exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_roofline_bound_rule():
    """bench.py's roofline: the resource whose peak time is larger bounds a
    stencil; tensor-core schedules are held to HBM (the FP32 FMA pipe does
    not do their multiply-adds)."""
    import types
    import bench
    hbm, fma = 6773.5, 39.2e12
    # FMA-heavy (the 7x7 layer's bytes and FMAs) on an FMA-pipe stencil: alu
    c = types.SimpleNamespace(bytes=154.15e6, fma=1.888e9, schedule="dw_row8")
    r = bench.roofline_of(c, 107.3, hbm, fma)
    assert r["bound"] == "alu" and 0.44 < r["frac"] < 0.46
    # the same layer on the tensor cores: hbm
    for s in ("dw_tcl", "dw_tc", "grp_tc"):
        c.schedule = s
        r = bench.roofline_of(c, 96.4, hbm, fma)
        assert r["bound"] == "hbm" and r["unit"] == "GB/s"
        assert abs(r["achieved"] - 154.15e6 / 96.4e-6 / 1e9) < 0.01
    # byte-heavy on a stencil: hbm
    c = types.SimpleNamespace(bytes=57.81e6, fma=0.13e9, schedule="dw_row8")
    assert bench.roofline_of(c, 17.4, hbm, fma)["bound"] == "hbm"


def test_per_config_record_layout(monkeypatch):
    """bench.py's per-config record, assembled with the GPU parts faked (the
    case objects and the graph timer): every workload has its entry, the
    grouped layer carries its direct-stencil timing and the channels-last
    7x7 layer its tensor-core timing."""
    import types
    import bench
    from grouped_convolution_gb300.inputs import WORKLOADS

    picked = {"grp4x8_9x9_s2_bf16_cl": "grp_tc", "dw4x4_m4_f16_nchw": "dw_tc",
              "dw3x3_f32_nchw": "dw_small"}

    class FakeCase:
        def __init__(self, name, sets, dev, schedule=None, *rest):
            self.schedule = schedule or picked.get(name, "dw_row8")
            self.bytes, self.fma, self.pix = 100e6, 1e9, 1e6

        def footprint(self):
            return 1 << 20

    monkeypatch.setattr(bench, "ConvCase", FakeCase)
    monkeypatch.setattr(bench, "BackwardCase", FakeCase)
    monkeypatch.setattr(bench, "time_graph", lambda cases, steps, warm, world: (steps * 0.05, None))
    args = types.SimpleNamespace(steps=20, warmup=3, no_configs=False)
    out = bench.per_config(args, 1, 126 << 20, 6773.5, 39.2e12, None)
    for name in WORKLOADS:
        assert out[name]["us"] == 50.0
    assert out["grp4x8_9x9_s2_bf16_cl"]["direct_stencil"]["schedule"] == "grp_plane"
    tc = out["dw7x7_bf16_cl"]["tensor_cores"]
    assert tc["schedule"] == "dw_tcl" and tc["roofline"]["bound"] == "hbm"
    assert out["dw7x7_bf16_cl"]["schedule"] == "dw_row8"
    assert "tensor_cores" not in out["mbv2_dw3x3_s1_bf16_cl"]
