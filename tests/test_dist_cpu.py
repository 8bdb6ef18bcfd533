"""The N > 1 path of bench.py on CPU (gloo, world size 2): replicas only, so
the only cross-rank operations are the barrier around the timed region and
the maximum of the ranks' times; the reference arm runs on rank 0 alone."""
import argparse
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    args = argparse.Namespace(impl="reference", gpus=world, steps=1, warmup=0)
    w, r, _ = bench.setup_dist(args)
    t = bench.max_over_ranks(1.0 + 2.0 * r, w)     # rank 1 is the slow one
    bench.barrier(w)
    out.put((r, w, t, bench.replica_value(w, 1.0e9, 10, t)))
    dist.destroy_process_group()


def test_max_over_ranks_and_replica_value_gloo():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, w, t, v) in enumerate(got):
        assert rank == r and w == world
        assert t == 3.0                          # the slowest rank's time, on every rank
        assert v == pytest.approx(2 * 1.0e9 * 10 / 3.0 / 1e9)


def test_reference_arm_prints_once_under_torchrun():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_clock_record_parsing():
    """The clocks record the bench prints beside every number: median SM
    clock and power over the samples taken during the timed region, and the
    throttle reasons seen active in any of them (nvidia-smi csv, no units)."""
    import bench
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 2070, 2070, 812.50, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1201.50, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1000.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "power_w": 1000.0,
                 "reasons": ["sw_power_cap"], "samples": 3}
    c.lines = []
    assert bench.ClockSampler.summary(c)["sm_mhz"] is None
