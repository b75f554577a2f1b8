"""Multi-process paths of bench.py on the CPU (gloo, world size 2).

The forward pass has no cross-GPU exchange: `bench.py --gpus N` runs one
replica per GPU, and the job's time is the slowest rank's.  These tests cover
that host logic without a GPU: the max-over-ranks reduction and the job rate
on two gloo ranks, and the reference arm under torchrun, where rank 0 alone
works and prints one JSON line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 1.5 + rank  # rank 1 is the slow one
        worst = bench.max_over_ranks(mine, world, torch.device("cpu"))
        rate = bench.job_throughput(1000, world, worst)
        out[rank] = (worst, rate)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (2.5, 1000 * 2 / 2.5)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, None) == 3.25
    assert bench.job_throughput(10, 1, 2.0) == 5.0


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` under torchrun: rank 0 times the oracle and
    prints one line; rank 1 exits 0 without work."""
    pytest.importorskip("torch.distributed.run")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "ref_small"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
