"""The N > 1 path of bench.py on the CPU: independent replicas coordinated by
a barrier and a max over ranks (gloo, world size 2), and the reference arm
under torchrun, where rank 0 alone runs and prints one line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.launch_env()
        assert (r, w, lr) == (rank, world, rank)
        rep = bench.Replicas(dist, "cpu")
        rep.barrier()
        # each replica's own step time; the reported time is the slowest one
        got = rep.max(1.5 + rank)
        rep.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_replica, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_group():
    rep = bench.Replicas(None)
    rep.barrier()
    assert rep.max(3.25) == 3.25


def test_reference_arm_under_torchrun_prints_one_line():
    """Two ranks of `bench.py --impl reference`: rank 0 times the oracle and
    prints the line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=%d" % _free_port(), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
