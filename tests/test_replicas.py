"""The multi-GPU path is replicas only: each rank runs its own layer copy and the
ranks meet only to time the job (barrier, maximum of the elapsed times). These
tests run that host logic as two gloo ranks on the CPU."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [12.5, 40.0][rank]  # the second replica is the slower one
        m = bench.max_over_ranks(dist, elapsed, torch.device("cpu"))
        dist.barrier()
        out[rank] = (m, bench.job_rate(world, 100, 4, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_on_two_gloo_ranks():
    world = 2
    # the manager process is started with spawn too: no fork of a threaded process
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = {r: out[r] for r in range(world)}
    for r in range(world):
        m, rate = res[r]
        assert m == 40.0  # every rank sees the slowest replica's time
        assert rate == pytest.approx(2 * 100 * 4 / 0.040)  # all ranks' tokens over that time


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(None, 7.0, "cpu") == 7.0
    assert bench.job_rate(1, 10, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm's rank 0 alone works and prints; the other
    ranks exit 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
