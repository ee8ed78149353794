"""The multi-GPU mode is replicas only: N ranks each run the whole step on
their own GPU, the job's time is the slowest rank's, and the job's rate is
the bytes of all ranks over that time. The host logic of that mode, on two
CPU ranks with the gloo backend (no GPU)."""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        mine = 1.0 + 0.5 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(mine, world, "cpu")
        results[rank] = (slowest, bench.whole_job_gbs(1_000_000_000, world, 10, slowest))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_the_job_rate():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_rank, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    for r in range(world):
        slowest, rate = got[r]
        assert slowest == 1.5
        assert rate == pytest.approx(2 * 10 * 1.0 / 1.5)  # GB/s: 2 ranks x 10 steps x 1 GB over 1.5 s


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(2.0, 1, "cpu") == 2.0
    assert bench.whole_job_gbs(2_000_000_000, 1, 5, 2.0) == pytest.approx(5.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == ""
