"""The replicas path of bench.py on CPU: two gloo ranks (no GPU).

bench.py runs one full step per GPU and reports the slowest rank's time; the whole-job rate
counts every replica's tokens.  These tests exercise that reduction with real
torch.distributed ranks over gloo, and the reference arm's rank rule (rank 0 alone works)."""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured 10 + r ms: every rank must see the slowest, 10 + world - 1
        out[rank] = bench.max_over_ranks(10.0 + rank, dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert [out[r] for r in range(world)] == [11.0, 11.0]


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25


def test_whole_job_rate_scales_with_replicas():
    one = bench.whole_job_rate(20.0, 1)              # 12 layers in 20 ms: 1984 tokens per 20/12 ms
    assert one == pytest.approx(1984 / (20e-3 / 12))
    assert bench.whole_job_rate(20.0, 4) == pytest.approx(4 * one)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
