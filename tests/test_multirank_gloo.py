"""The bench's multi-rank path on the CPU: two gloo ranks (world_size 2) take the
slowest rank's time and report the whole job's tokens; under torchrun the
reference arm runs on rank 0 only and the other ranks exit without work."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(10.0 + 20.0 * rank, world, torch.device("cpu"))
        out[rank] = (ms, bench.job_tokens_per_s(world, 4, 32, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork of a threaded process
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    assert out[0][0] == out[1][0] == 30.0
    assert out[0][1] == pytest.approx(2 * 4 * 32 / 0.030)


def test_single_rank_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1, None) == 12.5
    assert bench.job_tokens_per_s(1, 8, 10, 100.0) == pytest.approx(800.0)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env["RANK"], env["LOCAL_RANK"] = "0", "0"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["unit"] == "tok/s" and line["value"] > 0
