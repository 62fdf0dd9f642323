"""The replica path's host logic with two gloo ranks on CPU: the slowest
rank's time is taken, whole-job throughput counts every rank's bytes, and
the reference arm runs on rank 0 alone."""

import importlib.util
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


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        elapsed = [3.0, 5.0][rank]                      # ms: rank 1 is the slow one
        slowest = bench.max_over_ranks(elapsed, torch.device("cpu"))
        out[rank] = (slowest, bench.job_gbs(1e9, 10, world, slowest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as manager:
        out = manager.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        results = dict(out)
    assert results[0] == results[1]
    slowest, gbs = results[0]
    assert slowest == 5.0
    # 2 ranks x 10 steps x 1 GB in 5 ms
    assert gbs == pytest.approx(2 * 10 * 1e9 / 5e-3 / 1e9)


def test_single_process_needs_no_group():
    bench = _bench()
    assert bench.max_over_ranks(7.5, torch.device("cpu")) == 7.5
    assert bench.job_gbs(2e9, 4, 1, 8.0) == pytest.approx(1000.0)


def _reference_arm(rank):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--gpus", "2", "--steps", "1", "--warmup", "0"],
                          env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_runs_on_rank_zero_only():
    other = _reference_arm(1)
    assert other.returncode == 0 and other.stdout.strip() == ""
    zero = _reference_arm(0)
    assert zero.returncode == 0, zero.stderr[-2000:]
    line = json.loads(zero.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("llama3-70b")
