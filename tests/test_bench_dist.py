"""The multi-GPU bench path's host logic on CPU ranks (gloo, world size 2).

bench.py runs one replica of the workload per rank (the write has no
exchange step) and reports the whole job's throughput over the slowest
rank's time.  These tests run that aggregation with two gloo ranks on the
CPU: the max-over-ranks reduction, the whole-job rate, distinct inputs per
replica, and the reference arm printing on rank 0 only."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wk

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        mx = bench.max_over_ranks(local_ms, dist, "cpu")
        wl = wk.WORKLOADS[0]
        inp = wk.generate(wl, seed=bench.replica_seed(wl, rank))
        digest = float(inp.all_kv.float().sum())
        gathered = [None] * world
        dist.all_gather_object(gathered, digest)
        out[rank] = (mx, gathered)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork from this multi-threaded process
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 5.0
    d0, d1 = res[0][1]
    assert d0 != d1  # each replica has its own seeded inputs


def test_whole_job_rate_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench

    # 2 ranks x 10 steps x 1e6 bytes over 4 ms (the slowest rank) = 5e9 B/s
    assert bench.whole_job_rate(1e6, 10, 2, 4.0) == pytest.approx(5e9)
    assert bench.whole_job_rate(1e6, 10, 1, 4.0) == pytest.approx(2.5e9)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
