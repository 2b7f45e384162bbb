"""The multi-GPU path of the bench on CPU: N independent replicas over gloo.

The GEMV does not shard (each GPU runs its own replica of the workload), so
the only cross-rank logic is the bench's aggregation: the timed region is the
slowest rank's, the job's value counts every rank's bytes, and the end-to-end
rate is the slowest rank's rate times the number of ranks.  Two gloo ranks on
127.0.0.1 feed different per-rank figures through the same helpers the bench
uses and check what every rank gets back.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_ms = [10.0, 12.5][rank]          # rank 1 is the slower replica
        e2e = [700.0, 650.0][rank]         # GB/s each replica saw end to end
        t = bench.slowest_time_ms(dist, t_ms)
        rate = bench.job_rate(dist, e2e)
        value = bench.job_value(world, 1_000_000, 100, t)
        out.put((rank, t, rate, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_aggregate_like_the_bench():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, t, rate, value in got:
        assert t == pytest.approx(12.5)              # max over ranks
        assert rate == pytest.approx(650.0 * world)  # slowest rate x ranks
        # every rank's bytes (2 x 1e6 x 100) over the slowest rank's 12.5 ms
        assert value == pytest.approx(world * 1e8 / 12.5e-3 / 1e9)


def test_one_gpu_passes_through():
    assert bench.slowest_time_ms(None, 3.5) == 3.5
    assert bench.job_rate(None, 42.0) == 42.0
    assert bench.job_value(1, 2_000, 10, 1.0) == pytest.approx(2e4 / 1e-3 / 1e9)
