"""The benchmark's multi-rank logic on CPU (gloo, world size 2): every rank
is an independent replica; the job time is the slowest rank's and the job
throughput counts every rank's work.  The GPU path runs one process per GPU
with the same two functions over NCCL."""
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


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        t = bench.max_over_ranks(times[rank], world, device="cpu")
        v = bench.job_throughput(world, 1e12, 10, t)
        out.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [120.0, 150.0]                     # ms for 10 steps on each rank
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, v in res:
        assert t == 150.0                      # the slowest rank
        assert v == pytest.approx(2 * 1e12 * 10 / 0.150 / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1, 2e12, 5, 1000.0) == pytest.approx(10.0)
