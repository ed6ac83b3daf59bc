"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, each timing its own
independent replay problem; the job's time is the slowest rank's and its throughput
counts the units of every rank."""
import os
import socket
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


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [40.0, 55.0][rank]                      # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world)
        rate = bench.whole_job_rate(1e12, world, slowest)
        seed = bench.rank_seed(7, rank)
        seeds = [None] * world
        dist.all_gather_object(seeds, seed)
        q.put((rank, slowest, rate, seeds))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_units():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate, seeds in out:
        assert slowest == 55.0
        assert rate == pytest.approx(1e12 * 2 / 55e-3)
        assert len(set(seeds)) == world              # every rank draws its own problem


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(2.0, 1, 1000.0) == pytest.approx(2.0)
