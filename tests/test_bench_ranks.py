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


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line
    with the reference arm's keys; it needs no GPU."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["steps"] == 1 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_latent_flop_counts_match_a_pair_count():
    """The latent sweep's algorithmic FLOPs are the visible (query row, key) pairs times
    the per-pair products: 576 + 512 MACs forward; 576 + 512 + 576 backward plus
    512 + 576 for each pair with a response key (the response rows' gradient)."""
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    for P, R, H in [(0, 1, 1), (37, 5, 3), (1000, 64, 64)]:
        pairs = sum((P + t + 1) * H for t in range(R))
        resp = sum((t + 1) * H for t in range(R))
        fwd, fwd_exe = bench.mla_flops(P, R, H)
        bwd, bwd_exe = bench.mla_bwd_flops(P, R, H)
        assert fwd == pytest.approx(pairs * 2 * (576 + 512), rel=1e-12)
        assert bwd == pytest.approx(pairs * 2 * (576 + 512 + 576) + resp * 2 * (512 + 576),
                                    rel=1e-12)
        assert fwd_exe >= fwd and bwd_exe >= bwd
