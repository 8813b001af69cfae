"""Multi-rank logic of bench.py on CPU: two gloo ranks (replicas, weak scaling).

The decode step shards by sequence with no exchange, so N GPUs run N
independent replicas; the only collectives are the host-side timing
reductions: the slowest rank's time (max) and the total bytes (sum).
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, use_cuda=False)
    t = bench.max_over_ranks(1.5 + rank, w, "cpu")          # rank 1 is the slowest
    b = bench.sum_over_ranks(1000.0 * (rank + 1), w, "cpu")  # bytes add up over replicas
    bench.barrier(w)
    # Timed regions: rank 1's regions take longer; both ranks must stop after
    # the same region, each region counted at the slowest rank's time.
    regions = bench.timed_regions(lambda: 40.0 + 20.0 * rank, 200.0, w, "cpu")
    q.put((rank, t, b, tuple(regions)))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_bytes():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 2.5, 3000.0, (60.0,) * 4), (1, 2.5, 3000.0, (60.0,) * 4)]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
    assert bench.sum_over_ranks(7.0, 1, "cpu") == 7.0
    # Regions are repeated until their sum reaches the floor (at least one).
    assert bench.timed_regions(lambda: 30.0, 100.0, 1, "cpu") == [30.0] * 4
    assert bench.timed_regions(lambda: 500.0, 100.0, 1, "cpu") == [500.0]
