"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

The path shards by tokens with no exchange (weak scaling, one batch per
rank), so the only collectives are the bench's barrier and the max over ranks
of the measured time; both are exercised here without a GPU.
"""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        my_ms = 2.0 + rank                      # rank 1 is the slow one
        dist.barrier()
        job_ms = bench.max_over_ranks(my_ms, world)
        value = bench.job_throughput(1000, world, job_ms * 1e-3)
        # every rank draws a different batch of the same shape
        from moe_routing_precision_gb300 import workloads
        s = workloads.make_scores(workloads.WORKLOADS["tiny"], seed=bench.shard_seed(rank))
        digest = float(s.sum())
        q.put((rank, job_ms, value, digest, tuple(s.shape)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_scaling():
    world = 2
    port = 29500 + (os.getpid() % 2000)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert all(r[1] == 3.0 for r in res)                  # the slowest rank's time
    assert all(r[2] == pytest.approx(1000 * 2 / 3e-3) for r in res)
    assert res[0][3] != res[1][3]                          # distinct shards
    assert res[0][4] == res[1][4]                          # same shape per rank


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_throughput(10, 1, 2.0) == 5.0
