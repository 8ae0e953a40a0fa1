"""The multi-GPU host logic of bench.py on CPU: two gloo ranks, each with
its own shard of tokens (no collective on the data path); the timing is the
maximum over ranks and the throughput counts every rank's tokens."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from birkhoff_projection_gb300 import workloads

    # each rank's shard is distinct
    X, _ = workloads.sweep(10, 1.0, shard=rank)
    first = float(X.reshape(-1)[0])
    local_ms = 100.0 + 50.0 * rank  # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms, dist)
    v = bench.whole_job_tokens_per_s(1 << 10, world, 4, m)
    firsts = [None] * world
    dist.all_gather_object(firsts, first)
    out[rank] = (m, v, firsts)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = 29500 + (os.getpid() % 1000)
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        m, v, firsts = res[r]
        assert m == 150.0
        assert v == pytest.approx(2 * 1024 * 4 / 0.150)
        assert firsts[0] != firsts[1]


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tokens_per_s(100, 1, 10, 1000.0) == pytest.approx(1000.0)
