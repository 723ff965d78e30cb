"""Multi-rank path of bench.py on CPU (gloo, world size 2): the layer runs as
independent replicas, so the only cross-rank steps are the barrier, the
max-over-ranks time and the whole-job token count."""

import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        my_ms = 10.0 + 5.0 * rank           # rank 1 is the slow one
        ms = bench.max_over_ranks_ms(my_ms, world)
        out[rank] = (ms, bench.job_tokens_per_s(4096, world, 50, ms))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    world, port = 2, 29400 + os.getpid() % 500
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == pytest.approx(4096 * 2 * 50 / 0.015)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks_ms(12.5, 1) == 12.5
    assert bench.job_tokens_per_s(4096, 1, 10, 20.0) == pytest.approx(4096 * 10 / 0.02)
