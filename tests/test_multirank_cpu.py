"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each with
its own copy of the workload (weak scaling, no data-path collective), agree
on the max-over-ranks timing that rank 0 reports."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        times = [1.0 + rank, 10.0 - rank]
        out[rank] = bench.max_over_ranks(times, dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == [2.0, 10.0]


def test_single_rank_max_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1.0]) == [3.5, 1.0]
