"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Each GPU runs its own full call (replicas, no data-path collective); the only cross-rank
step is the timing aggregation: the job's time is the slowest rank's.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, values, results):
    sys.path.insert(0, ROOT)
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        import bench
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        results[rank] = bench.max_over_ranks(values[rank], world)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("values", [(1.5, 4.25), (9.0, 2.0)])
def test_max_over_ranks_gloo(values):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), list(values), results), nprocs=world,
             join=True)
    assert [results[r] for r in range(world)] == [max(values)] * world


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
