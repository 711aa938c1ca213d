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


def test_replica_command_starts_one_rank_per_gpu():
    sys.path.insert(0, ROOT)
    import bench
    cmd = bench.replica_command(4, ["--steps", "7", "--gpus", "4"], port=29555)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--master-addr=127.0.0.1" in cmd
    assert "--master-port=29555" in cmd
    assert cmd[-4:] == ["--steps", "7", "--gpus", "4"]
    assert cmd[-5].endswith("bench.py")


def test_gpus_must_match_world_size(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit, match="WORLD_SIZE=2"):
        bench.main(["--gpus", "4"])
    monkeypatch.delenv("WORLD_SIZE")
    with pytest.raises(SystemExit, match="at least 1"):
        bench.main(["--gpus", "0"])


def test_algorithmic_bytes_and_flops():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    inp = workloads.make(workloads.WORKLOADS["tiny_causal_64x256"])
    pairs = workloads.valid_pairs(inp["ks"], inp["ke"], inp["N"])
    assert bench.valid_flops(inp) == 2 * 32 * 128 * pairs
    inputs = 64 * 32 * 128 + 64 * 32 * 4 + 256 * 132 + 8 * 64
    assert bench.algorithmic_bytes(inp, 1) == 4 * 64 * 256 + inputs
    assert bench.algorithmic_bytes(inp, 0) == 4 * pairs + inputs
