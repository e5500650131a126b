"""bench.py's multi-rank path (replicas) on CPU with gloo, world size 2.

Each rank reports its own elapsed time; the whole-job figure must use the
slowest rank's time and the bytes of all ranks.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.dist_init(world, "gloo")
    elapsed = 1.0 + rank            # rank 1 is the slow one
    agg = bench.aggregate_throughput(units_per_rank=10.0, elapsed_s=elapsed, world=world)
    rank_env = bench.dist_env()
    bench.barrier(world)
    results[rank] = (agg["elapsed_s"], agg["units"], agg["throughput"], rank_env)
    dist.destroy_process_group()


def test_replica_aggregation_gloo_world2():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        elapsed, units, thr, env = res[rank]
        assert elapsed == 2.0                       # max over ranks
        assert units == 20.0                        # all ranks' work
        assert abs(thr - 10.0) < 1e-12              # 20 units / 2 s
        assert env == (rank, world, rank)


def test_single_rank_is_identity():
    import bench
    agg = bench.aggregate_throughput(5.0, 0.5, world=1)
    assert agg == {"elapsed_s": 0.5, "units": 5.0, "throughput": 10.0}
