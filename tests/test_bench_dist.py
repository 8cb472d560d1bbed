"""The benchmark's multi-process bookkeeping on CPU (gloo, world size 2).

Each rank runs its own replica of the workload (weak scaling, no data-path
collective); the only collectives are the timing bookkeeping: the max of the
elapsed times and the sum of the tokens over ranks."""
from __future__ import annotations

import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    ws, r, _ = bench.dist_env()
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    elapsed, units = bench.aggregate(1.5 + rank, 1000.0 * (rank + 1), ws)
    out[rank] = (elapsed, units, r)
    torch.distributed.destroy_process_group()


def test_aggregate_two_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in range(2):
        elapsed, units, r = out[rank]
        assert r == rank
        assert elapsed == 2.5  # max over ranks
        assert units == 3000.0  # sum over ranks


def test_single_rank_is_identity():
    import bench

    assert bench.aggregate(1.25, 42.0, 1) == (1.25, 42.0)
