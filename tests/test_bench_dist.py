"""bench.py's multi-rank plumbing on the CPU: two gloo ranks, sum of work and
max of time (replicas only: no data-path collective)."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(w)
    units, secs = bench.aggregate(10.0 * (rank + 1), 0.5 + rank, w)
    out[rank] = (units, secs)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (30.0, 1.5)


def test_single_process_is_identity():
    import bench
    assert bench.aggregate(7.0, 2.0, 1) == (7.0, 2.0)
