"""bench.py's multi-rank host logic on two gloo ranks (CPU only): the timed region is the
max over ranks and the units add up (independent replicas, weak scaling)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, world, rank)
    bench.barrier(world)
    el, units = bench.reduce_over_ranks(0.5 + rank, 100.0 * (rank + 1), world)
    out[rank] = (el, units)
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == (1.5, 300.0) and out[1] == (1.5, 300.0)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_over_ranks(2.5, 7.0, 1) == (2.5, 7.0)
