"""bench.py's multi-rank bookkeeping on CPU (gloo, world size 2): the path
shards as independent replicas, so the only cross-rank steps are the
max-over-ranks device time and the sum of work; both are checked here."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.reduce_scalar(1.5 + rank, "max", world)
    s = bench.reduce_scalar(10.0 * (rank + 1), "sum", world)
    bench.barrier(world)
    q.put((rank, t, s))
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_single_rank_identity():
    import bench
    assert bench.reduce_scalar(3.25, "max", 1) == 3.25
    assert bench.reduce_scalar(3.25, "sum", 1) == 3.25


def test_algorithmic_counts():
    import bench
    f, b = bench.algorithmic(R=512, E_act=29, E=32, N=4096, K=6144)
    assert f == 2.0 * 512 * 4096 * 6144
    assert b == 29 * 4096 * 6144 / 2 + 29 * 4096 * 6144 / 32 + 512 * 6144 + 512 * 48 \
        + 2 * 512 * 4096 + 4 * 33
