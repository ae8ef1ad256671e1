"""Host logic of the multi-replica benchmark path on CPU: two gloo ranks,
max-over-ranks timing and the barrier, as bench.py uses them under torchrun."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.barrier(world)
    local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
    m = bench.reduce_max(local_ms, world)
    q.put((rank, m))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_rank_max_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
