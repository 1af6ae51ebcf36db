"""The bench's multi-rank host logic (barrier, max over ranks, whole-job value) on CPU with
gloo, world size 2.  Each rank runs an independent replica; nothing on the data path is
exchanged, only the timing reduction."""
import os
import socket

import pytest
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
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(world)
    mine = 1.0 + rank * 2.5                   # per-rank mean step time (ms)
    worst = bench.max_over_ranks(mine, world)
    out[rank] = worst
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 3.5, 1: 3.5}
