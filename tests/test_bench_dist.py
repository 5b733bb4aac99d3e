"""The bench's multi-rank host logic on CPU: two gloo ranks, barrier, the
max-over-ranks time and the sum of units over ranks (no GPU)."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, lr, w = bench.dist_env()
    assert (r, lr, w) == (rank, rank, world)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    mx = bench.max_over_ranks(1.0 + rank, w)
    sm = bench.sum_over_ranks(10.0 * (rank + 1), w)
    out.put((rank, mx, sm))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(3.5, 1) == 3.5
