"""The bench's target split over ranks, on CPU with two gloo ranks: each
rank fills the rows of its shard of the Morton-ordered groups (stub rows from
the oracle's group walk) into a zeroed buffer, gather_rows combines them, and
every rank must then hold the whole oracle call's rows, bit for bit."""
import os
import socket

import numpy as np


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_rows(shards, shard):
    import oracle as O
    import workloads as W
    import bench
    src = W.plummer(3000, seed=41)
    o = O.OracleBH(src, theta=0.5, eps=1e-3, leaf_cap=16)
    group = 32
    ng = (src.shape[0] + group - 1) // group
    g0, g1 = bench.shard_groups(ng, shards, shard)
    out, rows, _ = o.bh_group(group=group, mode=0, groups=np.arange(g0, g1))
    whole, wrows, _ = o.bh_group(group=group, mode=0)
    full = np.zeros((src.shape[0], 4), np.float32)
    full[wrows] = whole.astype(np.float32)
    mine = np.zeros((src.shape[0], 4), np.float32)
    mine[rows] = out.astype(np.float32)
    return mine, full


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import bench
    bench.dist_init(world, "gloo")
    mine, full = _oracle_rows(world, rank)
    walked = int((np.abs(mine).sum(1) > 0).sum())
    t = torch.from_numpy(mine.copy())
    bench.gather_rows(t, world)
    out.put((rank, bool(np.array_equal(t.numpy(), full)), walked))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_split_targets_and_gather_rows():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [True, True]
    # both ranks walked a share, and the shares cover all 3000 rows
    assert res[0][2] > 0 and res[1][2] > 0 and res[0][2] + res[1][2] == 3000


def test_shard_groups_partition():
    import bench
    for ng in (1, 7, 94, 15625):
        for shards in (1, 2, 3, 8):
            spans = [bench.shard_groups(ng, shards, s) for s in range(shards)]
            assert spans[0][0] == 0 and spans[-1][1] == ng
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))


def test_stage_ms_is_the_gpu_breakdown():
    """stage_ms comes from the GPU's per-stage times (one key per
    bh_get_stage_times stage); the CPU oracle's stages live elsewhere."""
    import bench
    import barnes_hut_body_gb300 as B
    steps = [{k: float(i + j) for j, k in enumerate(B.STAGES)} for i in range(5)]
    med = bench.gpu_stage_medians(steps)
    assert list(med) == list(B.STAGES)
    assert med["bbox"] == 2.0 and med["traverse"] == 2.0 + len(B.STAGES) - 1
    hb = bench.stage_hbm(med, bench.stage_bytes(1000, 1000, 500, True), 6790.7)
    assert set(hb["frac"]) <= set(B.STAGES)
    # build = 8 B per key + 32 B per node, centre of mass = 16 B per particle
    # + 32 B per node
    b = bench.stage_bytes(1000, 1000, 500, True)
    assert b["build"] == 8 * 1000 + 32 * 500 and b["com"] == 16 * 1000 + 32 * 500
