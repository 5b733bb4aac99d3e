"""Group schedule (BH_OPT_SCHEDULE): a call over the same groups as the
previous one hands them to the walk heaviest first, by the terms each group
evaluated in that call.  Each group is walked by one warp (pair) in a fixed
way whatever the order the groups are taken in, so every result, counter and
per-group cost is the Morton-order walk's, bit for bit.  These sets have
fewer groups than the walk takes at once, where the default (1) keeps Morton
order, so most tests force the schedule (2).
"""
import numpy as np
import pytest

import workloads as W
from tests import gpu_helpers as H
from tests.test_gpu_parity import SETS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import barnes_hut_body_gb300 as B
    return B


def _calls(B, src, tgt, k, **opts):
    """k calls on one context: outputs, counters, group costs and orders."""
    import torch
    bh = B.BarnesHut(theta=0.5, eps=1e-3, **opts)
    d_src = H.to_dev(src)
    d_tgt = None if tgt is None else H.to_dev(tgt)
    res = []
    for _ in range(k):
        out = bh.compute(d_src, d_tgt)
        torch.cuda.synchronize()
        ex, ng = B.bh_get_counters(bh.ctx)
        cost = order = None
        if opts.get("schedule", 1):
            cost = B.bh_debug_export(bh.ctx, B.BH_EXPORT_GROUP_COST, ng)
            try:
                order = B.bh_debug_export(bh.ctx, B.BH_EXPORT_GROUP_ORDER, ng)
            except B.BHError:
                order = None
        res.append((out.cpu().numpy(), ex, ng, cost, order))
    assert bh.status() == 0
    bh.close()
    return res


def _check_order(cost_prev, order):
    """A permutation of the groups whose previous costs fall in
    non-increasing power-of-two classes."""
    ng = cost_prev.shape[0]
    np.testing.assert_array_equal(np.sort(order), np.arange(ng, dtype=np.uint32))
    c = cost_prev[order].astype(np.uint64)
    cls = np.where(c > 0, np.floor(np.log2(np.maximum(c, 1))).astype(np.int64), -1)
    assert np.all(np.diff(cls) <= 0)


@pytest.mark.parametrize("name", ["uniform4096", "plummer_2e15", "galaxy_2e16", "ragged_12345"])
@pytest.mark.parametrize("group,pipeline", [(0, 1), (64, 0), (32, 1)])
@pytest.mark.parametrize("graph", [0, 1])
def test_scheduled_walk_is_the_morton_order_walk(B, name, group, pipeline, graph):
    src = SETS[name]
    ref = _calls(B, src, None, 1, schedule=0, group=group, pipeline=pipeline, graph=graph)[0]
    got = _calls(B, src, None, 4, schedule=2, group=group, pipeline=pipeline, graph=graph)
    assert got[0][4] is None                       # no history: Morton order
    for k, (out, ex, ng, cost, order) in enumerate(got):
        np.testing.assert_array_equal(out, ref[0])
        assert (ex, ng) == (ref[1], ref[2])
        # the per-group costs add up to the executed-term counter, and do not
        # depend on the order
        assert int(cost.astype(np.uint64).sum()) == ex
        np.testing.assert_array_equal(cost, got[0][3])
        if k > 0:
            assert order is not None
            _check_order(got[k - 1][3], order)


def test_scheduled_source_target_walk(B):
    src = SETS["galaxy_2e16"]
    tgt = W.query_grid(src, side=27)
    tgt = np.ascontiguousarray(tgt[np.random.default_rng(2).permutation(tgt.shape[0])])
    ref = _calls(B, src, tgt, 1, schedule=0)[0]
    for out, ex, ng, _, _ in _calls(B, src, tgt, 3, schedule=2):
        np.testing.assert_array_equal(out, ref[0])
        assert (ex, ng) == (ref[1], ref[2])


def test_schedule_follows_the_group_count(B):
    # a call over a different number of groups walks in Morton order and
    # starts a new history; results stay exact throughout
    import torch
    a, b = SETS["ragged_12345"], SETS["plummer_2e15"]
    bh = B.BarnesHut(theta=0.5, eps=1e-3, graph=0, schedule=2)
    seq = [a, a, b, b, a]
    ordered = []
    for src in seq:
        out = bh.compute(H.to_dev(src)).cpu().numpy().astype(np.float64)
        torch.cuda.synchronize()
        try:
            B.bh_debug_export(bh.ctx, B.BH_EXPORT_GROUP_ORDER, 1 << 16)
            ordered.append(True)
        except B.BHError:
            ordered.append(False)
        _, ref, rc = H.gpu_bh(src, eps=1e-3, schedule=0)
        assert rc == 0
        np.testing.assert_array_equal(out, ref)
    assert ordered == [False, True, False, True, False]
    assert bh.status() == 0
    bh.close()


def test_shards_and_stochastic_estimator_keep_morton_order(B):
    src = SETS["plummer_2e15"]
    bh = B.BarnesHut(theta=0.5, eps=1e-3, schedule=2)
    bh.set_option("shards", 2)
    d = H.to_dev(src)
    for _ in range(3):
        bh.compute(d)
        with pytest.raises(B.BHError):
            B.bh_debug_export(bh.ctx, B.BH_EXPORT_GROUP_ORDER, 1 << 16)
    bh.close()
    bh = B.BarnesHut(theta=0.5, eps=1e-3, estimator=B.BH_EST_STOCHASTIC, seed=3, schedule=2)
    for _ in range(3):
        bh.compute(d)
        with pytest.raises(B.BHError):
            B.bh_debug_export(bh.ctx, B.BH_EXPORT_GROUP_COST, 1 << 16)
    assert bh.status() == 0
    bh.close()


def test_default_schedule_keeps_morton_order_when_all_groups_start_at_once(B):
    # 2048 groups of 32 < 16 warps per SM taking groups: no reordering, but
    # the costs are recorded
    src = SETS["galaxy_2e16"]
    got = _calls(B, src, None, 3, schedule=1)
    for out, ex, ng, cost, order in got:
        assert order is None
        assert int(cost.astype(np.uint64).sum()) == ex


def test_default_schedule_reorders_a_large_walk(B):
    # a uniform cube of 400k points: 6250 groups of 64, more than the walk
    # takes at once on a GB300 (16 per SM)
    src = W.uniform_cube(400_000, seed=12)
    ref = _calls(B, src, None, 1, schedule=0)[0]
    got = _calls(B, src, None, 3, schedule=1)
    assert got[0][4] is None and got[1][4] is not None
    for k, (out, ex, ng, cost, order) in enumerate(got):
        np.testing.assert_array_equal(out, ref[0])
        assert (ex, ng) == (ref[1], ref[2])
        if k > 0:
            _check_order(got[k - 1][3], order)


def test_schedule_option_is_checked(B):
    bh = B.BarnesHut()
    with pytest.raises(B.BHError):
        bh.set_option("schedule", 3)
    bh.set_option("schedule", 0)
    bh.close()
