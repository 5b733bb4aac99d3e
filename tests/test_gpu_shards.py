"""Disjoint target shards concatenate to the whole call, bit for bit.

The walk is independent per group of Morton-ordered targets once the tree
is built, so the work splits over devices by replicating the sources and
giving each device a contiguous range of groups.  One GPU runs every shard
in turn here: each call builds the same tree, forms the same groups and
writes only its own targets' rows.
"""
import numpy as np
import pytest

import workloads as W
from tests import gpu_helpers as H
from tests.test_gpu_parity import SETS

pytestmark = pytest.mark.gpu


def _sharded(src, tgt, shards, **opts):
    import torch
    import barnes_hut_body_gb300 as B
    rows = src.shape[0] if tgt is None else tgt.shape[0]
    d_src = H.to_dev(src)
    d_tgt = None if tgt is None else H.to_dev(tgt)
    bh = B.BarnesHut(theta=0.5, eps=1e-3, **opts)
    bh.set_option("shards", shards)
    out = torch.full((rows, 4), float("nan"), device="cuda")
    written, groups, executed = [], 0, 0
    for s in range(shards):
        bh.set_option("shard", s)
        bh.compute(d_src, d_tgt, out)
        assert bh.status() == 0, B.bh_last_error(bh.ctx)
        written.append(int((~torch.isnan(out[:, 3])).sum().item()))
        ex, ng = B.bh_get_counters(bh.ctx)
        groups += ng
        executed += ex
    bh.close()
    return out.cpu().numpy().astype(np.float64), written, groups, executed


@pytest.mark.parametrize("name", ["uniform4096", "galaxy_2e16", "ragged_12345"])
@pytest.mark.parametrize("shards", [2, 3, 7])
@pytest.mark.parametrize("group,pipeline", [(64, 0), (32, 0), (64, 1)])
def test_self_mode_shards_are_the_whole_call(name, shards, group, pipeline):
    import barnes_hut_body_gb300 as B
    src = SETS[name]
    n = src.shape[0]
    bh, ref, rc = H.gpu_bh(src, eps=1e-3, group=group, pipeline=pipeline)
    assert rc == 0
    ex_all, ng_all = B.bh_get_counters(bh.ctx)
    bh.close()
    got, written, groups, executed = _sharded(src, None, shards, group=group,
                                              pipeline=pipeline)
    np.testing.assert_array_equal(got, ref)
    ng = (n + group - 1) // group
    # shard s writes exactly the targets of its groups, nothing else
    ends = [min(n, group * (ng * (s + 1) // shards)) for s in range(shards)]
    assert written == ends
    assert groups == ng_all == ng and executed == ex_all


@pytest.mark.parametrize("name", ["uniform4096", "dups_5000"])
def test_target_mode_shards_are_the_whole_call(name):
    src = SETS[name]
    tgt = W.query_grid(src, side=29)
    tgt = np.ascontiguousarray(tgt[np.random.default_rng(4).permutation(tgt.shape[0])])
    _, ref, rc = H.gpu_bh(src, tgt, eps=1e-3)
    assert rc == 0
    got, written, _, _ = _sharded(src, tgt, 5)
    np.testing.assert_array_equal(got, ref)
    assert written[-1] == tgt.shape[0]


def test_stochastic_estimator_shards_are_the_whole_call():
    import barnes_hut_body_gb300 as B
    src = SETS["plummer_2e15"]
    opts = dict(estimator=B.BH_EST_STOCHASTIC, seed=11)
    _, ref, rc = H.gpu_bh(src, eps=1e-3, **opts)
    assert rc == 0
    got, _, _, _ = _sharded(src, None, 4, **opts)
    np.testing.assert_array_equal(got, ref)


def test_shard_options_are_checked():
    import barnes_hut_body_gb300 as B
    bh = B.BarnesHut()
    with pytest.raises(B.BHError):
        bh.set_option("shards", 0)
    bh.set_option("shards", 3)
    with pytest.raises(B.BHError):
        bh.set_option("shard", 3)
    bh.set_option("shard", 2)
    bh.close()
