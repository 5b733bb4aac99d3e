"""Tree-topology order (BH_ORDER_TREE) against the oracle and the radix path.

The GASPHiA tree-code page (section 排序算法) takes the spatial order from
the tree: leaves read depth first, each parent handing its children ranges
of the sort array sized by their counts.  Built over Morton digits and then
index digits, that order is the stable (key, index) sort, so the permutation
must equal the oracle's stable sort bit for bit, and every later stage must
give the radix path's results bit for bit.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H
from tests.test_gpu_parity import SETS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import barnes_hut_body_gb300 as B
    return B


def _near_duplicate_pairs(pairs, seed=0):
    """Pairs of points a few quanta apart: each pair shares ~17 Morton digits,
    so the insertion tree needs ~17 nodes per pair (beyond 2 per row)."""
    p = W.uniform_cube(pairs, seed=seed)
    q = p.copy()
    q[:, 2] += 2e-6
    return np.ascontiguousarray(np.concatenate([p, q]), np.float32)


@pytest.mark.parametrize("name", list(SETS))
@pytest.mark.parametrize("bits", [21, 10])
def test_tree_order_is_the_stable_sort_and_the_radix_path(B, name, bits):
    src = SETS[name]
    n = src.shape[0]
    bh_r, a, rc_r = H.gpu_bh(src, key_bits=bits, order=B.BH_ORDER_RADIX, graph=0)
    bh_t, b, rc_t = H.gpu_bh(src, key_bits=bits, order=B.BH_ORDER_TREE, graph=0)
    assert rc_r == 0 and rc_t == 0
    ref = O.sort(O.keys(src, O.bbox(src), bits))
    perm = B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_PERM, n)
    np.testing.assert_array_equal(perm, ref)
    np.testing.assert_array_equal(B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_KEYS, n),
                                  B.bh_debug_export(bh_r.ctx, B.BH_EXPORT_KEYS, n))
    nn = int(B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_NODE_COUNT)[0])
    assert nn == int(B.bh_debug_export(bh_r.ctx, B.BH_EXPORT_NODE_COUNT)[0])
    np.testing.assert_array_equal(B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_NODES, nn),
                                  B.bh_debug_export(bh_r.ctx, B.BH_EXPORT_NODES, nn))
    np.testing.assert_array_equal(a, b)
    bh_r.close()
    bh_t.close()


@pytest.mark.parametrize("name", ["uniform4096", "galaxy_2e16", "dups_5000"])
def test_tree_order_of_separate_targets(B, name):
    src = SETS[name]
    tgt = W.query_grid(src, side=23)
    rng = np.random.default_rng(3)
    tgt = np.ascontiguousarray(tgt[rng.permutation(tgt.shape[0])])
    bh_r, a, rc_r = H.gpu_bh(src, tgt, order=B.BH_ORDER_RADIX, graph=0)
    bh_t, b, rc_t = H.gpu_bh(src, tgt, order=B.BH_ORDER_TREE, graph=0)
    assert rc_r == 0 and rc_t == 0
    m = tgt.shape[0]
    ref = O.sort(O.keys(tgt, O.bbox(tgt), 10))     # targets: 30-bit keys by default
    np.testing.assert_array_equal(B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_TARGET_PERM, m), ref)
    np.testing.assert_array_equal(a, b)
    bh_r.close()
    bh_t.close()


def test_tree_order_repeated_calls_and_graph_replay(B):
    # the insertion tree is rebuilt from scratch by every call (replayed
    # graphs included); the results stay identical
    src = SETS["plummer_2e15"]
    bh = B.BarnesHut(theta=0.5, eps=1e-3, order=B.BH_ORDER_TREE)
    d = H.to_dev(src)
    outs = [bh.compute(d).cpu().numpy() for _ in range(4)]
    assert bh.status() == 0
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])
    _, ref, rc = H.gpu_bh(src, eps=1e-3, order=B.BH_ORDER_RADIX)
    assert rc == 0
    np.testing.assert_array_equal(outs[0].astype(np.float64), ref)
    bh.close()


def test_tree_order_neighbour_search(B):
    import torch
    src = W.uniform_cube(20000, seed=8)
    h = torch.full((src.shape[0],), 0.02, dtype=torch.float32, device="cuda")
    res = []
    for order in (B.BH_ORDER_RADIX, B.BH_ORDER_TREE):
        bh = B.BarnesHut(order=order)
        c, o, lst = B.bh_neighbors(bh.ctx, H.to_dev(src), h, 2.0, B.BH_NB_SYMMETRIC)
        torch.cuda.synchronize()
        assert bh.status() == 0
        res.append((c.cpu().numpy(), o.cpu().numpy()))
        bh.close()
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])


def test_tree_order_pool_overflow_is_reported_and_recovers(B):
    # 2000 pairs need ~17 trie nodes per pair, far beyond the pool of
    # 2 x rows + 64 nodes: the build flags BH_ETREE_OVERFLOW and later stages
    # run on the identity order; the status read grows the pool 4x, so the
    # same call repeated is exact (the radix path's result, bit for bit);
    # and another input is exact too
    src = _near_duplicate_pairs(2000, seed=5)
    for graph in (0, 1):
        bh = B.BarnesHut(theta=0.5, eps=1e-3, order=B.BH_ORDER_TREE, graph=graph)
        d = H.to_dev(src)
        bh.compute(d)
        assert bh.status() == B.BH_ETREE_OVERFLOW
        again = [bh.compute(d).cpu().numpy().astype(np.float64) for _ in range(3)]
        assert bh.status() == 0
        _, ref_pairs, rc = H.gpu_bh(src, eps=1e-3)
        assert rc == 0
        for a in again:
            np.testing.assert_array_equal(a, ref_pairs)
        bh.close()
    bh = B.BarnesHut(theta=0.5, eps=1e-3, order=B.BH_ORDER_TREE, graph=0)
    bh.compute(H.to_dev(src))
    assert bh.status() == B.BH_ETREE_OVERFLOW
    ok = H.to_dev(SETS["uniform4096"])
    got = bh.compute(ok).cpu().numpy().astype(np.float64)
    assert bh.status() == 0
    _, ref, rc = H.gpu_bh(SETS["uniform4096"], eps=1e-3)
    assert rc == 0
    np.testing.assert_array_equal(got, ref)
    bh.close()


@pytest.mark.parametrize("name", ["lattice1m_shuffled", "galaxy5m"])
def test_tree_order_full_size(B, name):
    """The two workloads bench.py --order tree times, at full size (1M
    shuffled lattice, 5M galaxy pair): the permutation equals the oracle's
    stable sort, the sorted keys and every tree node equal the oracle's, and
    the results equal the radix path's bit for bit."""
    src, tgt, G, eps, theta = W.make(name)
    n = src.shape[0]
    bh_t, b, rc_t = H.gpu_bh(src, theta=theta, G=G, eps=eps, order=B.BH_ORDER_TREE)
    assert rc_t == 0
    o = O.OracleBH(src, theta=theta, G=G, eps=eps, leaf_cap=16)
    np.testing.assert_array_equal(B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_PERM, n), o.perm)
    np.testing.assert_array_equal(B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_KEYS, n), o.skeys)
    nn = int(B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_NODE_COUNT)[0])
    H.assert_tree_equal(B.bh_debug_export(bh_t.ctx, B.BH_EXPORT_NODES, nn), o.tree)
    bh_t.close()
    bh_r, a, rc_r = H.gpu_bh(src, theta=theta, G=G, eps=eps, order=B.BH_ORDER_RADIX)
    assert rc_r == 0
    np.testing.assert_array_equal(a, b)
    bh_r.close()
