"""Pins for the oracle's SPH neighbour search ("树结构（基于根据 Burtscher 和
Pingali 的研究）" page, sections 粒子领域搜索 and 树遍历计算; GASPHiA's per-node
maximum smoothing length for the symmetric search).

What fixes it independently of its own code: a lattice whose neighbour counts
follow from counting lattice offsets; scipy's KD-tree ball query (a separate
library implementation of the gather search); the identity between the
symmetric search and the union of the two gather relations; degenerate
smoothing lengths.
"""
import itertools

import numpy as np
import pytest

import oracle as O
import workloads as W


def test_lattice_counts_from_offsets():
    side, a = 10, 0.1
    pm = W.lattice(side, spacing=a)
    h = np.full(pm.shape[0], 0.75 * a, np.float32)     # kappa h = 1.5 a
    counts, lists = O.neighbors(pm, h, kappa=2.0, mode=O.NB_GATHER)
    # offsets with |d|^2 in {1, 2} (lattice units) lie inside 1.5 a; |d|^2 = 3
    # (1.73 a) and 4 (2 a) lie outside
    offs = [d for d in itertools.product((-1, 0, 1), repeat=3) if 1 <= sum(x * x for x in d) <= 2]
    assert len(offs) == 18
    idx = np.arange(side ** 3)
    ijk = np.stack([idx % side, (idx // side) % side, idx // side ** 2], axis=1)
    expect = np.zeros(idx.size, np.int64)
    for d in offs:
        q = ijk + np.array(d)
        expect += np.all((q >= 0) & (q < side), axis=1)
    np.testing.assert_array_equal(counts, expect)
    interior = np.all((ijk > 0) & (ijk < side - 1), axis=1)
    assert np.all(counts[interior] == 18)


def test_gather_matches_scipy_ball_query():
    spatial = pytest.importorskip("scipy.spatial")
    pm, h = W.sph_plummer(4000, seed=9)
    kappa = 2.0
    counts, lists = O.neighbors(pm, h, kappa, O.NB_GATHER)
    x = pm[:, :3].astype(np.float64)
    tree = spatial.cKDTree(x)
    for i in range(0, 4000, 7):
        r = kappa * float(h[i])
        ref = set(tree.query_ball_point(x[i], r)) - {i}
        got = set(lists[i].tolist())
        # pairs within rounding of the support radius may fall either way
        sym = ref ^ got
        for j in sym:
            d = np.linalg.norm(x[i] - x[j])
            assert abs(d - r) <= 1e-5 * r, (i, j, d, r)
        assert counts[i] == len(got)


def test_symmetric_is_union_of_gather_relations():
    pm, h = W.sph_plummer(3000, seed=10)
    _, g = O.neighbors(pm, h, 2.0, O.NB_GATHER)
    _, s = O.neighbors(pm, h, 2.0, O.NB_SYMMETRIC)
    union = [set(x.tolist()) for x in g]
    for i, gi in enumerate(g):
        for j in gi.tolist():
            union[j].add(i)
    for i in range(len(s)):
        assert set(s[i].tolist()) == union[i], i
        # symmetric: i in N(j) iff j in N(i)
    pairs = {(i, j) for i in range(len(s)) for j in s[i].tolist()}
    assert all((j, i) in pairs for i, j in pairs)


def test_lists_sorted_without_self():
    pm, h = W.uniform_sph(2000, seed=4, n_ngb=30)
    counts, lists = O.neighbors(pm, h, 2.0, O.NB_SYMMETRIC)
    for i, l in enumerate(lists):
        assert counts[i] == l.size
        assert i not in set(l.tolist())
        assert np.all(np.diff(l) > 0)
    assert 20 < counts.mean() < 40


def test_degenerate_smoothing_lengths():
    pm = np.zeros((5, 4), np.float32)
    pm[:, 3] = 1.0
    pm[3:, 0] = 1.0                        # two groups of coincident points
    h0 = np.zeros(5, np.float32)
    counts, _ = O.neighbors(pm, h0, 2.0, O.NB_SYMMETRIC)
    assert np.all(counts == 0)              # r^2 < 0 never holds
    h = np.full(5, 1e-3, np.float32)
    counts, lists = O.neighbors(pm, h, 2.0, O.NB_GATHER)
    np.testing.assert_array_equal(counts, [2, 2, 2, 1, 1])
    assert lists[3].tolist() == [4]
    # one large h reaches the other group only in the symmetric search
    h[0] = 1.0
    cg, _ = O.neighbors(pm, h, 2.0, O.NB_GATHER)
    cs, _ = O.neighbors(pm, h, 2.0, O.NB_SYMMETRIC)
    assert cg.tolist() == [4, 2, 2, 1, 1]
    assert cs.tolist() == [4, 2, 2, 2, 2]
