"""Pins for the CPU oracle: closed forms, invariants and brute force.

None of these compares the oracle with itself.  Each targets a plausible
mistake: a dropped G or eps, a sign, a swapped axis, a wrong exponent, a
missing self-skip, a non-strict opening test, a half-edge w, a wrong tree.
"""
import math
import os

import numpy as np
import pytest

import workloads as W
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# direct sum: closed forms
# --------------------------------------------------------------------------
def test_two_body_closed_form(orc):
    """Two softened masses: a_1 = G m_2 d/(|d|^2+eps^2)^{3/2} toward body 2,
    phi_1 = -G m_2/sqrt(|d|^2+eps^2); every axis distinct so a swap shows."""
    p = np.array([[0.125, -0.25, 0.5, 2.0], [0.5, 0.0, -0.375, 3.0]], np.float32)
    G, eps = 1.75, 0.0625
    out = orc.direct(p, None, G, eps)
    d = p[1, :3].astype(np.float64) - p[0, :3]
    s = d @ d + eps * eps
    np.testing.assert_allclose(out[0, :3], G * 3.0 * d / s ** 1.5, rtol=1e-14)
    np.testing.assert_allclose(out[1, :3], -G * 2.0 * d / s ** 1.5, rtol=1e-14)
    np.testing.assert_allclose(out[0, 3], -G * 3.0 / math.sqrt(s), rtol=1e-14)
    np.testing.assert_allclose(out[1, 3], -G * 2.0 / math.sqrt(s), rtol=1e-14)
    # the tree walk reaches the same closed form (N=2: both terms exact)
    o = orc.OracleBH(p, theta=0.7, G=G, eps=eps)
    b, terms = o.bh()
    np.testing.assert_allclose(b, out, rtol=1e-14)
    assert list(terms) == [1, 1]


def test_single_softened_source_field(orc):
    """One source of mass m seen from targets is the Plummer-sphere field of
    scale eps: phi = -G m/sqrt(r^2+eps^2), a = -G m (x-c)/(r^2+eps^2)^{3/2}."""
    c = np.array([[0.25, 0.5, -0.75, 1.5]], np.float32)
    g = W.rng(11)
    t = np.zeros((64, 4), np.float32)
    t[:, :3] = (c[0, :3] + g.normal(size=(64, 3)) * 0.3).astype(np.float32)
    G, eps = 0.5, 0.01
    out = orc.direct(c, t, G, eps)
    x = t[:, :3].astype(np.float64) - c[0, :3]
    s = (x * x).sum(1) + eps * eps
    np.testing.assert_allclose(out[:, 3], -G * 1.5 / np.sqrt(s), rtol=1e-14)
    np.testing.assert_allclose(out[:, :3], -G * 1.5 * x / s[:, None] ** 1.5, rtol=1e-13)


def test_self_pair_skipped_and_duplicates_kept(orc):
    """N=1 in self mode feels nothing; two coincident bodies feel a = 0 and
    phi = -G m/eps from each other (the self pair is skipped by index only)."""
    one = np.array([[0.3, 0.2, 0.1, 5.0]], np.float32)
    assert np.all(orc.direct(one, None, 1.0, 0.1) == 0.0)
    two = np.array([[0.3, 0.2, 0.1, 5.0], [0.3, 0.2, 0.1, 2.0]], np.float32)
    out = orc.direct(two, None, 1.0, 0.25)
    np.testing.assert_allclose(out[:, :3], 0.0, atol=0)
    np.testing.assert_allclose(out[:, 3], [-2.0 / 0.25, -5.0 / 0.25], rtol=1e-15)


def test_newton_third_law(orc):
    """sum_i m_i a_i = 0 for the direct sum in self mode."""
    p = W.uniform_cube(512, seed=7)
    out = orc.direct(p, None, 1.0, 1e-3)
    m = p[:, 3].astype(np.float64)[:, None]
    net = np.abs((m * out[:, :3]).sum(0)).max()
    scale = (m[:, 0] * np.linalg.norm(out[:, :3], axis=1)).sum()
    assert net <= 1e-12 * scale


def test_uniform_ball_interior(orc):
    """Inside a uniform ball (mass M, radius R): a(r) = -G M r/R^3 and
    phi(r) = -G M (3R^2 - r^2)/(2R^3).  The shell-mean radial field is
    checked to 3/sqrt(N(<r)), the Poisson noise of the enclosed mass."""
    n = 1 << 16
    p = W.uniform_ball(n, seed=6, radius=1.0, total_mass=1.0)
    g = W.rng(60)
    t = np.zeros((3000, 4), np.float32)
    d = g.normal(size=(3000, 3))
    d /= np.linalg.norm(d, axis=1)[:, None]
    t[:, :3] = d * (0.25 + 0.35 * g.random(3000))[:, None]
    out = orc.direct(p, t, 1.0, 1e-3)
    x = t[:, :3].astype(np.float64)
    rr = np.linalg.norm(x, axis=1)
    ar = (out[:, :3] * x).sum(1) / rr                # radial component
    edges = np.linspace(0.25, 0.6, 6)
    for lo, hi in zip(edges[:-1], edges[1:]):
        s = (rr >= lo) & (rr < hi)
        rel = ar[s].mean() / (-rr[s].mean()) - 1.0
        assert abs(rel) < 3.0 / math.sqrt(n * lo ** 3)
    phi_exact = -(3.0 - rr * rr) / 2.0
    np.testing.assert_allclose(out[:, 3], phi_exact, rtol=0.02)


def test_plummer_acceleration(orc):
    """Truncated Plummer sphere (scale a, masses scaled so the sample inside
    20a has mass 1): inside the truncation the field is the untruncated one of
    mass 1/u_max, a(r) = -G M r/(r^2+a^2)^{3/2}."""
    n = 1 << 16
    a = 0.1
    p = W.plummer(n, seed=4, a=a)
    r = np.linalg.norm(p[:, :3].astype(np.float64), axis=1)
    idx = np.nonzero((r > 0.03) & (r < 0.5))[0][:3000]
    out = orc.direct(p, None, 1.0, 1e-3, idx=idx)
    rr = r[idx]
    ar = (out[:, :3] * p[idx, :3].astype(np.float64)).sum(1) / rr
    mfull = 1.0 / (400.0 / 401.0) ** 1.5
    edges = np.array([0.03, 0.06, 0.1, 0.16, 0.25, 0.5])
    for lo, hi in zip(edges[:-1], edges[1:]):
        s = (rr >= lo) & (rr < hi)
        exact = (-mfull * rr[s] / (rr[s] ** 2 + a * a) ** 1.5).mean()
        assert abs(ar[s].mean() - exact) < 0.03 * abs(exact)


def test_scale_and_translation(orc):
    """Positions x2 and eps x2 scale a by 1/4 and phi by 1/2 exactly (powers
    of two); a translation by an exactly representable shift leaves the tree
    and (to rounding) the forces unchanged."""
    g = W.rng(21)
    pos = g.integers(0, 1024, size=(300, 3)) / 1024.0
    p = np.zeros((300, 4), np.float32)
    p[:, :3] = pos
    p[:, 3] = g.integers(1, 8, size=300) / 8.0
    q = p.copy()
    q[:, :3] *= 2.0
    o1 = orc.OracleBH(p, theta=0.6, eps=1e-3, leaf_cap=4)
    o2 = orc.OracleBH(q, theta=0.6, eps=2e-3, leaf_cap=4)
    assert np.array_equal(o1.keys, o2.keys)
    b1, _ = o1.bh()
    b2, _ = o2.bh()
    np.testing.assert_array_equal(b2[:, :3], b1[:, :3] / 4.0)
    np.testing.assert_array_equal(b2[:, 3], b1[:, 3] / 2.0)
    s = p.copy()
    s[:, :3] += 8.0
    o3 = orc.OracleBH(s, theta=0.6, eps=1e-3, leaf_cap=4)
    assert np.array_equal(o1.keys, o3.keys)
    b3, _ = o3.bh()
    np.testing.assert_allclose(b3, b1, rtol=1e-9, atol=1e-9 * np.abs(b1).max())


# --------------------------------------------------------------------------
# keys and sort
# --------------------------------------------------------------------------
def test_interleave_pins(orc):
    assert orc.interleave(1, 0, 0) == 1
    assert orc.interleave(0, 1, 0) == 2
    assert orc.interleave(0, 0, 1) == 4
    assert orc.interleave(2, 0, 0) == 8
    assert orc.interleave(0, 0, 2) == 32
    m21 = (1 << 21) - 1
    assert orc.interleave(m21, m21, m21) == (1 << 63) - 1
    assert orc.interleave(1023, 1023, 1023, 10) == (1 << 30) - 1
    g = W.rng(3)
    for _ in range(200):
        q = tuple(int(v) for v in g.integers(0, 1 << 21, size=3))
        assert brute.decode(orc.interleave(*q), 21) == q


def test_quantisation_pins(orc):
    """Cube [0,1]^3 (lo=0, L=1): q = trunc(x * 2^b), clamped; a point on a
    split plane goes to the upper half."""
    p = np.array([[0, 0, 0, 1], [1, 1, 1, 1], [0.5, 0.25, 0.75, 1],
                  [np.nextafter(np.float32(0.5), np.float32(0)), 0.125, 0.0, 1]],
                 np.float32)
    cube = orc.bbox(p)
    assert list(cube) == [0, 0, 0, 1]
    q = orc.quantise(p, cube, 21)
    assert list(q[0]) == [0, 0, 0]
    assert list(q[1]) == [(1 << 21) - 1] * 3
    assert list(q[2]) == [1 << 20, 1 << 19, 3 << 19]
    assert list(q[3]) == [(1 << 20) - 1, 1 << 18, 0]
    k = orc.keys(p, cube, 21)
    assert k[2] == orc.interleave(1 << 20, 1 << 19, 3 << 19)
    # top-level octant of (0.5, 0.25, 0.75): x upper (+1), y lower, z upper (+4)
    assert int(k[2]) >> 60 == 5


def test_bbox_rules(orc):
    p = np.array([[1, 2, 3, 1], [1, 2, 3, 1]], np.float32)
    assert list(orc.bbox(p)) == [1, 2, 3, 1]           # coincident: L = 1
    p = np.array([[0, 0, 0, 1], [0.5, 2.0, -1.0, 1]], np.float32)
    assert list(orc.bbox(p)) == [0, 0, -1, 2]          # L = largest extent
    bad = np.array([[0, np.nan, 0, 1]], np.float32)
    with pytest.raises(ValueError):
        orc.bbox(bad)


def test_lattice_keys_distinct(orc):
    p = W.lattice(100)
    k = orc.keys(p, orc.bbox(p), 21)
    assert np.unique(k).size == k.size


def test_sort_is_stable_key_order(orc):
    g = W.rng(5)
    k = g.integers(0, 50, size=5000).astype(np.uint64)
    perm = orc.sort(k)
    assert np.array_equal(perm, np.argsort(k, kind="stable"))


# --------------------------------------------------------------------------
# tree, centre of mass, Barnes-Hut against a second implementation
# --------------------------------------------------------------------------
def _tiny_sets():
    g = W.rng(9)
    sets = []
    for n in (1, 2, 3, 17, 64):
        sets.append(W.uniform_cube(n, seed=100 + n))
    d = W.uniform_cube(40, seed=41)
    d[20:30] = d[5]                                       # exact duplicates
    sets.append(d)
    c = np.zeros((33, 4), np.float32)                     # collinear points
    c[:, 0] = np.linspace(0, 1, 33)
    c[:, 3] = 1.0 / 33
    sets.append(c)
    e = np.tile(np.array([[0.3, 0.3, 0.3, 0.5]], np.float32), (9, 1))
    sets.append(e)                                        # all equal
    cl = np.zeros((48, 4), np.float32)                    # a tight cluster
    cl[:, :3] = 0.5 + g.normal(size=(48, 3)) * 1e-5
    cl[0, :3] = 0.0
    cl[1, :3] = 1.0
    cl[:, 3] = 1.0
    sets.append(cl)
    return sets


@pytest.mark.parametrize("leaf_cap", [1, 3, 8])
def test_tree_equals_brute_enumeration(orc, leaf_cap):
    for p in _tiny_sets():
        o = orc.OracleBH(p, leaf_cap=leaf_cap)
        cells = brute.brute_cells([int(k) for k in o.skeys], 21, leaf_cap)
        t = o.tree
        got = {}
        for c in range(o.nnodes):
            lvl = int(t["level"][c])
            pre = int(o.skeys[t["first"][c]]) >> (3 * (21 - lvl))
            got[(lvl, pre)] = (int(t["first"][c]), int(t["count"][c]))
        assert got == cells
        # breadth-first order with children contiguous and in octant order
        assert np.all(np.diff(t["level"]) >= 0)
        for c in range(o.nnodes):
            if t["child"][c] >= 0:
                ch = np.arange(t["child"][c], t["child"][c] + t["nchild"][c])
                assert t["first"][ch[0]] == t["first"][c]
                assert t["count"][ch].sum() == t["count"][c]
                assert np.all(t["first"][ch[1:]] == t["first"][ch[:-1]] + t["count"][ch[:-1]])
                assert np.all(t["level"][ch] == t["level"][c] + 1)
        # centre of mass per cell, directly
        for c in range(o.nnodes):
            com, m = brute.cell_com(o.spm, int(t["first"][c]), int(t["count"][c]))
            np.testing.assert_allclose(o.com[c, :3], com, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(o.com[c, 3], m, rtol=1e-13)


@pytest.mark.parametrize("theta", [0.0, 0.5, 0.9])
def test_bh_equals_recursive(orc, theta):
    for p in _tiny_sets():
        o = orc.OracleBH(p, theta=theta, G=1.3, eps=1e-2, leaf_cap=2)
        b, terms = o.bh()
        L = float(o.cube[3])
        for i in range(o.n):
            ref, nt = brute.recursive_bh(o.spm, o.skeys, 21, 2, L, theta, 1.3, 1e-2,
                                         o.src[i, :3], self_j=int(o.rank[i]))
            np.testing.assert_allclose(b[i], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
            assert terms[i] == nt


def test_group_walk_equals_recursive_vote(orc):
    """The group (warp-vote) walk: accept a cell only if all group members do."""
    p = W.uniform_cube(64, seed=77)
    o = orc.OracleBH(p, theta=0.6, eps=1e-2, leaf_cap=2)
    out, rows, _ = o.bh_group(group=8, mode=0)
    order = o.target_order()
    L = float(o.cube[3])
    for g0 in range(0, 64, 8):
        members = order[g0:g0 + 8]
        for i in members:
            ref, _ = brute.recursive_bh(o.spm, o.skeys, 21, 2, L, 0.6, 1.0, 1e-2,
                                        o.src[i, :3], self_j=int(o.rank[i]),
                                        group_x=o.src[members, :3])
            r = int(np.nonzero(rows == i)[0][0])
            np.testing.assert_allclose(out[r], ref, rtol=1e-12, atol=1e-14)


def _box_group_case(orc, n, group, theta, seed):
    p = W.uniform_cube(n, seed=seed)
    o = orc.OracleBH(p, theta=theta, eps=1e-2, leaf_cap=2)
    out, rows, _ = o.bh_group(group=group, mode=1)
    return p, o, out, rows, o.target_order()


def _box_group_brute(o, members, i, theta, rule, log=None):
    ref, _ = brute.recursive_bh(o.spm, o.skeys, 21, 2, float(o.cube[3]), theta, 1.0, 1e-2,
                                o.src[i, :3], self_j=int(o.rank[i]),
                                group_x=o.src[members, :3], group_rule=rule, log=log)
    return ref


@pytest.mark.parametrize("n,group,theta,seed", [(64, 8, 0.6, 78), (128, 64, 0.5, 79)])
def test_group_box_rule_equals_recursive_box(orc, n, group, theta, seed):
    """The box opening rule with groups larger than one (so the box is a
    real box, not a point): accept a cell iff w^2/theta^2 < d^2, d the
    distance from its centre of mass to the nearest point of the group's
    bounding box.  Every row equals the recursive restatement with that
    rule; the same inputs under a plausible wrong distance (farthest corner,
    box centre, the clip with lo and hi exchanged) give other results, and
    the walks decide cells whose centre of mass lies inside the box on one
    or two axes and outside on the others, where those rules part."""
    p, o, out, rows, order = _box_group_case(orc, n, group, theta, seed)
    wrong = {"far_corner": 0, "centre": 0, "swapped": 0}
    partial = 0
    for g0 in range(0, n, group):
        members = order[g0:g0 + group]
        lo = o.src[members, :3].astype(np.float64).min(axis=0)
        hi = o.src[members, :3].astype(np.float64).max(axis=0)
        for i in members:
            log = []
            ref = _box_group_brute(o, members, i, theta, "box", log)
            r = int(np.nonzero(rows == i)[0][0])
            np.testing.assert_allclose(out[r], ref, rtol=1e-12, atol=1e-14)
            for lvl, com, ok in log:
                inside = int(((com >= lo) & (com <= hi)).sum())
                if inside in (1, 2):
                    far = (float(o.cube[3]) / 2 ** lvl) ** 2 / theta ** 2 < \
                        brute.box_distance2(com, lo, hi, "far_corner")
                    partial += int(far != ok)
            for rule in wrong:
                bad = _box_group_brute(o, members, i, theta, rule)
                wrong[rule] += int(not np.allclose(out[r], bad, rtol=1e-9, atol=1e-12))
    assert partial > 0
    for rule, nbad in wrong.items():
        assert nbad > 0, rule


def test_box_distance_definition():
    """Hand cases of the distance to a box: inside (0), beside a face, off an
    edge, off a corner, and inside on one axis only."""
    lo, hi = np.array([0.0, 0.0, 0.0]), np.array([1.0, 2.0, 3.0])
    assert brute.box_distance2([0.5, 1.0, 1.5], lo, hi) == 0.0
    assert brute.box_distance2([1.5, 1.0, 1.5], lo, hi) == 0.25
    assert brute.box_distance2([-1.0, 3.0, 1.5], lo, hi) == 2.0
    assert brute.box_distance2([2.0, -2.0, 5.0], lo, hi) == 1.0 + 4.0 + 4.0
    assert brute.box_distance2([0.5, 4.0, -1.0], lo, hi) == 4.0 + 1.0
    assert brute.box_distance2([0.5, 4.0, -1.0], lo, hi, "far_corner") == 0.25 + 16.0 + 16.0


def test_group_of_one_is_per_target(orc):
    p = W.uniform_cube(2000, seed=8)
    o = orc.OracleBH(p, theta=0.5, eps=1e-3, leaf_cap=4)
    b, _ = o.bh()
    for mode in (0, 1):
        out, rows, _ = o.bh_group(group=1, mode=mode)
        np.testing.assert_allclose(out, b[rows], rtol=1e-13, atol=1e-13 * np.abs(b).max())


def test_theta_zero_is_direct(orc):
    p = W.plummer(3000, seed=12)
    for cap in (1, 8):
        o = orc.OracleBH(p, theta=0.0, eps=1e-3, leaf_cap=cap)
        b, terms = o.bh()
        d = o.direct()
        assert np.all(terms == p.shape[0] - 1)
        np.testing.assert_allclose(b, d, rtol=1e-12, atol=1e-12 * np.abs(d).max())


def test_mac_is_strict_and_uses_full_edge(orc):
    """Sources (0,0,0), (1/4,1/4,1/4) and (1,1,1): cube L = 1, the level-1
    cell [0,1/2)^3 holds the first two (leaf at capacity 2), centre of mass
    (1/8,1/8,1/8).  A target at (9/8,1/8,1/8) is at r = 1 exactly.  With the
    full edge w = 1/2 and theta = 1/2, w^2/theta^2 = 1 = r^2: the strict test
    must open the cell (two particle terms).  A half-edge w would accept it."""
    src = np.array([[0, 0, 0, 1], [0.25, 0.25, 0.25, 1], [1, 1, 1, 1]], np.float32)
    tgt = np.array([[1.125, 0.125, 0.125, 0]], np.float32)
    o = orc.OracleBH(src, theta=0.5, eps=0.0, leaf_cap=2)
    b, terms = o.bh(tgt)
    exact = orc.direct(src, tgt, 1.0, 0.0)
    assert terms[0] == 3
    np.testing.assert_allclose(b, exact, rtol=1e-15)
    b2, terms2 = o.bh(tgt, theta=0.5000001)          # just above: accepted
    assert terms2[0] == 2
    mono = orc.direct(np.array([[0.125, 0.125, 0.125, 2], [1, 1, 1, 1]], np.float32),
                      tgt, 1.0, 0.0)
    np.testing.assert_allclose(b2, mono, rtol=1e-15)
    assert abs(b2[0, 0] - b[0, 0]) > 1e-4


def test_rel_error_floor(orc):
    ref = np.array([[1.0, 0, 0], [0, 2.0, 0], [1e-9, 0, 0]])
    a = ref + np.array([[1e-3, 0, 0], [0, 0, 0], [1e-6, 0, 0]])
    e = orc.rel_error(a, ref)
    np.testing.assert_allclose(e, [1e-3, 0.0, 1e-6 / 1e-3])


def test_theta_table_sanity_band(orc):
    """The GASPHiA page's theta table (1M particles) is a loose band only: the
    oracle's mean relative error on the 1M lattice must grow with theta and
    stay within a factor 10 of the printed mean at each theta."""
    rows = np.loadtxt(os.path.join(GOLDEN, "theta_table_gasphia.txt"))
    page = {round(r[0], 1): r for r in rows}
    p = W.lattice(100)
    o = orc.OracleBH(p, eps=5e-3)
    idx = W.error_sample(p.shape[0], 256)
    d = o.direct(idx=idx)
    means = []
    for th in (0.3, 0.5, 0.8):
        b, _ = o.bh(idx=idx, theta=th)
        m = orc.rel_error(b[:, :3], d[:, :3]).mean()
        means.append(m)
        assert page[th][3] / 10 < m < page[th][3] * 10
    assert means[0] < means[1] < means[2]


# --------------------------------------------------------------------------
# time integration
# --------------------------------------------------------------------------
@pytest.mark.parametrize("G", [1.0, 4.0])
def test_leapfrog_circular_binary(orc, G):
    """Two masses 1/2 at distance 1: circular orbit about the centre of mass
    with speed sqrt(G m / (2 d)) = sqrt(G)/2 and period 2*pi*(d/2)/v; after one
    period the leapfrog returns to the start to O(dt^2) and conserves energy
    to O(dt^2)."""
    sp = np.sqrt(G) / 2
    period = 2 * np.pi * 0.5 / sp
    p = np.array([[-0.5, 0, 0, 0.5], [0.5, 0, 0, 0.5]], np.float64)
    v = np.array([[0, -sp, 0], [0, sp, 0]], np.float64)
    nsteps = 2000
    dt = period / nsteps
    pe, ve = orc.leapfrog(p, v, G, 0.0, dt, nsteps)
    np.testing.assert_allclose(pe[:, :3], p[:, :3], atol=2e-5)
    np.testing.assert_allclose(ve, v, atol=2e-5 * sp / 0.5)
    # quarter period: bodies on the y axis
    pq, _ = orc.leapfrog(p, v, G, 0.0, dt, nsteps // 4)
    np.testing.assert_allclose(pq[:, :3], [[0, -0.5, 0], [0, 0.5, 0]], atol=2e-5)
    def energy(pp, vv):
        d = np.linalg.norm(pp[0, :3] - pp[1, :3])
        return 0.5 * (pp[:, 3] * (vv * vv).sum(1)).sum() - G * pp[0, 3] * pp[1, 3] / d
    assert abs(energy(pe, ve) / energy(p, v) - 1.0) < 1e-5


def test_leapfrog_time_reversible_and_conserves_momentum(orc):
    g = W.rng(44)
    n = 64
    p = np.zeros((n, 4))
    p[:, :3] = g.normal(size=(n, 3))
    p[:, 3] = g.uniform(0.5, 1.5, n) / n
    v = g.normal(size=(n, 3)) * 0.1
    p1, v1 = orc.leapfrog(p, v, 1.0, 0.05, 1e-2, 50)
    mom0 = (p[:, 3:4] * v).sum(0)
    mom1 = (p1[:, 3:4] * v1).sum(0)
    assert np.abs(mom1 - mom0).max() < 1e-13
    p2, v2 = orc.leapfrog(p1, -v1, 1.0, 0.05, 1e-2, 50)      # run it backwards
    np.testing.assert_allclose(p2[:, :3], p[:, :3], atol=1e-10)
    np.testing.assert_allclose(-v2, v, atol=1e-10)
