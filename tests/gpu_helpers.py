"""Shared helpers for the GPU parity tests (they call the CUDA path through
the C ABI binding and compare with the CPU oracle)."""
from __future__ import annotations

import numpy as np

import oracle as O

# Tolerances (stated with the tests that use them):
#  direct sum vs fp64: median 1e-5, max 1e-4 relative (floored denominator)
#  tree walk vs the oracle's walk with the same opening rule: relative
#  difference <= 1e-5 for all but the targets where an fp32/fp64 opening
#  decision flips (<= FLIP_FRAC of them, each within BH-error size)
DIRECT_MEDIAN, DIRECT_MAX = 1e-5, 1e-4
WALK_TOL = 1e-5
FLIP_FRAC = 0.01
FLIP_MAX = 0.05
DIST_SLACK = 1e-5


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def gpu_bh(src, tgt=None, theta=0.5, G=1.0, eps=1e-3, **opts):
    import barnes_hut_body_gb300 as B
    bh = B.BarnesHut(theta=theta, G=G, eps=eps, **opts)
    out = bh.compute(to_dev(src), None if tgt is None else to_dev(tgt))
    rc = bh.status()
    return bh, out.cpu().numpy().astype(np.float64), rc


def gpu_direct(src, tgt=None, G=1.0, eps=1e-3):
    import barnes_hut_body_gb300 as B
    bh = B.BarnesHut(theta=0.5, G=G, eps=eps)
    out = bh.direct(to_dev(src), None if tgt is None else to_dev(tgt))
    rc = bh.status()
    bh.close()
    return out.cpu().numpy().astype(np.float64), rc


def rel(a, ref):
    """(acceleration error, potential error) per row, floored denominators."""
    return O.rel_error(a[:, :3], ref[:, :3]), O.rel_error(a[:, 3], ref[:, 3])


def assert_direct_close(got, ref):
    ea, ep = rel(got, ref)
    for e in (ea, ep):
        assert np.median(e) <= DIRECT_MEDIAN, np.median(e)
        assert e.max() <= DIRECT_MAX, e.max()


def assert_walk_close(got, ref, label="", mag=None, nterms=None, flip_rows=0):
    """Same opening rule on both sides: equal up to fp32 rounding, except
    targets where an opening decision taken in fp32 vs fp64 flips.

    The acceleration difference is measured against ``mag`` = G * sum of the
    term magnitudes (from the oracle), the natural scale of summation
    rounding -- it matters where many terms cancel, e.g. near a cluster
    centre; the potential's terms share one sign, so its plain relative
    difference is used."""
    ea, ep = rel(got, ref)
    if mag is not None:
        num = np.linalg.norm(got[:, :3] - ref[:, :3], axis=1)
        den = np.maximum(mag, 1e-3 * np.median(mag))
        ea = num / den
    e = np.maximum(ea, ep)
    tol = WALK_TOL
    if nterms is not None:
        # fp32 recursive summation of n terms is exact only to about n*u of
        # sum |term| (u = 2^-24; Higham, "Accuracy and Stability of Numerical
        # Algorithms", section 4.2); long same-sign sums (the potential in a
        # dense, strongly softened cluster) reach that bound
        tol = np.maximum(WALK_TOL, np.asarray(nterms, np.float64) * 2.0 ** -24)
    bad = e > tol
    # flips: a decision taken in fp32 on one side and fp64 on the other
    # changes the terms of a whole group; ``flip_rows`` lets one group flip
    # in sets so small that a group is more than FLIP_FRAC of the rows
    allowed = max(FLIP_FRAC * bad.size, flip_rows)
    assert bad.sum() <= allowed, (label, bad.mean(), np.sort(e)[-5:])
    assert e.max() <= FLIP_MAX, (label, e.max())


def assert_error_no_worse(gpu_vals, orc_vals, direct_ref, label=""):
    """GPU error distribution (median, p99) vs the fp64 direct sum is no worse
    than the per-target oracle walk's, plus DIST_SLACK."""
    g = O.error_stats(O.rel_error(gpu_vals[:, :3], direct_ref[:, :3]))
    o = O.error_stats(O.rel_error(orc_vals[:, :3], direct_ref[:, :3]))
    assert g["median"] <= o["median"] + DIST_SLACK, (label, g, o)
    assert g["p99"] <= o["p99"] + DIST_SLACK, (label, g, o)
    return g, o


def export_state(bh, n):
    import barnes_hut_body_gb300 as B
    keys = B.bh_debug_export(bh.ctx, B.BH_EXPORT_KEYS, n)
    perm = B.bh_debug_export(bh.ctx, B.BH_EXPORT_PERM, n)
    nn = int(B.bh_debug_export(bh.ctx, B.BH_EXPORT_NODE_COUNT)[0])
    nodes = B.bh_debug_export(bh.ctx, B.BH_EXPORT_NODES, nn)
    com = B.bh_debug_export(bh.ctx, B.BH_EXPORT_COM, nn)
    cube = B.bh_debug_export(bh.ctx, B.BH_EXPORT_CUBE)
    return keys, perm, nodes, com, cube


def assert_tree_equal(nodes, tree):
    nn = tree["level"].shape[0]
    assert nodes.shape[0] == nn
    np.testing.assert_array_equal(nodes[:, 0], tree["level"])
    np.testing.assert_array_equal(nodes[:, 1], tree["first"])
    np.testing.assert_array_equal(nodes[:, 2], tree["count"])
    np.testing.assert_array_equal(nodes[:, 3], tree["child"])
    np.testing.assert_array_equal(nodes[:, 4], tree["nchild"])
