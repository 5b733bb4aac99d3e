"""GPU parity at the benchmark's full sizes, in the launch configuration
bench.py times (theta 0.5, vote opening, groups of 64, leaf capacity 16,
63-bit keys): keys, permutation and tree bit-exact against the oracle on the
whole problem; forces on sampled targets (the oracle walks them one by one)
and on sampled groups (the oracle's group walk with the same rule)."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _check_full(name, src, tgt, G, eps, theta, sample, ngroups_sample=256):
    bh, got, rc = H.gpu_bh(src, tgt, theta=theta, G=G, eps=eps)
    assert rc == 0
    n = src.shape[0]
    keys, perm, nodes, com, cube = H.export_state(bh, n)
    o = O.OracleBH(src, theta=theta, G=G, eps=eps, leaf_cap=16)
    np.testing.assert_array_equal(perm, o.perm)
    np.testing.assert_array_equal(keys, o.skeys)
    H.assert_tree_equal(nodes, o.tree)
    m = n if tgt is None else tgt.shape[0]
    idx = W.error_sample(m, sample)
    direct = o.direct(tgt, idx=idx)
    per_target, _ = o.bh(tgt, idx=idx)
    g, ostats = H.assert_error_no_worse(got[idx], per_target, direct, name)
    ng = (m + 63) // 64
    gsel = np.sort(W.rng(13).choice(ng, size=min(ngroups_sample, ng), replace=False))
    ref, rows, _, mag = o.bh_group(tgt, group=64, mode=0, groups=gsel, with_abs=True)
    H.assert_walk_close(got[rows], ref, name, mag)
    return g, ostats


@pytest.mark.parametrize("shuffled", [False, True])
def test_lattice_1m(shuffled):
    src = W.lattice(100, permute_seed=1 if shuffled else None)
    _check_full("lattice1m", src, None, 1.0, 5e-3, 0.5, 16384)


def test_galaxy_5m():
    src = W.galaxy_pair(5_000_000, seed=3)
    _check_full("galaxy5m", src, None, 1.0, 1e-3, 0.5, 4096, 128)


def test_surface_2e20_with_grid_targets():
    src = W.ellipsoid_surfaces(1 << 20, seed=2)
    tgt = W.query_grid(src)
    _check_full("surface2e20", src, tgt, 1.0, 1e-4, 0.5, 4096, 128)


@pytest.mark.parametrize("theta", [0.3, 0.8])
def test_plummer_2e22(theta):
    src = W.plummer(1 << 22, seed=4)
    _check_full("plummer2e22", src, None, 1.0, 1e-3, theta, 2048, 64)
