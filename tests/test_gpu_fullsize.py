"""GPU parity at the benchmark's full sizes, in the launch configuration
bench.py times (theta 0.5, vote opening, groups of 64, leaf capacity 16,
63-bit keys): keys, permutation and tree bit-exact against the oracle on the
whole problem; forces on sampled targets (the oracle walks them one by one)
and on sampled groups (the oracle's group walk with the same rule)."""
import functools

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
    # the default group size: 64, or 32 when there are too few targets to
    # fill the GPU with groups of 64 (read back from the number walked)
    import barnes_hut_body_gb300 as B
    _, walked = B.bh_get_counters(bh.ctx)
    gs = 32 if walked == (m + 31) // 32 and m > 32 else 64
    ng = (m + gs - 1) // gs
    gsel = np.sort(W.rng(13).choice(ng, size=min(ngroups_sample, ng), replace=False))
    ref, rows, _, mag = o.bh_group(tgt, group=gs, mode=0, groups=gsel, with_abs=True)
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


@functools.lru_cache(maxsize=2)
def _plummer(log2n):
    return W.plummer(1 << log2n, seed=4)


@pytest.mark.parametrize("theta", [0.3, 0.5, 0.8])
def test_plummer_2e22(theta):
    src = _plummer(22)
    _check_full("plummer2e22", src, None, 1.0, 1e-3, theta, 2048, 64)


@pytest.mark.parametrize("theta", [0.3, 0.5, 0.8])
@pytest.mark.parametrize("log2n", [16, 18, 20])
def test_plummer_sweep(log2n, theta):
    """The Plummer scaling sweep's sizes below 2^22 at every theta."""
    src = _plummer(log2n)
    _check_full(f"plummer2e{log2n}", src, None, 1.0, 1e-3, theta, 2048, 64)


def test_plummer_2e24():
    """The sweep's largest size, 16,777,216 particles (theta 0.5)."""
    src = W.plummer(1 << 24, seed=4)
    _check_full("plummer2e24", src, None, 1.0, 1e-3, 0.5, 1024, 32)


@pytest.mark.parametrize("log2m", [15, 17])
def test_surface_with_grid_targets(log2m):
    """The source/target workload's smaller source counts, 10^6 grid targets."""
    src = W.ellipsoid_surfaces(1 << log2m, seed=2)
    tgt = W.query_grid(src)
    _check_full(f"surface2e{log2m}", src, tgt, 1.0, 1e-4, 0.5, 4096, 128)
