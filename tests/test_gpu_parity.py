"""GPU parity at sizes the oracle finishes in seconds (several tiles + a
ragged tail): every stage of the CUDA path against the CPU oracle.

Bit-exact: Morton keys, the sort permutation, every tree node (level, first,
count, first child, child count).  Tolerance: centre of mass (fp32 sums vs
fp64), direct sum (1e-5 median / 1e-4 max relative), tree walk (equal to the
oracle's walk with the same opening rule up to fp32 rounding, bar decision
flips), error distribution vs the fp64 direct sum (no worse than the oracle's
per-target walk + 1e-5).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _sets():
    d = W.uniform_cube(5000, seed=41)
    d[1000:1300] = d[7]                           # a block of exact duplicates
    return {
        "uniform4096": W.uniform_cube(4096, 0),
        "plummer_2e15": W.plummer(1 << 15, seed=4),
        "galaxy_2e16": W.galaxy_pair(1 << 16, seed=3),
        "lattice_27k_shuffled": W.lattice(30, spacing=1.0 / 30, permute_seed=1),
        "dups_5000": d,
        "ragged_12345": W.uniform_cube(12345, seed=5),
    }


SETS = _sets()


@pytest.mark.parametrize("name", list(SETS))
@pytest.mark.parametrize("bits", [21, 10])
def test_keys_and_permutation_bit_exact(name, bits):
    src = SETS[name]
    bh, _, rc = H.gpu_bh(src, key_bits=bits)
    assert rc == 0
    keys, perm, _, _, cube = H.export_state(bh, src.shape[0])
    o = O.OracleBH(src, bits=bits, leaf_cap=16)
    np.testing.assert_array_equal(cube, o.cube)
    np.testing.assert_array_equal(perm, o.perm)
    np.testing.assert_array_equal(keys, o.skeys)


def _dup_points(n, seed):
    d = W.uniform_cube(n, seed=seed)
    d[n // 2:] = d[: n - n // 2]                  # every point twice (ties by index)
    return d


@pytest.mark.parametrize("n", [2, 3, 33, 1000, 4095, 4096, 4097, 8191])
@pytest.mark.parametrize("bits", [21, 10])
def test_permutation_bit_exact_around_the_one_block_sort(n, bits):
    # up to 4096 keys the sort runs in one block (all digit passes in shared
    # memory); above, one kernel per digit pass: both give the stable sort
    src = _dup_points(n, seed=n)
    bh, _, rc = H.gpu_bh(src, key_bits=bits)
    assert rc == 0
    keys, perm, _, _, cube = H.export_state(bh, n)
    o = O.OracleBH(src, bits=bits, leaf_cap=16)
    np.testing.assert_array_equal(cube, o.cube)
    np.testing.assert_array_equal(perm, o.perm)
    np.testing.assert_array_equal(keys, o.skeys)
    bh.close()


@pytest.mark.parametrize("tbits", [10, 21])
@pytest.mark.parametrize("m", [7, 4096, 4097])
def test_target_permutation_around_the_one_block_sort(m, tbits):
    import barnes_hut_body_gb300 as B
    src = SETS["uniform4096"]
    tgt = _dup_points(m, seed=m + 1)
    bh, _, rc = H.gpu_bh(src, tgt, target_key_bits=tbits)
    assert rc == 0
    ref = O.sort(O.keys(tgt, O.bbox(tgt), tbits))
    np.testing.assert_array_equal(B.bh_debug_export(bh.ctx, B.BH_EXPORT_TARGET_PERM, m), ref)
    bh.close()


@pytest.mark.parametrize("name", ["uniform4096", "plummer_2e15", "galaxy_2e16",
                                  "dups_5000", "ragged_12345"])
@pytest.mark.parametrize("leaf_cap", [1, 8, 16, 64])
def test_tree_bit_exact_and_com(name, leaf_cap):
    src = SETS[name]
    bh, _, rc = H.gpu_bh(src, leaf_cap=leaf_cap)
    assert rc == 0
    keys, perm, nodes, com, cube = H.export_state(bh, src.shape[0])
    o = O.OracleBH(src, leaf_cap=leaf_cap)
    H.assert_tree_equal(nodes, o.tree)
    # parent links: every non-root node is listed among its parent's children
    par = nodes[1:, 5]
    idx = np.arange(1, nodes.shape[0])
    assert np.all(nodes[par, 3] <= idx) and np.all(idx < nodes[par, 3] + nodes[par, 4])
    _assert_com_close(com, o)


def _assert_com_close(com, o):
    """Centre of mass against the fp64 oracle.  The GPU sums each cell's
    mass and mass moments m (x - lo) exactly (64-bit fixed point, prefix
    differences), from d = x - lo rounded once in fp32 (error <= u L, u =
    2^-24, L the cube side); the two sums are each rounded once to fp32, their
    quotient once (<= 3u of com - lo <= L), and adding lo once more (<= u
    |com|).  So |com - exact| <= u (5 L + |lo|) and the mass is within u
    (relative), fixed-point quantisation being ~1e-10 smaller at these mass
    ratios; the tolerances are 6u and 2u."""
    u = 2.0 ** -24
    scale = float(o.cube[3]) + float(np.abs(o.cube[:3]).max())
    np.testing.assert_allclose(com[:, :3], o.com[:, :3], rtol=0, atol=6 * u * scale)
    np.testing.assert_allclose(com[:, 3], o.com[:, 3], rtol=2 * u)


@pytest.mark.parametrize("leaf_cap", [1, 16])
def test_com_spread_masses_and_massless_cells(leaf_cap):
    """Masses log-uniform over six decades, and a tight cluster of massless
    particles far from the rest (its cells take their geometric centres)."""
    rng = W.rng(61)
    src = W.plummer(20000, seed=61)
    src[:, 3] = (10.0 ** rng.uniform(-6, 0, size=20000)).astype(np.float32)
    src[-300:, :3] = (1.5 + 1e-3 * rng.random((300, 3))).astype(np.float32)
    src[-300:, 3] = 0.0
    bh, _, rc = H.gpu_bh(src, leaf_cap=leaf_cap)
    assert rc == 0
    keys, perm, nodes, com, cube = H.export_state(bh, src.shape[0])
    o = O.OracleBH(src, leaf_cap=leaf_cap)
    H.assert_tree_equal(nodes, o.tree)
    assert (o.com[:, 3] == 0).sum() > 0          # some cells hold no mass
    _assert_com_close(com, o)
    bh.close()


@pytest.mark.parametrize("name", ["uniform4096", "plummer_2e15", "galaxy_2e16", "ragged_12345"])
def test_direct_sum(name):
    src = SETS[name]
    got, rc = H.gpu_direct(src, eps=1e-3)
    assert rc == 0
    idx = W.error_sample(src.shape[0], 4096)
    ref = O.direct(src, None, 1.0, 1e-3, idx=idx)
    H.assert_direct_close(got[idx], ref)


def test_direct_source_target():
    src = W.ellipsoid_surfaces(1 << 15, seed=2)
    tgt = W.query_grid(src, side=20)
    got, rc = H.gpu_direct(src, tgt, G=1.0, eps=1e-4)
    assert rc == 0
    ref = O.direct(src, tgt, 1.0, 1e-4)
    H.assert_direct_close(got, ref)


@pytest.mark.parametrize("name", ["uniform4096", "plummer_2e15", "galaxy_2e16", "ragged_12345"])
@pytest.mark.parametrize("theta", [0.3, 0.5, 0.8])
@pytest.mark.parametrize("group,opening,pipeline", [(64, 0, 0), (32, 0, 0), (64, 1, 0),
                                                    (64, 0, 1)])
def test_walk_matches_oracle_group_walk(name, theta, group, opening, pipeline):
    src = SETS[name]
    G, eps = 1.0, 1e-3
    bh, got, rc = H.gpu_bh(src, theta=theta, G=G, eps=eps, group=group, opening=opening,
                           pipeline=pipeline)
    assert rc == 0
    o = O.OracleBH(src, theta=theta, G=G, eps=eps, leaf_cap=16)
    ref, rows, _, mag = o.bh_group(group=group, mode=opening, with_abs=True)
    H.assert_walk_close(got[rows], ref, f"{name} th={theta} g={group} m={opening}", mag)
    idx = W.error_sample(src.shape[0], 2048)
    direct = o.direct(idx=idx)
    per_target, _ = o.bh(idx=idx)
    H.assert_error_no_worse(got[idx], per_target, direct, name)
    ex, ng = __import__("barnes_hut_body_gb300").bh_get_counters(bh.ctx)
    assert ng == (src.shape[0] + group - 1) // group and ex > 0


@pytest.mark.parametrize("name", ["uniform4096", "galaxy_2e16", "dups_5000", "ragged_12345"])
@pytest.mark.parametrize("opening", [0, 1])
def test_pipelined_walk_is_the_fused_walk_bit_for_bit(name, opening):
    # same list order, same pairing, same arithmetic: identical results
    src = SETS[name]
    bh0, a, rc0 = H.gpu_bh(src, theta=0.5, eps=1e-3, opening=opening, pipeline=0, group=64)
    bh1, b, rc1 = H.gpu_bh(src, theta=0.5, eps=1e-3, opening=opening, pipeline=1, group=64)
    assert rc0 == 0 and rc1 == 0
    np.testing.assert_array_equal(a, b)
    import barnes_hut_body_gb300 as B
    assert B.bh_get_counters(bh0.ctx) == B.bh_get_counters(bh1.ctx)
    tgt = W.query_grid(src, side=17)
    _, a, rc0 = H.gpu_bh(src, tgt, theta=0.5, eps=0.0, opening=opening, pipeline=0, group=64)
    _, b, rc1 = H.gpu_bh(src, tgt, theta=0.5, eps=0.0, opening=opening, pipeline=1, group=64)
    assert rc0 == 0 and rc1 == 0
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("name", ["uniform4096", "plummer_2e15", "ragged_12345"])
def test_automatic_group_size(name):
    # with the default group option, targets that fill fewer groups of 64
    # than the walk has warps (16 per SM) are walked in groups of 32: the
    # vote over 32 targets, exactly the oracle's group walk of 32
    import barnes_hut_body_gb300 as B
    import torch
    src = SETS[name]
    n = src.shape[0]
    bh, got, rc = H.gpu_bh(src, theta=0.5, eps=1e-3)
    assert rc == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    group = 32 if (n + 63) // 64 < 16 * sms else 64
    assert B.bh_get_counters(bh.ctx)[1] == (n + group - 1) // group
    o = O.OracleBH(src, theta=0.5, eps=1e-3, leaf_cap=16)
    ref, rows, _, mag = o.bh_group(group=group, mode=0, with_abs=True)
    H.assert_walk_close(got[rows], ref, f"{name} auto group {group}", mag)
    bh.close()


def test_theta_zero_is_the_direct_sum():
    src = SETS["plummer_2e15"]
    _, got, rc = H.gpu_bh(src, theta=0.0, eps=1e-3)
    assert rc == 0
    idx = W.error_sample(src.shape[0], 4096)
    H.assert_direct_close(got[idx], O.direct(src, None, 1.0, 1e-3, idx=idx))


@pytest.mark.parametrize("opening,tbits", [(0, 10), (1, 10), (0, 21)])
def test_source_target_walk(opening, tbits):
    src = W.ellipsoid_surfaces(1 << 15, seed=2)
    tgt = W.query_grid(src, side=30)
    # a shuffled grid: the target order then comes from the keys alone
    tgt = np.ascontiguousarray(tgt[np.random.default_rng(9).permutation(tgt.shape[0])])
    bh, got, rc = H.gpu_bh(src, tgt, theta=0.5, G=1.0, eps=1e-4, opening=opening, group=64,
                           target_key_bits=tbits)
    assert rc == 0
    import barnes_hut_body_gb300 as B
    tperm = B.bh_debug_export(bh.ctx, B.BH_EXPORT_TARGET_PERM, tgt.shape[0])
    o = O.OracleBH(src, theta=0.5, G=1.0, eps=1e-4, leaf_cap=16, target_bits=tbits)
    np.testing.assert_array_equal(tperm, o.target_order(tgt))
    ref, rows, _, mag = o.bh_group(tgt, group=64, mode=opening, with_abs=True)
    H.assert_walk_close(got[rows], ref, "surface", mag)
    direct = o.direct(tgt)
    per_target, _ = o.bh(tgt)
    H.assert_error_no_worse(got, per_target, direct, "surface")


def test_eps_zero():
    src = W.uniform_cube(4096, seed=12)
    _, got, rc = H.gpu_bh(src, theta=0.5, eps=0.0, group=64)
    assert rc == 0
    o = O.OracleBH(src, theta=0.5, eps=0.0, leaf_cap=16)
    ref, rows, _, mag = o.bh_group(group=64, mode=0, with_abs=True)
    H.assert_walk_close(got[rows], ref, "eps0", mag)
    dgot, rc = H.gpu_direct(src, eps=0.0)
    assert rc == 0
    H.assert_direct_close(dgot, O.direct(src, None, 1.0, 0.0))


@pytest.mark.parametrize("leaf_cap", [1, 64])
def test_walk_other_leaf_caps(leaf_cap):
    src = SETS["plummer_2e15"]
    _, got, rc = H.gpu_bh(src, theta=0.5, leaf_cap=leaf_cap, group=64)
    assert rc == 0
    o = O.OracleBH(src, theta=0.5, leaf_cap=leaf_cap)
    ref, rows, _, mag = o.bh_group(group=64, mode=0, with_abs=True)
    H.assert_walk_close(got[rows], ref, f"B={leaf_cap}", mag)


def test_gravity_constant_and_thirty_bit_keys():
    src = SETS["uniform4096"]
    _, got, rc = H.gpu_bh(src, theta=0.6, G=2.5, eps=2e-3, key_bits=10, group=64)
    assert rc == 0
    o = O.OracleBH(src, theta=0.6, G=2.5, eps=2e-3, bits=10, leaf_cap=16)
    ref, rows, _, mag = o.bh_group(group=64, mode=0, with_abs=True)
    H.assert_walk_close(got[rows], ref, "G=2.5 bits=10", mag)


@pytest.mark.parametrize("name", ["uniform4096", "plummer_2e15", "galaxy_2e16"])
def test_interaction_count_matches_oracle_terms(name):
    """bh_count_interactions = the oracle's per-target term count (same tree,
    same theta); an fp32/fp64 opening decision may flip for a few targets."""
    import torch
    import barnes_hut_body_gb300 as B
    src = SETS[name]
    bh, _, rc = H.gpu_bh(src, theta=0.5, eps=1e-3)
    assert rc == 0
    counts = torch.zeros(src.shape[0], dtype=torch.int32, device="cuda")
    total = B.bh_count_interactions(bh.ctx, counts)
    o = O.OracleBH(src, theta=0.5, eps=1e-3, leaf_cap=16)
    _, terms = o.bh()
    c = counts.cpu().numpy().astype(np.int64)
    assert total == c.sum()
    assert (c != terms).mean() <= 0.01
    assert abs(int(c.sum()) - int(terms.sum())) <= 1e-3 * terms.sum()
