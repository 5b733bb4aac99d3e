"""Randomised parity cases: many small seeded inputs, each with its own size
(ragged tails), distribution, softening, opening angle, leaf capacity, key
width and group size, checked against the oracle through the C ABI.

Bars as in the parity tests: keys, permutation and every tree node
bit-exact; the group walk within max(1e-5, n * 2^-24) of the oracle's group
walk (relative to G * sum |term|, n = terms per target: the fp32 summation
bound, reached by the long same-sign potential sums of dense, strongly
softened clusters) bar fp32/fp64 decision flips (up to one group: grid
inputs put cells exactly on the opening boundary); neighbour counts exact.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

CASES = 24


def _case(k):
    rng = np.random.default_rng(1000 + k)
    n = int(rng.integers(1, 3000))
    kind = k % 4
    if kind == 0:
        src = W.uniform_cube(n, seed=k)
    elif kind == 1:
        src = W.plummer(n, seed=k)
    elif kind == 2:                       # two tight clusters apart
        src = W.uniform_cube(n, seed=k)
        src[:, :3] *= 1e-2
        src[n // 2:, :3] += 0.5
    else:                                 # coarse grid with duplicates
        src = W.uniform_cube(n, seed=k)
        src[:, :3] = np.round(src[:, :3] * 8.0) / 8.0
    theta = float(rng.choice([0.2, 0.5, 0.9]))
    eps = float(rng.choice([0.0, 1e-3, 5e-2]))
    leaf_cap = int(rng.choice([1, 4, 16, 64]))
    key_bits = int(rng.choice([21, 10]))
    group = int(rng.choice([32, 64]))
    return src.astype(np.float32), theta, eps, leaf_cap, key_bits, group


@pytest.mark.parametrize("k", range(CASES))
def test_random_case(k):
    src, theta, eps, leaf_cap, key_bits, group = _case(k)
    label = f"case {k}: n={src.shape[0]} th={theta} eps={eps} B={leaf_cap} bits={key_bits} g={group}"
    bh, got, rc = H.gpu_bh(src, theta=theta, eps=eps, leaf_cap=leaf_cap,
                           key_bits=key_bits, group=group)
    assert rc == 0, label
    bits = 21 if key_bits == 21 else 10
    o = O.OracleBH(src, theta=theta, G=1.0, eps=eps, bits=bits, leaf_cap=leaf_cap)
    keys, perm, nodes, com, cube = H.export_state(bh, src.shape[0])
    np.testing.assert_array_equal(keys, o.skeys, err_msg=label)
    np.testing.assert_array_equal(perm, o.perm, err_msg=label)
    H.assert_tree_equal(nodes, o.tree)
    ref, rows, gterms, mag = o.bh_group(group=group, mode=0, with_abs=True)
    # terms per target of each row's group (every target of a group sees the
    # same list)
    n = src.shape[0]
    sizes = np.minimum(group, n - np.arange(gterms.shape[0]) * group)
    nterms = np.repeat(gterms / sizes, sizes)
    H.assert_walk_close(got[rows], ref, label, mag, nterms, flip_rows=group)
    bh.close()


@pytest.mark.parametrize("k", range(0, CASES, 3))
def test_random_neighbour_case(k):
    import torch
    import barnes_hut_body_gb300 as B
    src, _, _, leaf_cap, key_bits, _ = _case(k)
    rng = np.random.default_rng(2000 + k)
    h = (rng.random(src.shape[0]) * 0.08).astype(np.float32)
    mode = k % 2
    bh = B.BarnesHut(leaf_cap=leaf_cap, key_bits=key_bits)
    c, off, lst = B.bh_neighbors(bh.ctx, H.to_dev(src), torch.from_numpy(h).cuda(), 2.0, mode)
    assert bh.status() == 0
    bh.close()
    oc, ol = O.neighbors(src, h, 2.0, mode)
    c = c.cpu().numpy()
    off = off.cpu().numpy()
    lst = lst.cpu().numpy()
    np.testing.assert_array_equal(c, oc)
    for i in range(src.shape[0]):
        np.testing.assert_array_equal(np.sort(lst[off[i]:off[i + 1]]), ol[i])
