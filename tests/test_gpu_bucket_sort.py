"""The sort's bucket path against the oracle.

With 63-bit keys the sort first sorts on the top digit (key bits 55..62: the
octree's first two levels and two bits of the third); when every one of those
256 buckets holds at most 4608 keys, one block per bucket finishes it in
shared memory and writes the rows in key order, and the digit passes and the
gather do nothing.  Otherwise the digit passes run as before.  Either way the
permutation must be the oracle's stable sort (ties by index) bit for bit and
everything after it the same; BH_EXPORT_SORT_PATH says which path ran.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

BUCKET_CAP = 4608


def _with_bucket_of(count, seed=71):
    """50,000 uniform points plus a tight cluster inside one top-digit
    bucket, so that this bucket (the largest) holds exactly `count` keys."""
    base = W.uniform_cube(50000, seed=seed)
    cube = O.bbox(base)
    g = W.rng(seed)
    cluster = np.zeros((count, 4), np.float32)
    cluster[:, :3] = (0.2 + 1e-4 * g.random((count, 3))).astype(np.float32)
    cluster[:, 3] = base[0, 3]
    key = O.keys(cluster[:1], cube, 21)[0]
    top = int(key >> np.uint64(55))
    have = int(((O.keys(base, cube, 21) >> np.uint64(55)) == top).sum())
    src = np.ascontiguousarray(np.concatenate([base, cluster[:count - have]]), np.float32)
    # the points stay inside the uniform points' box, so the cube is unchanged
    tops = (O.keys(src, O.bbox(src), 21) >> np.uint64(55)).astype(np.int64)
    counts = np.bincount(tops, minlength=256)
    assert counts[top] == count and counts.max() == count
    return src


def _check(src, tgt=None, walk=True, **opts):
    import barnes_hut_body_gb300 as B
    bh, got, rc = H.gpu_bh(src, tgt, theta=0.5, eps=1e-3, group=64, **opts)
    assert rc == 0
    path = B.bh_debug_export(bh.ctx, B.BH_EXPORT_SORT_PATH)
    n = src.shape[0]
    keys, perm, nodes, com, cube = H.export_state(bh, n)
    o = O.OracleBH(src, theta=0.5, eps=1e-3, leaf_cap=16)
    np.testing.assert_array_equal(perm, o.perm)
    np.testing.assert_array_equal(keys, o.skeys)
    H.assert_tree_equal(nodes, o.tree)
    from tests.test_gpu_parity import _assert_com_close
    _assert_com_close(com, o)
    if not walk:
        return bh, path, got
    ref, rows, terms, mag = o.bh_group(tgt, group=64, mode=0, with_abs=True)
    # the cluster's targets sum thousands of near-equal softened terms: fp32
    # recursive summation is then good only to about (terms) * 2^-24
    sizes = np.diff(np.append(np.arange(0, rows.size, 64), rows.size))
    H.assert_walk_close(got[rows], ref, "bucket sort", mag, nterms=np.repeat(terms, sizes))
    return bh, path, got


@pytest.mark.parametrize("count,path", [(BUCKET_CAP, 1), (BUCKET_CAP + 1, 0)])
def test_bucket_limit(count, path):
    """Largest bucket at the limit (bucket path) and one key past it (digit
    passes): identical permutation, tree, centres of mass and forces."""
    bh, got_path, _ = _check(_with_bucket_of(count))
    assert int(got_path[0]) == path
    bh.close()


def test_lattice_takes_the_bucket_path():
    """The 1M lattice (its largest top-digit bucket holds 4225 keys)."""
    import barnes_hut_body_gb300 as B
    src = W.lattice(100, permute_seed=1)
    bh, got, rc = H.gpu_bh(src, theta=0.5, eps=5e-3)
    assert rc == 0
    assert int(B.bh_debug_export(bh.ctx, B.BH_EXPORT_SORT_PATH)[0]) == 1
    perm = B.bh_debug_export(bh.ctx, B.BH_EXPORT_PERM, src.shape[0])
    np.testing.assert_array_equal(perm, O.sort(O.keys(src, O.bbox(src), 21)))
    bh.close()


def test_separate_targets_with_63_bit_keys():
    """Targets ordered by 63-bit keys take the same path (which = 1)."""
    import barnes_hut_body_gb300 as B
    src = W.uniform_cube(30000, seed=72)
    tgt = W.uniform_cube(120000, seed=73)
    bh, got, rc = H.gpu_bh(src, tgt, theta=0.5, eps=1e-3, group=64, target_key_bits=21)
    assert rc == 0
    assert [int(x) for x in B.bh_debug_export(bh.ctx, B.BH_EXPORT_SORT_PATH)] == [1, 1]
    tperm = B.bh_debug_export(bh.ctx, B.BH_EXPORT_TARGET_PERM, tgt.shape[0])
    np.testing.assert_array_equal(tperm, O.sort(O.keys(tgt, O.bbox(tgt), 21)))
    o = O.OracleBH(src, theta=0.5, eps=1e-3, leaf_cap=16, target_bits=21)
    ref, rows, _, mag = o.bh_group(tgt, group=64, mode=0, with_abs=True)
    H.assert_walk_close(got[rows], ref, "targets", mag)
    bh.close()


@pytest.mark.parametrize("case,path", [("uniform", 1), ("over", 0)])
def test_repeated_calls_replay_the_same_result(case, path):
    """Identical calls give the same bits whichever path runs (the second
    call captures a graph of the step, later ones replay it, the device
    deciding the path on every replay); the permutation after a replay is
    still the oracle's."""
    import torch
    import barnes_hut_body_gb300 as B
    src = W.uniform_cube(200000, seed=74) if case == "uniform" else _with_bucket_of(BUCKET_CAP + 1)
    d = H.to_dev(src)
    bh = B.BarnesHut(theta=0.5, eps=1e-3)
    buf = torch.empty((src.shape[0], 4), dtype=torch.float32, device=d.device)
    outs = [bh.compute(d, out=buf).clone() for _ in range(4)]
    torch.cuda.synchronize()
    assert bh.status() == 0
    assert int(B.bh_debug_export(bh.ctx, B.BH_EXPORT_SORT_PATH)[0]) == path
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    perm = B.bh_debug_export(bh.ctx, B.BH_EXPORT_PERM, src.shape[0])
    np.testing.assert_array_equal(perm, O.sort(O.keys(src, O.bbox(src), 21)))
    bh.close()


def test_one_context_switching_between_branches():
    """One context alternating between inputs that take the two branches
    (each input repeated, so each is captured and replayed) keeps every
    result equal to a fresh context's."""
    import torch
    import barnes_hut_body_gb300 as B
    a = H.to_dev(W.uniform_cube(200000, seed=75))
    b = H.to_dev(_with_bucket_of(BUCKET_CAP + 1, seed=76))
    ref = {}
    for name, d in (("a", a), ("b", b)):
        fresh = B.BarnesHut(theta=0.5, eps=1e-3)
        ref[name] = fresh.compute(d).clone()
        fresh.close()
    bh = B.BarnesHut(theta=0.5, eps=1e-3)
    bufs = {k: torch.empty_like(v) for k, v in ref.items()}
    for name, d in (("a", a), ("a", a), ("a", a), ("b", b), ("b", b), ("b", b), ("a", a)):
        out = bh.compute(d, out=bufs[name])
        torch.cuda.synchronize()
        assert bh.status() == 0
        assert torch.equal(out, ref[name]), name
    bh.close()


def test_all_points_equal_fall_back():
    """One bucket holding every key: the digit passes run."""
    n = 8000
    src = np.tile(np.array([[0.5, 0.5, 0.5, 1e-3]], np.float32), (n, 1))
    bh, path, got = _check(src, walk=False)
    assert int(path[0]) == 0
    # every pair at distance zero: no force, and the potential is the same
    # n - 1 softened terms for every particle (fp32 sum of n equal terms)
    assert np.all(got[:, :3] == 0)
    ref = O.direct(src, None, 1.0, 1e-3, idx=np.arange(4))
    np.testing.assert_allclose(got[:, 3], ref[0, 3], rtol=n * 2.0 ** -24)
    bh.close()


def test_above_the_bucket_capacity_uses_the_digit_passes():
    """More than 256 * 4608 keys cannot all fit: the digit passes run even
    for uniform points (whose buckets would each hold ~4700 keys)."""
    import barnes_hut_body_gb300 as B
    n = 256 * BUCKET_CAP + 1
    src = W.uniform_cube(n, seed=77)
    bh, _, rc = H.gpu_bh(src, theta=0.5, eps=1e-3)
    assert rc == 0
    assert int(B.bh_debug_export(bh.ctx, B.BH_EXPORT_SORT_PATH)[0]) == 0
    perm = B.bh_debug_export(bh.ctx, B.BH_EXPORT_PERM, n)
    np.testing.assert_array_equal(perm, O.sort(O.keys(src, O.bbox(src), 21)))
    bh.close()


SUB_CAP = 64


def _with_sub_buckets(counts, seed=81, spread=1e-5, identical=False):
    """200,000 uniform points plus, for each c in `counts`, a tight cluster
    inside its own sub-bucket (keys sharing bits 47..62) topped up so that
    the sub-bucket holds exactly c keys; identical=True makes each cluster
    one repeated point (equal keys: ties by index)."""
    base = W.uniform_cube(200000, seed=seed)
    cube = O.bbox(base)
    g = W.rng(seed)
    parts = [base]
    sub = (O.keys(base, cube, 21) >> np.uint64(47)).astype(np.int64)
    have_all = np.bincount(sub, minlength=1 << 16)
    used = []
    for c in counts:
        while True:
            ctr = (0.05 + 0.9 * g.random(3)).astype(np.float32)
            probe = np.zeros((1, 4), np.float32)
            probe[0, :3] = ctr
            s = int(O.keys(probe, cube, 21)[0] >> np.uint64(47))
            if s not in used and have_all[s] < c:
                break
        used.append(s)
        extra = c - int(have_all[s])
        pts = np.zeros((extra, 4), np.float32)
        pts[:, :3] = ctr if identical else (ctr + spread * g.random((extra, 3))).astype(np.float32)
        pts[:, 3] = base[0, 3]
        parts.append(pts)
    src = np.ascontiguousarray(np.concatenate(parts), np.float32)
    # the clusters stay inside the uniform points' box and sub-bucket
    keys = O.keys(src, O.bbox(src), 21)
    got = np.bincount((keys >> np.uint64(47)).astype(np.int64), minlength=1 << 16)
    for s, c in zip(used, counts):
        assert got[s] == c, (got[s], c)
    return src


@pytest.mark.parametrize("counts", [[32], [33], [SUB_CAP], [SUB_CAP + 1],
                                    [2, 17, 31, 32, 33, 47, 63, SUB_CAP]])
def test_sub_bucket_sizes(counts):
    """Sub-buckets sorted by counting (up to 32 keys), by the bitonic
    network (33 to 64) and, past 64, the whole bucket by digit passes:
    the permutation and keys are the oracle's either way."""
    import barnes_hut_body_gb300 as B
    src = _with_sub_buckets(counts)
    bh, _, rc = H.gpu_bh(src, theta=0.5, eps=1e-3)
    assert rc == 0
    assert int(B.bh_debug_export(bh.ctx, B.BH_EXPORT_SORT_PATH)[0]) == 1
    n = src.shape[0]
    keys, perm, nodes, com, cube = H.export_state(bh, n)
    o = O.OracleBH(src, theta=0.5, eps=1e-3, leaf_cap=16)
    np.testing.assert_array_equal(perm, o.perm)
    np.testing.assert_array_equal(keys, o.skeys)
    H.assert_tree_equal(nodes, o.tree)
    bh.close()


@pytest.mark.parametrize("count", [40, SUB_CAP])
def test_sub_bucket_of_equal_keys(count):
    """A sub-bucket of identical points (one key repeated): ties go by index
    through the bitonic network."""
    import barnes_hut_body_gb300 as B
    src = _with_sub_buckets([count], identical=True)
    bh, _, rc = H.gpu_bh(src, theta=0.5, eps=1e-3)
    assert rc == 0
    perm = B.bh_debug_export(bh.ctx, B.BH_EXPORT_PERM, src.shape[0])
    np.testing.assert_array_equal(perm, O.sort(O.keys(src, O.bbox(src), 21)))
    bh.close()
