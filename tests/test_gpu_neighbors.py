"""GPU parity of the SPH neighbour search ("树结构（基于根据 Burtscher 和
Pingali 的研究）" page, sections 粒子领域搜索 and 树遍历计算; GASPHiA's per-node
maximum smoothing length) against the oracle's brute force.

Both sides take the pair test in fp32 with the same rounded operations, so
the bar is exact: counts equal element by element, every list equal as a set
(the GPU lists come in walk order, the oracle's ascending).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def gpu_nb(pm, h, kappa=2.0, mode=1, lists=True, **opts):
    import torch
    import barnes_hut_body_gb300 as B
    bh = B.BarnesHut(**opts)
    d_pm = H.to_dev(pm)
    d_h = torch.from_numpy(np.ascontiguousarray(h, np.float32)).cuda()
    c, o, l = B.bh_neighbors(bh.ctx, d_pm, d_h, kappa, mode, lists=lists)
    rc = bh.status()
    bh.close()
    c = c.cpu().numpy().astype(np.int64)
    if not lists:
        return rc, c, None, None
    return rc, c, o.cpu().numpy().astype(np.int64), l.cpu().numpy().astype(np.int64)


def _sets():
    lat = W.lattice(20, spacing=0.05, permute_seed=3)
    d = W.uniform_cube(3000, seed=12)
    d[500:700, :3] = d[11, :3]                         # 200 coincident particles
    return {
        "uniform_5000": W.uniform_sph(5000, seed=1, n_ngb=40),
        "plummer_20000": W.sph_plummer(20000, seed=2),
        "lattice_8000_shuffled": (lat, np.full(lat.shape[0], 0.75 * 0.05, np.float32)),
        "dups_3000": (d, np.full(3000, 0.03, np.float32)),
        "ragged_4099": W.uniform_sph(4099, seed=7, n_ngb=20),
    }


SETS = _sets()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("name", list(SETS))
def test_counts_and_lists_exact(name, mode):
    pm, h = SETS[name]
    rc, c, off, lst = gpu_nb(pm, h, 2.0, mode)
    assert rc == 0
    oc, ol = O.neighbors(pm, h, 2.0, mode)
    np.testing.assert_array_equal(c, oc)
    np.testing.assert_array_equal(off[1:], np.cumsum(oc))
    assert off[0] == 0
    for i in range(pm.shape[0]):
        got = np.sort(lst[off[i]:off[i + 1]])
        np.testing.assert_array_equal(got, ol[i])


@pytest.mark.parametrize("leaf_cap,key_bits", [(1, 21), (64, 21), (16, 10)])
def test_tree_options_do_not_change_the_answer(leaf_cap, key_bits):
    pm, h = SETS["plummer_20000"]
    rc, c, _, _ = gpu_nb(pm, h, 2.0, 1, lists=False, leaf_cap=leaf_cap, key_bits=key_bits)
    assert rc == 0
    oc, _ = O.neighbors(pm, h, 2.0, 1, with_lists=False)
    np.testing.assert_array_equal(c, oc)


def test_symmetric_lists_are_symmetric():
    pm, h = SETS["plummer_20000"]
    rc, c, off, lst = gpu_nb(pm, h, 2.0, 1)
    assert rc == 0
    i = np.repeat(np.arange(pm.shape[0]), c)
    fwd = i.astype(np.int64) * pm.shape[0] + lst
    bwd = lst.astype(np.int64) * pm.shape[0] + i
    assert np.array_equal(np.sort(fwd), np.sort(bwd))


def test_edge_cases():
    import torch
    import barnes_hut_body_gb300 as B
    one = np.array([[0.1, 0.2, 0.3, 1.0]], np.float32)
    rc, c, off, lst = gpu_nb(one, np.array([1.0], np.float32))
    assert rc == 0 and c.tolist() == [0] and off.tolist() == [0, 0] and lst.size == 0
    pm, h = SETS["uniform_5000"]
    rc, c, _, _ = gpu_nb(pm, np.zeros_like(h), 2.0, 1, lists=False)
    assert rc == 0 and np.all(c == 0)
    # negative smoothing length: the status word reports it
    bad = h.copy()
    bad[17] = -1.0
    rc, _, _, _ = gpu_nb(pm, bad, 2.0, 1, lists=False)
    assert rc == B.BH_EINVAL
    # a list buffer that is too small: nothing past its end is written and
    # the status word reports the overflow
    bh = B.BarnesHut()
    d_pm, d_h = H.to_dev(pm), torch.from_numpy(h).cuda()
    counts = torch.empty(pm.shape[0], dtype=torch.int32, device="cuda")
    offs = torch.empty(pm.shape[0] + 1, dtype=torch.int64, device="cuda")
    lst = torch.full((101,), -7, dtype=torch.int32, device="cuda")
    L = B.lib()
    st = torch.cuda.current_stream().cuda_stream
    assert L.bh_neighbors(bh.ctx, d_pm.data_ptr(), d_h.data_ptr(), pm.shape[0], 2.0, 1,
                          counts.data_ptr(), offs.data_ptr(), lst.data_ptr(), 100, st) == 0
    assert bh.status() == B.BH_ETREE_OVERFLOW
    assert int(lst[100].item()) == -7
    # bad arguments are refused before any launch
    assert L.bh_neighbors(bh.ctx, d_pm.data_ptr(), d_h.data_ptr(), pm.shape[0], 0.0, 1,
                          counts.data_ptr(), None, None, 0, st) == B.BH_EINVAL
    assert L.bh_neighbors(bh.ctx, d_pm.data_ptr(), d_h.data_ptr(), pm.shape[0], 2.0, 5,
                          counts.data_ptr(), None, None, 0, st) == B.BH_EINVAL
    assert L.bh_neighbors(bh.ctx, d_pm.data_ptr(), d_h.data_ptr(), pm.shape[0], 2.0, 1,
                          counts.data_ptr(), None, lst.data_ptr(), 100, st) == B.BH_EINVAL
    # the context still computes correctly afterwards
    c2, _, _ = B.bh_neighbors(bh.ctx, d_pm, d_h, 2.0, 1, lists=False)
    assert bh.status() == 0
    oc, _ = O.neighbors(pm, h, 2.0, 1, with_lists=False)
    np.testing.assert_array_equal(c2.cpu().numpy(), oc)
    bh.close()


def test_full_size_plummer_2e20_sampled_rows():
    pm, h = W.sph_plummer(1 << 20, seed=4)
    rc, c, off, lst = gpu_nb(pm, h, 2.0, 1)
    assert rc == 0
    rows = W.error_sample(pm.shape[0], 2048, seed=8)
    oc, ol = O.neighbors(pm, h, 2.0, 1, rows=rows)
    np.testing.assert_array_equal(c[rows], oc)
    for r, i in enumerate(rows):
        np.testing.assert_array_equal(np.sort(lst[off[i]:off[i + 1]]), ol[r])
    np.testing.assert_array_equal(off[1:], np.cumsum(c))
