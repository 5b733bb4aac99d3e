"""GPU parity of the stochastic Barnes-Hut estimator ("Stochastic Barnes-Hut
Approximation for Fast Summation on the GPU" page, section 方法).

The oracle draws the same Philox4x64-10 numbers for the same seed, group,
stratum and sample, and takes the roulette decision in fp32 as the kernel
does, so both follow the same paths and stop at the same steps (the
evaluation counts are compared).  The results then differ by two roundings:
summation (bounded by SBH_TOL times the oracle's sum of |weighted term|) and
the centres of mass, which the GPU sums in fp32 (the page computes in single
precision) and the oracle in fp64.  Unlike the deterministic walk, the
estimator evaluates cells close to the query, where the softened kernel is
steep: a com displacement d moves a weighted cell term by at most
2 |w| m d / s^3 in the acceleration and |w| m r d / s^3 in the potential
(s^2 = r^2 + eps^2).  d is the largest per-axis difference between the
GPU's centres of mass (exported after the call) and the oracle's, itself
checked against the bound of the centre-of-mass parity test,
2u (cmax + 8*22) (L + max|lo|).  A decision whose fp32 inputs differ by such a
rounding can flip; such rows are allowed up to SBH_FLIP_FRAC.

Independently of the oracle, the GPU estimator's Monte Carlo mean over many
seeds must converge to the fp64 direct sum (unbiasedness).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

SBH_TOL = 1e-5          # |gpu - oracle| / sum |weighted term|
SBH_FLIP_FRAC = 0.005   # rows allowed to differ by a flipped fp32 decision


def gpu_sbh(src, tgt=None, G=1.0, eps=1e-3, seed=0, samples=1, strata_level=2,
            leaf_cap=16, bh=None, with_com=False):
    import barnes_hut_body_gb300 as B
    own = bh is None
    if own:
        bh = B.BarnesHut(G=G, eps=eps, leaf_cap=leaf_cap, estimator=B.BH_EST_STOCHASTIC)
    bh.set_option("seed", seed)
    bh.set_option("samples", samples)
    bh.set_option("strata_level", strata_level)
    out = bh.compute(H.to_dev(src), None if tgt is None else H.to_dev(tgt))
    rc = bh.status()
    executed, _ = B.bh_get_counters(bh.ctx)
    res = out.cpu().numpy().astype(np.float64)
    com = None
    if with_com:
        nn = int(B.bh_debug_export(bh.ctx, B.BH_EXPORT_NODE_COUNT)[0])
        com = B.bh_debug_export(bh.ctx, B.BH_EXPORT_COM, nn).astype(np.float64)
    if own:
        bh.close()
    if with_com:
        return res, rc, executed, com
    return res, rc, executed


def com_delta(com_gpu, o, leaf_cap=16):
    """Largest per-axis centre-of-mass difference, GPU (fp32) vs oracle
    (fp64), after checking it against the centre-of-mass parity bound."""
    u = 2.0 ** -24
    cmax = max(leaf_cap, int(o.tree["count"][o.tree["child"] < 0].max()))
    bound = 2 * u * (cmax + 8 * 22) * (float(o.cube[3]) + float(np.abs(o.cube[:3]).max()))
    assert com_gpu.shape[0] == o.nnodes
    d = float(np.abs(com_gpu[:, :3] - o.com[:, :3]).max())
    assert d <= bound, (d, bound)
    return d


def assert_sbh_close(got, ref, sc, d, label=""):
    """sc: the oracle's scales (columns: sum |w t| acc, pot; com sensitivities
    acc, pot); d: the com rounding bound."""
    lim_a = SBH_TOL * sc[:, 0] + 2 * np.sqrt(3.0) * d * sc[:, 2]
    lim_p = SBH_TOL * sc[:, 1] + np.sqrt(3.0) * d * sc[:, 3]
    da = np.linalg.norm(got[:, :3] - ref[:, :3], axis=1) / np.maximum(lim_a, 1e-30)
    dp = np.abs(got[:, 3] - ref[:, 3]) / np.maximum(lim_p, 1e-30)
    e = np.maximum(da, dp)
    bad = e > 1.0
    assert bad.mean() <= SBH_FLIP_FRAC, (label, bad.mean(), np.sort(e)[-5:])
    return e


@pytest.mark.parametrize("strata_level,samples,seed", [(2, 1, 0), (1, 3, 7), (0, 2, 11), (3, 1, 5)])
def test_self_mode_matches_oracle(strata_level, samples, seed):
    src = W.uniform_cube(4096, 0)
    got, rc, executed, com = gpu_sbh(src, eps=1e-3, seed=seed, samples=samples,
                                     strata_level=strata_level, with_com=True)
    assert rc == 0
    o = O.OracleBH(src, G=1.0, eps=1e-3, leaf_cap=16)
    ref, terms, sc = o.sbh(None, seed=seed, samples=samples, strata_level=strata_level)
    assert_sbh_close(got, ref, sc, com_delta(com, o), f"s={strata_level} S={samples}")
    # the same paths: the evaluation counts agree up to flipped decisions
    assert abs(executed - terms.sum()) <= 0.01 * terms.sum(), (executed, terms.sum())


@pytest.mark.parametrize("name", ["surface2e15", "plummer2e16"])
def test_source_target_matches_oracle_on_sampled_rows(name):
    if name == "surface2e15":
        src, tgt, G, eps, _ = W.make(name)
    else:
        src = W.plummer(1 << 16, seed=4)
        tgt = W.uniform_cube(50_001, 8)            # ragged last group
        G, eps = 1.0, 1e-3
    got, rc, _, com = gpu_sbh(src, tgt, G=G, eps=eps, seed=3, with_com=True)
    assert rc == 0
    rows = W.error_sample(tgt.shape[0], 4096, seed=6)
    o = O.OracleBH(src, G=G, eps=eps, leaf_cap=16)
    ref, _, sc = o.sbh(tgt, rows=rows, seed=3)
    assert_sbh_close(got[rows], ref, sc, com_delta(com, o), name)


def test_unbiased_against_direct_sum():
    src = W.plummer(3000, seed=12)
    tgt = W.uniform_cube(64, 13)
    tgt[:, :3] = tgt[:, :3] * 2.0 - 1.0
    exact = O.direct(src, tgt, 1.0, 1e-2)
    import barnes_hut_body_gb300 as B
    bh = B.BarnesHut(G=1.0, eps=1e-2, leaf_cap=16, estimator=B.BH_EST_STOCHASTIC)
    outs = np.array([gpu_sbh(src, tgt, seed=s, samples=32, strata_level=1, bh=bh)[0]
                     for s in range(200)])
    bh.close()
    mean = outs.mean(0)
    se = outs.std(0, ddof=1) / np.sqrt(outs.shape[0])
    z = (mean - exact) / np.maximum(se, 1e-7 * np.abs(exact))
    assert np.abs(z).max() < 5.0, np.round(z, 2)


def test_reproducible_and_seed_dependent():
    import barnes_hut_body_gb300 as B
    src = W.galaxy_pair(1 << 15, seed=3)
    bh = B.BarnesHut(G=1.0, eps=1e-3, estimator=B.BH_EST_STOCHASTIC)
    a = gpu_sbh(src, seed=21, bh=bh)[0]
    b = gpu_sbh(src, seed=21, bh=bh)[0]          # graph replay of the same call
    c = gpu_sbh(src, seed=21, bh=bh)[0]
    d = gpu_sbh(src, seed=22, bh=bh)[0]
    bh.close()
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)
    assert np.mean(np.any(a != d, axis=1)) > 0.5


def test_edge_cases():
    import barnes_hut_body_gb300 as B
    one = np.array([[0.3, 0.4, 0.5, 2.0]], np.float32)
    # one source, self mode: nothing acts on it
    got, rc, _ = gpu_sbh(one, eps=0.0)
    assert rc == 0 and np.all(got == 0.0)
    # one source, separate targets (one of them on the source, eps = 0)
    tgt = np.array([[1.3, 0.4, 0.5, 0.0], [0.3, 0.4, 0.5, 0.0], [0.3, -1.6, 0.5, 0.0]], np.float32)
    got, rc, _ = gpu_sbh(one, tgt, eps=0.0, strata_level=6)
    assert rc == 0
    np.testing.assert_allclose(got[[0, 2]], O.direct(one, tgt[[0, 2]], 1.0, 0.0),
                               rtol=1e-6, atol=1e-7)
    assert np.all(got[1] == 0.0)
    # coincident sources (one leaf at the deepest level)
    dup = np.repeat(np.array([[0.1, 0.2, 0.3, 1.0]], np.float32), 100, axis=0)
    dup = np.concatenate([dup, W.uniform_cube(1000, 2)])
    got, rc, _, com = gpu_sbh(dup, eps=1e-2, seed=4, with_com=True)
    o = O.OracleBH(dup, G=1.0, eps=1e-2, leaf_cap=16)
    ref, _, sc = o.sbh(None, seed=4)
    assert rc == 0
    assert_sbh_close(got, ref, sc, com_delta(com, o), "duplicates")
    # bad option values are refused
    bh = B.BarnesHut()
    for key, val in (("estimator", 2), ("samples", 0), ("samples", 1025),
                     ("strata_level", 7), ("strata_level", -1)):
        with pytest.raises(B.BHError):
            bh.set_option(key, val)
    bh.close()


def test_full_size_surface2e20_sampled_rows():
    src, tgt, G, eps, _ = W.make("surface2e20")
    got, rc, _, com = gpu_sbh(src, tgt, G=G, eps=eps, seed=1, with_com=True)
    assert rc == 0
    rows = W.error_sample(tgt.shape[0], 2048, seed=7)
    o = O.OracleBH(src, G=G, eps=eps, leaf_cap=16)
    ref, _, sc = o.sbh(tgt, rows=rows, seed=1)
    assert_sbh_close(got[rows], ref, sc, com_delta(com, o), "surface2e20")
    # error against the exact potential is the oracle's, row for row
    exact = O.direct(src, tgt, G, eps, idx=rows)
    eg = np.abs(got[rows, 3] - exact[:, 3])
    eo = np.abs(ref[:, 3] - exact[:, 3])
    assert np.mean(eg) <= np.mean(eo) * 1.01 + 1e-6, (np.mean(eg), np.mean(eo))
