"""Pins for the oracle's stochastic Barnes-Hut estimator and its random
numbers ("Stochastic Barnes-Hut Approximation for Fast Summation on the GPU"
page, section 方法, 关键设计 1-4).

What fixes the estimator independently of its own code:
* Philox4x64-10 equals numpy's Philox bit generator (a separate library
  implementation of the same published generator);
* unbiasedness (the page's theorem 3.1): the mean over many independent
  samples converges to the exact fp64 direct sum, in source/target and in
  self mode -- a wrong path weight, a wrong roulette weight, a sign error in
  the refinement term or a missed stratum all bias it;
* a closed form of the roulette: along a chain of single-child cells seen
  from the far field, the child's ratio is exactly twice the parent's, so each
  step survives with probability exactly 1/2 and the number of surviving
  steps is geometric;
* a deterministic limit: with one particle per leaf and every leaf a stratum
  the refinement terms vanish and the estimate is the exact sum.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W


def test_philox_matches_numpy():
    rng = np.random.default_rng(11)
    cases = [([0, 0, 0, 0], [0, 0]), ([2**64 - 1, 5, 0, 0], [1, 2])]
    for _ in range(6):
        cases.append((rng.integers(0, 2**63, 4, dtype=np.uint64).tolist(),
                      rng.integers(0, 2**63, 2, dtype=np.uint64).tolist()))
    for ctr, key in cases:
        bg = np.random.Philox(key=np.array(key, np.uint64),
                              counter=np.array(ctr, np.uint64))
        # numpy advances the counter (with carry) before each block
        ref = bg.random_raw(4)
        nxt = list(ctr)
        for w in range(4):
            nxt[w] = (nxt[w] + 1) % 2**64
            if nxt[w] != 0:
                break
        np.testing.assert_array_equal(O.philox4x64(nxt, key), ref)


def _mc(o, tgt, n_seed, samples, strata_level, rows=None):
    outs = np.array([o.sbh(tgt, rows=rows, seed=1000 + s, samples=samples,
                           strata_level=strata_level)[0] for s in range(n_seed)])
    return outs.mean(0), outs.std(0, ddof=1) / np.sqrt(n_seed)


@pytest.mark.parametrize("strata_level", [0, 1, 2])
def test_unbiased_source_target(strata_level):
    src = W.uniform_cube(300, 7)
    tgt = W.uniform_cube(5, 9)
    o = O.OracleBH(src, G=1.3, eps=1e-2, leaf_cap=4)
    exact = o.direct(tgt)
    mean, se = _mc(o, tgt, 100, 400, strata_level)
    z = (mean - exact) / se
    assert np.abs(z).max() < 5.0, np.round(z, 2)
    # and the samples are not degenerate (the estimator is random)
    assert se.min() > 0.0


def test_unbiased_self_mode():
    src = W.plummer(400, seed=8)
    o = O.OracleBH(src, G=1.0, eps=2e-2, leaf_cap=8)
    rows = np.array([0, 17, 123, 399])
    exact = o.direct(None, idx=rows)
    mean, se = _mc(o, None, 100, 400, 1, rows=rows)
    z = (mean - exact) / se
    assert np.abs(z).max() < 5.0, np.round(z, 2)


def test_roulette_geometric_on_single_child_chain():
    # a tight cluster far from the query sits below a chain of single-child
    # cells; each chain step refines a cell into one child with the same
    # centre of mass, so the refinement term is exactly zero and the step
    # survives with probability exactly max(1, b) / (2 b) = 1/2 (b >= 1)
    rng = np.random.default_rng(3)
    cl = np.zeros((20, 4), np.float32)
    cl[:, :3] = 0.05 + 1e-5 * rng.random((20, 3), dtype=np.float32)
    cl[:, 3] = 1.0
    far = np.array([[1.0, 1.0, 1.0, 1.0]], np.float32)
    src = np.concatenate([cl, far])
    o = O.OracleBH(src, G=1.0, eps=0.0, leaf_cap=4)
    q = np.array([[1.0, 1.0, 0.9, 0.0]], np.float32)
    # chain length: levels between the cluster's level-1 cell and the level
    # where the cluster first splits
    t = o.tree
    lvl = t["level"]
    split = min(lvl[c] for c in range(o.nnodes) if t["nchild"][c] > 1 and t["count"][c] == 20)
    assert split >= 12
    S = 4000
    out, terms, _ = o.sbh(q, seed=5, strata_level=1, samples=S)
    # 2 strata monopoles; the lone far particle's leaf is near the query
    # (ratios below 1 for the leaf and its particle), so its one step always
    # survives: 2 terms per sample; then 2 terms (child, parent) per
    # surviving chain step; steps at or below the split add more, with
    # probability 2^-(split-1)
    chain_terms = terms[0] - 2 - 2 * S
    expect = S * 2 * (1.0 - 0.5 ** (split - 1))
    sd = 2 * np.sqrt(S * 2.0)
    tail = 40 * S * 0.5 ** (split - 1)      # samples that pass the split
    assert abs(chain_terms - expect) < 6 * sd + tail, (chain_terms, expect, sd, split)


def test_one_particle_leaves_give_the_exact_sum():
    src = W.uniform_cube(200, 21)
    tgt = W.uniform_cube(7, 22)
    o = O.OracleBH(src, G=0.7, eps=1e-3, leaf_cap=1)
    exact = o.direct(tgt)
    for seed in (0, 1):
        out = o.sbh(tgt, seed=seed, strata_level=21)[0]
        np.testing.assert_allclose(out, exact, rtol=1e-12, atol=1e-12)


def test_terms_and_scales_are_consistent():
    src = W.uniform_cube(500, 4)
    tgt = W.uniform_cube(40, 5)
    o = O.OracleBH(src, leaf_cap=16)
    out, terms, sc = o.sbh(tgt, seed=9)
    aa, ap = sc[:, 0], sc[:, 1]
    ns = sum(1 for c in range(o.nnodes)
             if o.tree["level"][c] == 2 or (o.tree["level"][c] < 2 and o.tree["child"][c] < 0))
    assert (terms >= ns).all()
    assert (aa >= np.linalg.norm(out[:, :3], axis=1) * (1 - 1e-12)).all()
    assert (ap >= np.abs(out[:, 3]) * (1 - 1e-12)).all()
    assert (sc[:, 2] > 0).all() and (sc[:, 3] > 0).all()
