"""Leapfrog time integration on the GPU (bh_leapfrog) against the oracle's
fp64 leapfrog, plus closed-form and consistency checks."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _run(pm, vel, theta, G, eps, dt, nsteps, acc_valid=False, acc=None, bh=None):
    import torch
    import barnes_hut_body_gb300 as B
    bh = bh or B.BarnesHut(theta=theta, G=G, eps=eps)
    d_pm = H.to_dev(pm)
    v4 = np.zeros((pm.shape[0], 4), np.float32)
    v4[:, :3] = vel[:, :3]
    d_v = H.to_dev(v4)
    d_a = H.to_dev(acc) if acc is not None else torch.zeros_like(d_pm)
    B.bh_leapfrog(bh.ctx, d_pm, d_v, d_a, dt, nsteps, acc_valid=acc_valid)
    assert bh.status() == 0
    return (d_pm.cpu().numpy().astype(np.float64), d_v.cpu().numpy().astype(np.float64),
            d_a.cpu().numpy().astype(np.float64), bh)


def test_theta_zero_matches_oracle_leapfrog():
    """theta = 0 opens every cell, so the forces are the brute-force sum; the
    fp32 trajectory must follow the oracle's fp64 one to rounding."""
    g = W.rng(51)
    pm = W.plummer(512, seed=51)
    vel = (g.normal(size=(512, 3)) * 0.3).astype(np.float32)
    G, eps, dt, nsteps = 1.0, 1e-2, 1e-3, 50
    p_gpu, v_gpu, _, _ = _run(pm, vel, 0.0, G, eps, dt, nsteps)
    p_ref, v_ref = O.leapfrog(pm, vel, G, eps, dt, nsteps)
    np.testing.assert_allclose(p_gpu[:, :3], p_ref[:, :3], rtol=0,
                               atol=2e-5 * np.abs(p_ref[:, :3]).max())
    np.testing.assert_allclose(v_gpu[:, :3], v_ref, rtol=0, atol=2e-4 * np.abs(v_ref).max())
    np.testing.assert_array_equal(p_gpu[:, 3], pm[:, 3])        # masses untouched


def test_circular_binary_on_gpu():
    G = 4.0
    sp = np.sqrt(G) / 2
    period = 2 * np.pi * 0.5 / sp
    pm = np.array([[-0.5, 0, 0, 0.5], [0.5, 0, 0, 0.5]], np.float32)
    vel = np.array([[0, -sp, 0], [0, sp, 0]], np.float32)
    p, v, _, _ = _run(pm, vel, 0.5, G, 0.0, period / 2000, 2000)
    np.testing.assert_allclose(p[:, :3], pm[:, :3], atol=5e-4)
    np.testing.assert_allclose(v[:, :3], vel, atol=5e-4 * sp / 0.5)


def test_chained_calls_equal_one_call():
    """Two calls of 5 steps (the second told the accelerations are valid)
    equal one call of 10 steps, bit for bit."""
    pm = W.plummer(20000, seed=52)
    g = W.rng(52)
    vel = (g.normal(size=(20000, 3)) * 0.2).astype(np.float32)
    p10, v10, a10, _ = _run(pm, vel, 0.5, 1.0, 1e-3, 1e-3, 10)
    p5, v5, a5, bh = _run(pm, vel, 0.5, 1.0, 1e-3, 1e-3, 5)
    v5f = v5.astype(np.float32)
    p55, v55, a55, _ = _run(p5.astype(np.float32), v5f, 0.5, 1.0, 1e-3, 1e-3, 5,
                            acc_valid=True, acc=a5.astype(np.float32), bh=bh)
    np.testing.assert_array_equal(p55, p10)
    np.testing.assert_array_equal(v55, v10)
    np.testing.assert_array_equal(a55, a10)


def test_energy_drift_small_with_tree_forces():
    """A Plummer sphere in virial equilibrium-ish (random isotropic speeds)
    advanced 100 steps with theta 0.5: total energy (direct-sum potential,
    evaluated by the oracle) drifts by far less than its size."""
    n = 4096
    pm = W.plummer(n, seed=53)
    g = W.rng(53)
    r = np.linalg.norm(pm[:, :3].astype(np.float64), axis=1)
    vesc = np.sqrt(2.0 / np.sqrt(r * r + 0.01))
    vel = (g.normal(size=(n, 3)) * (0.35 * vesc)[:, None] / np.sqrt(3)).astype(np.float32)
    eps = 1e-2

    def energy(p, v):
        phi = O.direct(p.astype(np.float32), None, 1.0, eps)[:, 3]
        m = p[:, 3].astype(np.float64)
        return 0.5 * (m * (v[:, :3] ** 2).sum(1)).sum() + 0.5 * (m * phi).sum()
    e0 = energy(pm.astype(np.float64), vel.astype(np.float64))
    p, v, _, _ = _run(pm, vel, 0.5, 1.0, eps, 1e-3, 100)
    e1 = energy(p, v)
    assert abs(e1 - e0) < 1e-3 * abs(e0)


def test_tree_force_trajectory_within_force_error_budget():
    """theta = 0.5 against the oracle's fp64 leapfrog with exact forces, 2048
    Plummer particles, 20 steps of 1e-3 (T = 0.02, about half a central
    dynamical time).

    Budget, derived from the force error: a force error |da| <= D applied
    over [0, T] moves a leapfrog trajectory by at most (T^2 / 2) D g and
    changes its velocity by at most T D g, where g = cosh(w T) bounds the
    growth of a deviation under tidal fields of rate w^2.  Here w^2 <= G M /
    a^3 = 1000 (Plummer centre; the softened pair tide G m / eps^3 = 488 is
    smaller), so g <= cosh(0.64) < 1.25; the test uses g = 2.  D is the
    largest Barnes-Hut force error of the GPU's opening rule (the oracle's
    group walk, groups of 32, vote) against the direct sum, taken at the
    first and the last positions of the exact trajectory.  Rounding adds the
    theta = 0 test's allowance."""
    n, G, eps, dt, nsteps, theta = 2048, 1.0, 1e-2, 1e-3, 20, 0.5
    pm = W.plummer(n, seed=54)
    g = W.rng(54)
    r = np.linalg.norm(pm[:, :3].astype(np.float64), axis=1)
    vesc = np.sqrt(2.0 / np.sqrt(r * r + 0.01))
    vel = (g.normal(size=(n, 3)) * (0.35 * vesc)[:, None] / np.sqrt(3)).astype(np.float32)
    p_gpu, v_gpu, _, _ = _run(pm, vel, theta, G, eps, dt, nsteps)
    p_ref, v_ref = O.leapfrog(pm, vel, G, eps, dt, nsteps)

    def force_error(p):
        p32 = np.ascontiguousarray(p, np.float32)
        o = O.OracleBH(p32, theta=theta, G=G, eps=eps, leaf_cap=16)
        bh, rows, _ = o.bh_group(group=32, mode=0)
        exact = O.direct(p32, None, G, eps)[rows]
        return np.linalg.norm(bh[:, :3] - exact[:, :3], axis=1).max()

    T = dt * nsteps
    D = max(force_error(pm), force_error(p_ref))
    growth = 2.0
    dx = np.linalg.norm(p_gpu[:, :3] - p_ref[:, :3], axis=1)
    dv = np.linalg.norm(v_gpu[:, :3] - v_ref[:, :3], axis=1)
    x_tol = 0.5 * T * T * D * growth + 2e-5 * np.abs(p_ref[:, :3]).max()
    v_tol = T * D * growth + 2e-4 * np.abs(v_ref).max()
    assert dx.max() <= x_tol, (dx.max(), x_tol)
    assert dv.max() <= v_tol, (dv.max(), v_tol)
    # the budget is well inside the motion it checks
    moved = np.linalg.norm(p_ref[:, :3] - pm[:, :3].astype(np.float64), axis=1)
    assert x_tol < 0.2 * np.median(moved), (x_tol, np.median(moved))
    np.testing.assert_array_equal(p_gpu[:, 3], pm[:, 3])
