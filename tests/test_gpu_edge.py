"""Edge cases and failure paths of the CUDA path (through the C ABI).

No test here faults or hangs the GPU: the timeout path is exercised by
giving the device waits a zero poll budget, after which the kernels return
and flag BH_ETIMEOUT; non-finite input is flagged by the bounding-box pass.
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import barnes_hut_body_gb300 as mod
    return mod


def test_empty_and_single(B):
    import torch
    bh = B.BarnesHut(theta=0.5, eps=1e-3)
    empty = torch.zeros((0, 4), device="cuda")
    out = bh.compute(empty)
    assert out.shape == (0, 4)
    tgt = H.to_dev(np.ones((5, 4), np.float32))
    out = bh.compute(empty, tgt)
    assert torch.all(out == 0)
    one = H.to_dev(np.array([[0.1, 0.2, 0.3, 2.0]], np.float32))
    out = bh.compute(one)
    assert bh.status() == 0
    assert torch.all(out == 0)


def test_two_bodies_closed_form(B):
    p = np.array([[0.125, -0.25, 0.5, 2.0], [0.5, 0.0, -0.375, 3.0]], np.float32)
    G, eps = 1.75, 0.0625
    _, got, rc = H.gpu_bh(p, theta=0.5, G=G, eps=eps)
    assert rc == 0
    d = p[1, :3].astype(np.float64) - p[0, :3]
    s = d @ d + eps * eps
    np.testing.assert_allclose(got[0, :3], G * 3.0 * d / s ** 1.5, rtol=2e-6)
    np.testing.assert_allclose(got[1, :3], -G * 2.0 * d / s ** 1.5, rtol=2e-6)
    np.testing.assert_allclose(got[:, 3], [-G * 3 / math.sqrt(s), -G * 2 / math.sqrt(s)], rtol=2e-6)


def test_all_points_coincide(B):
    p = np.tile(np.array([[0.3, 0.3, 0.3, 0.25]], np.float32), (100, 1))
    bh, got, rc = H.gpu_bh(p, theta=0.5, eps=0.01)
    assert rc == 0
    cube = B.bh_debug_export(bh.ctx, B.BH_EXPORT_CUBE)
    assert cube[3] == 1.0
    np.testing.assert_allclose(got[:, :3], 0.0, atol=1e-12)
    np.testing.assert_allclose(got[:, 3], -99 * 0.25 / 0.01, rtol=1e-5)


@pytest.mark.parametrize("bad", [np.nan, np.inf])
def test_non_finite_input_is_flagged(B, bad):
    p = W.uniform_cube(1000, seed=3)
    p[17, 1] = bad
    bh, _, rc = H.gpu_bh(p)
    assert rc == B.BH_EINVAL
    # the context stays usable
    _, got, rc = H.gpu_bh(W.uniform_cube(1000, seed=3))
    assert rc == 0 and np.all(np.isfinite(got))


def test_wait_budget_exhaustion_reports_timeout_and_recovers(B):
    """Zero polls: any look-back wait not satisfied at once gives up and sets
    BH_ETIMEOUT; the next call (normal budget) must be exact again."""
    src = W.plummer(1 << 20, seed=4)
    bh = B.BarnesHut(theta=0.5, eps=1e-3)
    B.bh_set_debug(bh.ctx, B.BH_DBG_SPIN_LIMIT, 0)
    dev = H.to_dev(src)
    seen = set()
    for _ in range(5):
        bh.compute(dev)
        seen.add(bh.status())
    assert seen <= {0, B.BH_ETIMEOUT}
    B.bh_set_debug(bh.ctx, B.BH_DBG_SPIN_LIMIT, 1 << 22)
    bh.compute(dev)
    assert bh.status() == 0
    keys = B.bh_debug_export(bh.ctx, B.BH_EXPORT_KEYS, src.shape[0])
    assert np.all(np.diff(keys.astype(np.uint64)) >= 0)


def test_deterministic(B):
    src = W.galaxy_pair(1 << 17, seed=3)
    _, a, _ = H.gpu_bh(src)
    _, b, _ = H.gpu_bh(src)
    np.testing.assert_array_equal(a, b)


def test_unsorted_targets_and_far_targets(B):
    """Targets outside the source cube, in random order."""
    src = W.uniform_cube(3000, seed=9)
    g = W.rng(10)
    tgt = np.zeros((777, 4), np.float32)
    tgt[:, :3] = g.uniform(-2.0, 3.0, size=(777, 3))
    _, got, rc = H.gpu_bh(src, tgt, theta=0.5, eps=1e-3, group=64)
    assert rc == 0
    o = O.OracleBH(src, theta=0.5, eps=1e-3, leaf_cap=16)
    ref, rows, _, mag = o.bh_group(tgt, group=64, mode=0, with_abs=True)
    H.assert_walk_close(got[rows], ref, "far targets", mag)


def test_bad_arguments(B):
    import torch
    bh = B.BarnesHut()
    with pytest.raises(B.BHError):
        B.bh_set_params(bh.ctx, -1.0, 1.0, 0.0)
    with pytest.raises(B.BHError):
        B.bh_set_option(bh.ctx, B.BH_OPT_LEAF_CAP, 0)
    with pytest.raises(ValueError):
        bh.compute(torch.zeros((10, 3), device="cuda"))
    base = torch.zeros(41, device="cuda")
    with pytest.raises(ValueError):       # 4-byte offset: not 16-byte aligned
        bh.compute(base[1:].view(10, 4))


def test_fp32_probe(B):
    """The FMA-chain probe runs, counts its flops from the launch shape, and
    its rate is physical: the scalar form at most the formula peak (SMs x
    128 lanes x 2 flop x 2070 MHz), neither form implausibly slow."""
    import torch
    bh = B.BarnesHut()
    stream = torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    formula = sms * 128 * 2 * 2070e6
    iters = 1 << 14
    for packed in (False, True):
        flops = B.bh_fp32_probe(bh.ctx, packed, iters, stream.cuda_stream)
        assert flops == sms * 2048 * iters * 8 * (2 if packed else 1) * 2
        best = float("inf")
        for _ in range(4):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            B.bh_fp32_probe(bh.ctx, packed, iters, stream.cuda_stream)
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b) / 1e3)
        rate = flops / best
        assert 0.2 * formula < rate < (1.05 if not packed else 2.1) * formula, (packed, rate)
    assert bh.status() == 0
    with pytest.raises(B.BHError):
        B.bh_fp32_probe(bh.ctx, False, 0, stream.cuda_stream)
    with pytest.raises(B.BHError):
        B.bh_fp32_probe(bh.ctx, False, (1 << 24) + 1, stream.cuda_stream)


def test_host_buffers_match_device(B):
    import torch
    src = W.plummer(50000, seed=7)
    bh = B.BarnesHut(theta=0.5, eps=1e-3)
    dev = bh.compute(H.to_dev(src)).cpu().numpy()
    host_in = torch.from_numpy(src).pin_memory()
    host_out = torch.empty((src.shape[0], 4), dtype=torch.float32).pin_memory()
    B.bh_compute_host(bh.ctx, host_in, None, host_out)
    np.testing.assert_array_equal(host_out.numpy(), dev)


def test_stage_times(B):
    src = W.plummer(1 << 18, seed=4)
    bh = B.BarnesHut(theta=0.5, eps=1e-3, timing=1)
    bh.compute(H.to_dev(src))
    t = B.bh_get_stage_times(bh.ctx)
    assert t["traverse"] > 0 and t["sort"] > 0 and t["targets"] == 0.0


def test_graph_replay_is_bit_identical(B):
    """Repeated identical calls are captured once as a CUDA graph and
    replayed; results must equal plain launches, and changing a parameter
    must not replay the old graph."""
    import torch
    src = H.to_dev(W.plummer(200000, seed=31))
    plain = B.BarnesHut(theta=0.5, eps=1e-3, graph=0)
    want = plain.compute(src).clone()
    want_t6 = None
    bh = B.BarnesHut(theta=0.5, eps=1e-3)
    out = torch.empty_like(src)
    for _ in range(4):                       # direct, capture, replay, replay
        out.fill_(float("nan"))
        bh.compute(src, None, out)
        assert bh.status() == 0
        assert torch.equal(out, want)
    bh.set_params(0.6, 1.0, 1e-3)            # new key: no stale replay
    plain.set_params(0.6, 1.0, 1e-3)
    want_t6 = plain.compute(src)
    for _ in range(3):
        bh.compute(src, None, out)
        assert torch.equal(out, want_t6)
    assert not torch.equal(want, want_t6)
