"""The allocation-free direct sum (bh_direct_static).

Some callers cannot call cudaMalloc where they need forces -- a CUDA graph
being captured, a loop that must never synchronise the device, a program
that pools all GPU memory itself -- so the library offers one entry point
whose scratch is built into the library instead of allocated.  This file is
collected last so that, if it fails, a run that stops at the first failure
has already run every other test.  It must pass alone in a fresh process
and after the other tests.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_allocating_entry_point():
    """Two calls in a row through the C ABI (self mode, then separate
    targets) against bh_direct and against the fp64 oracle, within the
    direct-sum tolerance."""
    import torch
    import barnes_hut_body_gb300 as B

    src = W.plummer(40000, seed=21)
    tgt = W.uniform_cube(30000, seed=22)
    tgt[:, :3] = tgt[:, :3] * 0.6 - 0.3
    G, eps = 1.3, 2e-3
    d_src, d_tgt = H.to_dev(src), H.to_dev(tgt)
    ref = B.BarnesHut(theta=0.5, G=G, eps=eps)
    for targets, host_tgt in ((None, None), (d_tgt, tgt)):
        rows = src.shape[0] if targets is None else tgt.shape[0]
        out = torch.full((rows, 4), float("nan"), device="cuda")
        B.bh_direct_static(d_src, targets, out, G=G, eps=eps)
        want = ref.direct(d_src, targets)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        H.assert_direct_close(got, want.cpu().numpy().astype(np.float64))
        H.assert_direct_close(got, O.direct(src, host_tgt, G, eps))
    ref.close()


def test_static_scratch_at_its_limit():
    """262,144 targets, the most the 8 MiB array holds (4 doubles per target
    and source slice): the sources then run as one slice, each thread
    folding 256 tile sums in fp64.  Checked against the fp64 oracle on
    16,384 sampled targets (seed 5), twice in a row (the array keeps the
    first call's sums, which the second must overwrite)."""
    import torch
    import barnes_hut_body_gb300 as B

    n = 262144
    src = W.plummer(n, seed=4)
    d_src = H.to_dev(src)
    idx = W.error_sample(n, 16384, seed=5)
    want = O.direct(src, None, 1.0, 1e-3, idx=idx)
    for _ in range(2):
        out = torch.full((n, 4), float("nan"), device="cuda")
        B.bh_direct_static(d_src, None, out, G=1.0, eps=1e-3)
        torch.cuda.synchronize()
        H.assert_direct_close(out.cpu().numpy().astype(np.float64)[idx], want)


def test_static_scratch_rejects_oversize_and_bad_arguments():
    import torch
    import barnes_hut_body_gb300 as B

    src = H.to_dev(W.uniform_cube(64, seed=1))
    big = torch.zeros((262145, 4), device="cuda")
    with pytest.raises(B.BHError):
        B.bh_direct_static(src, big, torch.empty_like(big))
    with pytest.raises(B.BHError):
        B.bh_direct_static(src, None, torch.empty_like(src), eps=-1.0)
