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

import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_allocating_entry_point():
    """Two calls in a row through the C ABI (self mode, then separate
    targets) against bh_direct, within the direct-sum tolerance."""
    import torch
    import barnes_hut_body_gb300 as B

    src = W.plummer(40000, seed=21)
    tgt = W.uniform_cube(30000, seed=22)
    tgt[:, :3] = tgt[:, :3] * 0.6 - 0.3
    G, eps = 1.3, 2e-3
    d_src, d_tgt = H.to_dev(src), H.to_dev(tgt)
    ref = B.BarnesHut(theta=0.5, G=G, eps=eps)
    for targets in (None, d_tgt):
        rows = src.shape[0] if targets is None else tgt.shape[0]
        out = torch.full((rows, 4), float("nan"), device="cuda")
        B.bh_direct_static(d_src, targets, out, G=G, eps=eps)
        want = ref.direct(d_src, targets)
        torch.cuda.synchronize()
        H.assert_direct_close(out.cpu().numpy().astype(np.float64),
                              want.cpu().numpy().astype(np.float64))
    ref.close()


def test_static_scratch_rejects_oversize_and_bad_arguments():
    import torch
    import barnes_hut_body_gb300 as B

    src = H.to_dev(W.uniform_cube(64, seed=1))
    big = torch.zeros((262145, 4), device="cuda")
    with pytest.raises(B.BHError):
        B.bh_direct_static(src, big, torch.empty_like(big))
    with pytest.raises(B.BHError):
        B.bh_direct_static(src, None, torch.empty_like(src), eps=-1.0)
