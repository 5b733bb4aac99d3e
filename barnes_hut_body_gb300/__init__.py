"""Python binding of libbh.so, the GB300 Barnes-Hut gravity library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/bh.h``.  The functions keep the
C names (``bh_create``, ``bh_set_params``, ``bh_compute``, ...); ``BarnesHut``
is a small convenience wrapper over one context.

Device buffers are torch CUDA tensors of shape (n, 4), float32, contiguous:
rows (x, y, z, m) in, rows (ax, ay, az, phi) out.  PyTorch only supplies the
memory and the stream; there is no CPU or PyTorch fallback -- importing
works without the library, but the first call raises if ``libbh.so`` has
not been built (``python -m barnes_hut_body_gb300.build``).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbh.so")

BH_OK, BH_EINVAL, BH_ENOMEM, BH_ECUDA, BH_ETIMEOUT, BH_ETREE_OVERFLOW = range(6)
BH_OPT_KEY_BITS, BH_OPT_LEAF_CAP, BH_OPT_OPENING, BH_OPT_TIMING, BH_OPT_GROUP, BH_OPT_GRAPH = 1, 2, 3, 4, 5, 6
BH_OPT_ESTIMATOR, BH_OPT_SEED, BH_OPT_SAMPLES, BH_OPT_STRATA_LEVEL = 7, 8, 9, 10
BH_OPT_PIPELINE = 11
BH_OPT_ORDER = 12
BH_OPT_SHARDS, BH_OPT_SHARD = 13, 14
BH_OPT_SCHEDULE = 15
BH_OPT_TARGET_KEY_BITS = 16
BH_ORDER_RADIX, BH_ORDER_TREE = 0, 1
BH_EST_BARNES_HUT, BH_EST_STOCHASTIC = 0, 1
BH_OPEN_VOTE, BH_OPEN_BOX = 0, 1
BH_DBG_SPIN_LIMIT = 1
BH_LF_ACC_VALID = 1
(BH_EXPORT_CUBE, BH_EXPORT_KEYS, BH_EXPORT_PERM, BH_EXPORT_NODE_COUNT,
 BH_EXPORT_NODES, BH_EXPORT_COM, BH_EXPORT_TARGET_PERM, BH_EXPORT_WALK_STATS,
 BH_EXPORT_GROUP_COST, BH_EXPORT_GROUP_ORDER, BH_EXPORT_SORT_PATH) = range(1, 12)
STAGES = ("bbox", "keys", "sort", "reorder", "build", "com", "targets", "traverse")

EXPORTED = ("bh_create", "bh_destroy", "bh_set_params", "bh_set_option",
            "bh_set_debug", "bh_compute", "bh_compute_host", "bh_direct",
            "bh_sync_status", "bh_get_stage_times", "bh_get_counters",
            "bh_debug_export", "bh_count_interactions", "bh_direct_static",
            "bh_leapfrog", "bh_neighbors", "bh_fp32_probe", "bh_last_error")

_lib = None


class BHError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"bh error {code}: {msg}")
        self.code = code


def lib():
    """Load libbh.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m barnes_hut_body_gb300.build` (there is no fallback)")
        L = C.CDLL(LIB_PATH)
        vp, sz, i, f = C.c_void_p, C.c_size_t, C.c_int, C.c_float
        L.bh_create.argtypes = [C.POINTER(vp), i, sz, sz]
        L.bh_destroy.argtypes = [vp]
        L.bh_set_params.argtypes = [vp, f, f, f]
        L.bh_set_option.argtypes = [vp, i, C.c_longlong]
        L.bh_set_debug.argtypes = [vp, i, C.c_longlong]
        for name in ("bh_compute", "bh_compute_host", "bh_direct"):
            getattr(L, name).argtypes = [vp, vp, sz, vp, sz, vp, vp]
        L.bh_sync_status.argtypes = [vp, vp]
        L.bh_get_stage_times.argtypes = [vp, C.POINTER(f), i]
        L.bh_get_counters.argtypes = [vp, C.POINTER(C.c_ulonglong), C.POINTER(C.c_ulonglong)]
        L.bh_debug_export.argtypes = [vp, i, vp, sz]
        L.bh_count_interactions.argtypes = [vp, vp, C.POINTER(C.c_ulonglong), vp]
        L.bh_direct_static.argtypes = [vp, sz, vp, sz, f, f, vp, vp]
        L.bh_leapfrog.argtypes = [vp, vp, vp, sz, vp, f, i, i, vp]
        L.bh_neighbors.argtypes = [vp, vp, vp, sz, f, i, vp, vp, vp, sz, vp]
        L.bh_fp32_probe.argtypes = [vp, i, i, C.POINTER(C.c_double), vp]
        L.bh_last_error.argtypes = [vp]
        L.bh_last_error.restype = C.c_char_p
        for name in EXPORTED:
            if name != "bh_last_error":
                getattr(L, name).restype = i
        _lib = L
    return _lib


def _check(ctx, rc: int) -> int:
    if rc != BH_OK:
        msg = lib().bh_last_error(ctx).decode() if ctx else ""
        raise BHError(rc, msg)
    return rc


def _rows_ptr(t, name: str):
    """Validate a (n,4) float32 contiguous CUDA tensor; return (ptr, rows)."""
    if t is None:
        return None, 0
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != torch.float32 or t.dim() != 2 or t.shape[1] != 4:
        raise ValueError(f"{name} must be float32 of shape (n, 4)")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.data_ptr() % 16:
        raise ValueError(f"{name} must be 16-byte aligned")
    return C.c_void_p(t.data_ptr()), t.shape[0]


def _stream(t, stream):
    if stream is not None:
        return C.c_void_p(stream)
    import torch
    return C.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


# ---- the C ABI, one function each ------------------------------------------
def bh_create(device: int = 0, max_sources: int = 0, max_targets: int = 0):
    h = C.c_void_p()
    rc = lib().bh_create(C.byref(h), int(device), int(max_sources), int(max_targets))
    if rc != BH_OK:
        raise BHError(rc, "bh_create failed")
    return h


def bh_destroy(ctx) -> None:
    lib().bh_destroy(ctx)


def bh_set_params(ctx, theta: float, G: float, eps: float) -> None:
    _check(ctx, lib().bh_set_params(ctx, float(theta), float(G), float(eps)))


def bh_set_option(ctx, key: int, value: int) -> None:
    _check(ctx, lib().bh_set_option(ctx, int(key), int(value)))


def bh_set_debug(ctx, key: int, value: int) -> None:
    _check(ctx, lib().bh_set_debug(ctx, int(key), int(value)))


def bh_compute(ctx, pos_mass, targets, acc_pot, stream=None) -> None:
    """Barnes-Hut on device tensors; targets None = self-gravity."""
    p, n = _rows_ptr(pos_mass, "pos_mass")
    t, m = _rows_ptr(targets, "targets")
    o, k = _rows_ptr(acc_pot, "acc_pot")
    if k != (n if targets is None else m):
        raise ValueError("acc_pot has the wrong number of rows")
    _check(ctx, lib().bh_compute(ctx, p, n, t, m, o, _stream(pos_mass, stream)))


def bh_direct(ctx, pos_mass, targets, acc_pot, stream=None) -> None:
    """Brute-force double loop on device tensors."""
    p, n = _rows_ptr(pos_mass, "pos_mass")
    t, m = _rows_ptr(targets, "targets")
    o, k = _rows_ptr(acc_pot, "acc_pot")
    if k != (n if targets is None else m):
        raise ValueError("acc_pot has the wrong number of rows")
    _check(ctx, lib().bh_direct(ctx, p, n, t, m, o, _stream(pos_mass, stream)))


def bh_direct_static(pos_mass, targets, acc_pot, G: float = 1.0, eps: float = 0.0,
                     stream=None) -> None:
    """Brute-force sum with no device allocation and no context.

    For callers that cannot allocate GPU memory where they need forces (a
    CUDA graph being captured, a loop that must not synchronise the device,
    a program that pools all GPU memory itself).  Scratch is an 8 MiB array
    built into the library: at most 262,144 targets per call, and calls that
    overlap on the GPU race.  The first call on a device should come before
    any stream capture.
    """
    import torch
    p, n = _rows_ptr(pos_mass, "pos_mass")
    t, m = _rows_ptr(targets, "targets")
    o, k = _rows_ptr(acc_pot, "acc_pot")
    if k != (n if targets is None else m):
        raise ValueError("acc_pot has the wrong number of rows")
    dev = pos_mass.device
    if acc_pot.device != dev or (targets is not None and targets.device != dev):
        raise ValueError("pos_mass, targets and acc_pot must be on one device")
    # the library finds its scratch array on the current device
    with torch.cuda.device(dev):
        rc = lib().bh_direct_static(p, n, t, m, float(G), float(eps), o,
                                    _stream(pos_mass, stream))
    if rc != BH_OK:
        raise BHError(rc, "bh_direct_static failed (bad argument, more than "
                          "262144 targets, or a CUDA error)")


def bh_fp32_probe(ctx, packed: bool, iters: int, stream) -> float:
    """Enqueue one launch of the fp32 FMA-chain probe on `stream` (a
    cudaStream_t as int); returns the fp32 flops that launch performs."""
    fl = C.c_double(0.0)
    _check(ctx, lib().bh_fp32_probe(ctx, 1 if packed else 0, int(iters), C.byref(fl),
                                    C.c_void_p(stream)))
    return fl.value


def bh_leapfrog(ctx, pos_mass, vel, acc_pot, dt: float, nsteps: int,
                acc_valid: bool = False, stream=None) -> None:
    """Kick-drift-kick time stepping with the Barnes-Hut forces, in place on
    device tensors (n, 4): positions+masses, velocities, accelerations."""
    p, n = _rows_ptr(pos_mass, "pos_mass")
    v, nv = _rows_ptr(vel, "vel")
    a, na = _rows_ptr(acc_pot, "acc_pot")
    if not (n == nv == na):
        raise ValueError("pos_mass, vel and acc_pot need the same number of rows")
    flags = BH_LF_ACC_VALID if acc_valid else 0
    _check(ctx, lib().bh_leapfrog(ctx, p, v, n, a, float(dt), int(nsteps), flags,
                                  _stream(pos_mass, stream)))


BH_NB_GATHER, BH_NB_SYMMETRIC = 0, 1


def bh_neighbors(ctx, pos_mass, h, kappa: float = 2.0, mode: int = BH_NB_SYMMETRIC,
                 lists: bool = True, stream=None):
    """SPH neighbour search on device tensors: pos_mass (n, 4) and h (n,)
    float32.  Returns (counts uint32 (n,), offsets uint64 (n+1,), list
    uint32 (total,)) as CUDA tensors; with ``lists`` False only counts (the
    other two None).  Sizing the list synchronises the stream once."""
    import torch
    p, n = _rows_ptr(pos_mass, "pos_mass")
    if h.dtype != torch.float32 or not h.is_contiguous() or h.numel() != n or \
            h.device != pos_mass.device:
        raise ValueError("h must be a contiguous float32 tensor of n values on the same device")
    dev = pos_mass.device
    counts = torch.empty(n, dtype=torch.int32, device=dev)
    st = _stream(pos_mass, stream)
    if not lists:
        _check(ctx, lib().bh_neighbors(ctx, p, h.data_ptr(), n, float(kappa), int(mode),
                                       counts.data_ptr(), None, None, 0, st))
        return counts, None, None
    offsets = torch.empty(n + 1, dtype=torch.int64, device=dev)
    _check(ctx, lib().bh_neighbors(ctx, p, h.data_ptr(), n, float(kappa), int(mode),
                                   counts.data_ptr(), offsets.data_ptr(), None, 0, st))
    total = int(offsets[n].item()) if n else 0
    lst = torch.empty(max(total, 1), dtype=torch.int32, device=dev)
    _check(ctx, lib().bh_neighbors(ctx, p, h.data_ptr(), n, float(kappa), int(mode),
                                   counts.data_ptr(), offsets.data_ptr(), lst.data_ptr(),
                                   total, st))
    return counts, offsets, lst[:total]


def _host_rows(a, name):
    if a is None:
        return None, 0
    if hasattr(a, "numpy") and not isinstance(a, np.ndarray):   # cpu tensor
        if a.is_cuda:
            raise ValueError(f"{name} must be host memory")
        if a.dtype.__str__() != "torch.float32" or a.dim() != 2 or a.shape[1] != 4 \
                or not a.is_contiguous():
            raise ValueError(f"{name} must be contiguous float32 (n, 4)")
        return C.c_void_p(a.data_ptr()), a.shape[0]
    if not (isinstance(a, np.ndarray) and a.dtype == np.float32 and a.ndim == 2
            and a.shape[1] == 4 and a.flags.c_contiguous):
        raise ValueError(f"{name} must be a contiguous float32 (n, 4) array")
    return C.c_void_p(a.ctypes.data), a.shape[0]


def bh_compute_host(ctx, pos_mass, targets, acc_pot, stream=None) -> None:
    """Barnes-Hut on HOST arrays (numpy or CPU tensors, ideally pinned):
    copies in, computes, copies out and synchronises."""
    p, n = _host_rows(pos_mass, "pos_mass")
    t, m = _host_rows(targets, "targets")
    o, k = _host_rows(acc_pot, "acc_pot")
    if k != (n if targets is None else m):
        raise ValueError("acc_pot has the wrong number of rows")
    s = C.c_void_p(stream) if stream is not None else C.c_void_p(0)
    _check(ctx, lib().bh_compute_host(ctx, p, n, t, m, o, s))


def bh_sync_status(ctx, stream=None) -> int:
    """Synchronise and return the device status code (0 = BH_OK)."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    return lib().bh_sync_status(ctx, C.c_void_p(stream))


def bh_get_stage_times(ctx) -> dict:
    buf = (C.c_float * len(STAGES))()
    _check(ctx, lib().bh_get_stage_times(ctx, buf, len(STAGES)))
    return dict(zip(STAGES, [float(x) for x in buf]))


def bh_get_counters(ctx) -> tuple[int, int]:
    a, b = C.c_ulonglong(), C.c_ulonglong()
    _check(ctx, lib().bh_get_counters(ctx, C.byref(a), C.byref(b)))
    return a.value, b.value


def bh_debug_export(ctx, what: int, count: int = 0) -> np.ndarray:
    """Copy internal state of the last call to numpy (see BH_EXPORT_*)."""
    if what == BH_EXPORT_NODE_COUNT:
        out = np.zeros(1, np.int64)
    elif what == BH_EXPORT_CUBE:
        out = np.zeros(4, np.float32)
    elif what == BH_EXPORT_KEYS:
        out = np.zeros(count, np.uint64)
    elif what in (BH_EXPORT_PERM, BH_EXPORT_TARGET_PERM, BH_EXPORT_GROUP_COST,
                  BH_EXPORT_GROUP_ORDER):
        out = np.zeros(count, np.uint32)
    elif what == BH_EXPORT_NODES:
        out = np.zeros((count, 6), np.int32)
    elif what == BH_EXPORT_COM:
        out = np.zeros((count, 4), np.float32)
    elif what == BH_EXPORT_WALK_STATS:
        out = np.zeros(4, np.uint64)
    elif what == BH_EXPORT_SORT_PATH:
        out = np.zeros(2, np.uint32)
    else:
        raise ValueError("unknown export key")
    _check(ctx, lib().bh_debug_export(ctx, int(what), C.c_void_p(out.ctypes.data), out.nbytes))
    return out


def bh_count_interactions(ctx, counts=None, stream=None) -> int:
    """Per-target interaction count of the last bh_compute (total returned;
    per-target counts written to ``counts``, a uint32/int32 CUDA tensor, if
    given)."""
    import torch
    ptr = None
    if counts is not None:
        if not counts.is_cuda or counts.dtype not in (torch.int32,) or not counts.is_contiguous():
            raise ValueError("counts must be a contiguous int32 CUDA tensor")
        ptr = C.c_void_p(counts.data_ptr())
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    tot = C.c_ulonglong()
    _check(ctx, lib().bh_count_interactions(ctx, ptr, C.byref(tot), C.c_void_p(stream)))
    return tot.value


def bh_last_error(ctx) -> str:
    return lib().bh_last_error(ctx).decode()


_OPTION_KEYS = dict(key_bits=BH_OPT_KEY_BITS, leaf_cap=BH_OPT_LEAF_CAP,
                    opening=BH_OPT_OPENING, timing=BH_OPT_TIMING, group=BH_OPT_GROUP,
                    graph=BH_OPT_GRAPH, estimator=BH_OPT_ESTIMATOR, seed=BH_OPT_SEED,
                    samples=BH_OPT_SAMPLES, strata_level=BH_OPT_STRATA_LEVEL,
                    pipeline=BH_OPT_PIPELINE, order=BH_OPT_ORDER, shards=BH_OPT_SHARDS,
                    shard=BH_OPT_SHARD, schedule=BH_OPT_SCHEDULE,
                    target_key_bits=BH_OPT_TARGET_KEY_BITS)


class BarnesHut:
    """One library context with its parameters.

    >>> bh = BarnesHut(theta=0.5, G=1.0, eps=1e-3)
    >>> acc_pot = bh.compute(pos_mass)            # (n, 4) CUDA tensor
    """

    def __init__(self, theta=0.5, G=1.0, eps=0.0, device=0, max_sources=0,
                 max_targets=0, **options):
        self.ctx = bh_create(device, max_sources, max_targets)
        self.device = device
        bh_set_params(self.ctx, theta, G, eps)
        for k, v in options.items():
            bh_set_option(self.ctx, _OPTION_KEYS[k], v)

    def set_option(self, key: str, value: int) -> None:
        bh_set_option(self.ctx, _OPTION_KEYS[key], value)

    def set_params(self, theta, G, eps) -> None:
        bh_set_params(self.ctx, theta, G, eps)

    def compute(self, pos_mass, targets=None, out=None, stream=None):
        import torch
        rows = pos_mass.shape[0] if targets is None else targets.shape[0]
        if out is None:
            out = torch.empty((rows, 4), dtype=torch.float32, device=pos_mass.device)
        bh_compute(self.ctx, pos_mass, targets, out, stream)
        return out

    def direct(self, pos_mass, targets=None, out=None, stream=None):
        import torch
        rows = pos_mass.shape[0] if targets is None else targets.shape[0]
        if out is None:
            out = torch.empty((rows, 4), dtype=torch.float32, device=pos_mass.device)
        bh_direct(self.ctx, pos_mass, targets, out, stream)
        return out

    def status(self, stream=None) -> int:
        return bh_sync_status(self.ctx, stream)

    def close(self) -> None:
        if getattr(self, "ctx", None) is not None:
            bh_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
