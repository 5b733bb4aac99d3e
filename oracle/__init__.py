"""Barnes-Hut gravity oracle -- TEST INFRASTRUCTURE ONLY.

Plain CPU reference for the GPU path: fp64 physics, fp32 only for the two
integer-valued decisions (bounding cube, Morton quantisation) that the GPU
also takes in fp32.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import it; the library never does.

The arithmetic lives in ``bh_oracle.c`` (built to ``liborc.so`` by
``oracle/build.py``); this module only marshals numpy arrays.  Each step cites
the web page section it restates (see the C file's header):

* ``bbox``/``keys``/``sort`` -- "树结构" page, section 实现步骤 (bounding box by
  reduction, Morton / Z-order keys, spatial sort), octant numbering of section
  构建树结构.
* ``build_tree`` -- canonical octree over the sorted keys (subdivide a cell
  while it holds more than the leaf capacity), "树结构" page, 构建树结构.
* ``com`` -- GASPHiA page, section 计算核函数 (计算节点质心).
* ``bh``/``bh_group`` -- GASPHiA page, section 性能瓶颈分析 (opening test
  w_sq/theta_sq < r_sq; the warp vote in the group form).
* ``direct`` -- GASPHiA page, section 精度与加速比验证 (brute-force double loop).
* ``sbh`` -- stochastic Barnes-Hut ("Stochastic Barnes-Hut Approximation for
  Fast Summation on the GPU" page, section 方法: telescoping path sums, Russian
  roulette on the path length, stratification), with ``philox4x64`` as its
  counter-based random numbers.
* ``neighbors`` -- SPH neighbour search written out as brute force ("树结构"
  page, sections 粒子领域搜索 and 树遍历计算; GASPHiA's per-node maximum
  smoothing length), the distance test in fp32.
* ``leapfrog`` -- kick-drift-kick time stepping with brute-force forces (the
  pages show an N-body run advanced in time but print no integrator).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_u64p = np.ctypeslib.ndpointer(np.uint64, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_vp = C.c_void_p


def lib():
    """Load (building on first use) the oracle's shared library."""
    global _LIB
    if _LIB is None:
        path = os.path.join(_HERE, "liborc.so")
        if not os.path.exists(path):
            from . import build as _b
            _b.build()
        L = C.CDLL(path)
        L.orc_bbox.argtypes = [_f32p, C.c_int64, _f32p]
        L.orc_bbox.restype = C.c_int
        L.orc_quantise.argtypes = [_f32p, C.c_int64, _f32p, C.c_int, _u32p]
        L.orc_interleave.argtypes = [C.c_uint32, C.c_uint32, C.c_uint32, C.c_int]
        L.orc_interleave.restype = C.c_uint64
        L.orc_keys.argtypes = [_f32p, C.c_int64, _f32p, C.c_int, _u64p]
        L.orc_sort.argtypes = [_u64p, C.c_int64, _u32p]
        L.orc_sort.restype = C.c_int
        L.orc_build_tree.argtypes = [_u64p, C.c_int64, C.c_int, C.c_int, C.c_int64,
                                     _i32p, _i64p, _i64p, _i64p, _i32p]
        L.orc_build_tree.restype = C.c_int64
        L.orc_com.argtypes = [_f32p, _u64p, C.c_int64, _i32p, _i64p, _i64p,
                              _f32p, C.c_int, _f64p]
        L.orc_direct.argtypes = [_f32p, C.c_int64, _vp, C.c_int64, _vp, C.c_int64,
                                 C.c_double, C.c_double, _f64p]
        L.orc_bh.argtypes = [_f32p, C.c_int64, _i32p, _i64p, _i64p, _i64p, _i32p,
                             _f64p, C.c_double, C.c_double, C.c_double, C.c_double,
                             _f32p, _vp, C.c_int64, _f64p, _vp]
        L.orc_bh_group.argtypes = [_f32p, C.c_int64, _i32p, _i64p, _i64p, _i64p,
                                   _i32p, _f64p, C.c_double, C.c_double, C.c_double,
                                   C.c_double, _f32p, _vp, C.c_int64, C.c_int64,
                                   C.c_int, _f64p, _vp, _vp]
        L.orc_philox4x64.argtypes = [_u64p, _u64p, _u64p]
        L.orc_sbh.argtypes = [_f32p, C.c_int64, _i32p, _i64p, _i64p, _i64p, _i32p,
                              _f64p, C.c_float, C.c_double, C.c_double, _f32p, _vp,
                              _i64p, C.c_int64, C.c_uint64, C.c_int, C.c_int, _f64p,
                              _i64p, _f64p]
        L.orc_neighbors.argtypes = [_f32p, _f32p, C.c_int64, C.c_float, C.c_int, _i64p,
                                    C.c_int64, _i64p, _vp, _vp]
        L.orc_leapfrog.argtypes = [_f64p, _f64p, C.c_int64, C.c_double, C.c_double,
                                   C.c_double, C.c_int64]
        L.orc_num_threads.restype = C.c_int
        L.orc_set_threads.argtypes = [C.c_int]
        _LIB = L
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def _rows(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    assert a.ndim == 2 and a.shape[1] == 4
    return a


def bbox(pm) -> np.ndarray:
    """(lo_x, lo_y, lo_z, L) as fp32; raises ValueError on NaN/Inf input."""
    pm = _rows(pm)
    cube = np.zeros(4, np.float32)
    if lib().orc_bbox(pm, pm.shape[0], cube) != 0:
        raise ValueError("empty or non-finite input")
    return cube


def quantise(pm, cube, bits: int = 21) -> np.ndarray:
    pm = _rows(pm)
    q = np.zeros((pm.shape[0], 3), np.uint32)
    lib().orc_quantise(pm, pm.shape[0], np.ascontiguousarray(cube, np.float32), bits, q)
    return q


def interleave(qx: int, qy: int, qz: int, bits: int = 21) -> int:
    return int(lib().orc_interleave(qx, qy, qz, bits))


def keys(pm, cube, bits: int = 21) -> np.ndarray:
    pm = _rows(pm)
    k = np.zeros(pm.shape[0], np.uint64)
    lib().orc_keys(pm, pm.shape[0], np.ascontiguousarray(cube, np.float32), bits, k)
    return k


def sort(k) -> np.ndarray:
    """perm[r] = original index of the r-th key in stable key order."""
    k = np.ascontiguousarray(k, np.uint64)
    perm = np.zeros(k.shape[0], np.uint32)
    lib().orc_sort(k, k.shape[0], perm)
    return perm


def node_capacity(n: int, leaf_cap: int, bits: int = 21) -> int:
    """Upper bound on the node count of the canonical tree.

    Leaves <= n; nodes with two or more children < leaves; single-child
    internal cells hold more than leaf_cap particles and are disjoint within a
    level, so at most n/(leaf_cap+1) per level below ``bits``.
    """
    return 2 * n + bits * (n // (leaf_cap + 1) + 1) + 8


def build_tree(skeys, bits: int = 21, leaf_cap: int = 1) -> dict:
    skeys = np.ascontiguousarray(skeys, np.uint64)
    n = skeys.shape[0]
    cap = node_capacity(n, leaf_cap, bits)
    lv = np.zeros(cap, np.int32)
    fi = np.zeros(cap, np.int64)
    co = np.zeros(cap, np.int64)
    ch = np.zeros(cap, np.int64)
    nc = np.zeros(cap, np.int32)
    nn = lib().orc_build_tree(skeys, n, bits, leaf_cap, cap, lv, fi, co, ch, nc)
    if nn < 0:
        raise RuntimeError("node capacity exceeded")
    return dict(level=lv[:nn].copy(), first=fi[:nn].copy(), count=co[:nn].copy(),
                child=ch[:nn].copy(), nchild=nc[:nn].copy())


def com(spm, skeys, tree, cube, bits: int = 21) -> np.ndarray:
    spm = _rows(spm)
    nn = tree["level"].shape[0]
    out = np.zeros((nn, 4), np.float64)
    lib().orc_com(spm, np.ascontiguousarray(skeys, np.uint64), nn, tree["level"],
                  tree["first"], tree["count"], np.ascontiguousarray(cube, np.float32),
                  bits, out)
    return out


def direct(src, tgt=None, G: float = 1.0, eps: float = 0.0, idx=None) -> np.ndarray:
    """fp64 brute force.  tgt None = self mode.  idx: target rows to evaluate."""
    src = _rows(src)
    t = None if tgt is None else _rows(tgt)
    m = src.shape[0] if t is None else t.shape[0]
    ii = None if idx is None else np.ascontiguousarray(idx, np.int64)
    k = m if ii is None else ii.shape[0]
    out = np.zeros((k, 4), np.float64)
    lib().orc_direct(src, src.shape[0], _ptr(t), m, _ptr(ii), k, float(G), float(eps), out)
    return out


class OracleBH:
    """The whole Barnes-Hut pipeline on the CPU for one set of sources.

    Stages in the pages' order: bounding cube -> Morton keys -> stable sort ->
    canonical octree -> centre of mass.  ``bh`` then walks the tree per target;
    ``bh_group`` walks it per group of consecutive Morton-ordered targets.
    """

    def __init__(self, src, theta=0.5, G=1.0, eps=1e-3, bits=21, leaf_cap=1,
                 target_bits=10):
        self.src = _rows(src)
        self.target_bits = int(target_bits)
        self.n = self.src.shape[0]
        self.theta, self.G, self.eps = float(theta), float(G), float(eps)
        self.bits, self.leaf_cap = int(bits), int(leaf_cap)
        self.cube = bbox(self.src)
        self.keys = keys(self.src, self.cube, bits)
        self.perm = sort(self.keys)
        self.skeys = self.keys[self.perm]
        self.spm = np.ascontiguousarray(self.src[self.perm])
        self.rank = np.empty(self.n, np.int64)
        self.rank[self.perm] = np.arange(self.n)
        self.tree = build_tree(self.skeys, bits, leaf_cap)
        self.com = com(self.spm, self.skeys, self.tree, self.cube, bits)

    @property
    def nnodes(self) -> int:
        return self.tree["level"].shape[0]

    def _walk_args(self):
        t = self.tree
        return (self.spm, self.nnodes, t["level"], t["first"], t["count"], t["child"],
                t["nchild"], self.com, float(self.cube[3]), self.theta, self.G, self.eps)

    def bh(self, tgt=None, idx=None, theta=None):
        """Per-target Barnes-Hut.  Returns (out[k,4], terms[k]) in the order of idx.

        tgt None: self mode (targets = sources, own pair skipped); idx are
        original source (or target) indices, default all.
        """
        args = list(self._walk_args())
        if theta is not None:
            args[9] = float(theta)
        if tgt is None:
            ii = np.arange(self.n) if idx is None else np.asarray(idx, np.int64)
            pos = np.ascontiguousarray(self.src[ii])
            selfj = np.ascontiguousarray(self.rank[ii])
        else:
            t = _rows(tgt)
            ii = np.arange(t.shape[0]) if idx is None else np.asarray(idx, np.int64)
            pos = np.ascontiguousarray(t[ii])
            selfj = None
        k = pos.shape[0]
        out = np.zeros((k, 4), np.float64)
        terms = np.zeros(k, np.int64)
        lib().orc_bh(*args, pos, _ptr(selfj), k, out, terms.ctypes.data_as(C.c_void_p))
        return out, terms

    def target_order(self, tgt=None):
        """Morton order of the targets (the sources' own order in self mode).

        Separate targets are ordered by Morton keys of ``target_bits`` bits
        per axis on their own bounding cube (10 by default: the order only
        decides which targets share a group walk), ties by index."""
        if tgt is None:
            return self.perm.astype(np.int64)
        t = _rows(tgt)
        return sort(keys(t, bbox(t), self.target_bits)).astype(np.int64)

    def bh_group(self, tgt=None, group=32, mode=0, groups=None, theta=None,
                 with_abs=False):
        """Group walk over Morton-ordered targets.

        mode 0: a cell is accepted iff every target of the group accepts it
        (the warp vote); mode 1: iff the test holds at the distance from the
        centre of mass to the group's bounding box.  ``groups``: indices of the
        groups to evaluate (default all).  Returns (out rows, original target
        indices of those rows, terms per evaluated group), plus, with
        ``with_abs``, G * sum |acceleration term| per row.
        """
        args = list(self._walk_args())
        if theta is not None:
            args[9] = float(theta)
        order = self.target_order(tgt)
        k_all = order.shape[0]
        ng = (k_all + group - 1) // group
        gsel = np.arange(ng) if groups is None else np.sort(np.asarray(groups, np.int64))
        rows = np.concatenate([order[g * group:min(k_all, (g + 1) * group)] for g in gsel]) \
            if gsel.size else np.zeros(0, np.int64)
        if tgt is None:
            pos = np.ascontiguousarray(self.src[rows])
            selfj = np.ascontiguousarray(self.rank[rows])
        else:
            pos = np.ascontiguousarray(_rows(tgt)[rows])
            selfj = None
        k = pos.shape[0]
        out = np.zeros((k, 4), np.float64)
        terms = np.zeros(gsel.size, np.int64)
        absacc = np.zeros(k, np.float64)
        lib().orc_bh_group(*args, pos, _ptr(selfj), k, int(group), int(mode), out,
                           terms.ctypes.data_as(C.c_void_p), absacc.ctypes.data_as(C.c_void_p))
        if with_abs:
            return out, rows, terms, absacc
        return out, rows, terms

    def direct(self, tgt=None, idx=None):
        return direct(self.src, tgt, self.G, self.eps, idx)

    def sbh(self, tgt=None, rows=None, seed=0, strata_level=2, samples=1,
            group=32):
        """Stochastic Barnes-Hut estimate for target rows ``rows`` (original
        indices, default all), in that order.  Queries share random numbers
        within a group of ``group`` consecutive Morton-ordered targets.
        Returns (out[k,4], terms[k], scale[k,4]); scale columns: G * sum
        |weighted term| of the acceleration and of the potential, and G * the
        sums over cell terms of |weight| m / s^3 and |weight| m r / s^3
        (s^2 = r^2 + eps^2), the sensitivities to centre-of-mass rounding."""
        order = self.target_order(tgt)
        k_all = order.shape[0]
        gpos = np.empty(k_all, np.int64)
        gpos[order] = np.arange(k_all) // group
        rr = np.arange(k_all) if rows is None else np.asarray(rows, np.int64)
        if tgt is None:
            pos = np.ascontiguousarray(self.src[rr])
            selfj = np.ascontiguousarray(self.rank[rr])
        else:
            pos = np.ascontiguousarray(_rows(tgt)[rr])
            selfj = None
        k = pos.shape[0]
        grp = np.ascontiguousarray(gpos[rr])
        out = np.zeros((k, 4), np.float64)
        terms = np.zeros(k, np.int64)
        scale = np.zeros((k, 4), np.float64)
        t = self.tree
        lib().orc_sbh(self.spm, self.nnodes, t["level"], t["first"], t["count"],
                      t["child"], t["nchild"], self.com, float(self.cube[3]), self.G,
                      self.eps, pos, _ptr(selfj), grp, k, int(seed) & (2**64 - 1),
                      int(strata_level), int(samples), out, terms, scale)
        return out, terms, scale


NB_GATHER, NB_SYMMETRIC = 0, 1


def neighbors(pm, h, kappa: float = 2.0, mode: int = NB_SYMMETRIC, rows=None,
              with_lists: bool = True):
    """Brute-force neighbour search.  Returns (counts[k], lists) for query
    rows ``rows`` (default all); lists[r] holds row r's neighbour indices in
    ascending order (None without ``with_lists``)."""
    pm = _rows(pm)
    h = np.ascontiguousarray(h, np.float32)
    n = pm.shape[0]
    rr = np.arange(n, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    k = rr.shape[0]
    counts = np.zeros(k, np.int64)
    lib().orc_neighbors(pm, h, n, float(kappa), int(mode), rr, k, counts, None, None)
    if not with_lists:
        return counts, None
    offs = np.zeros(k + 1, np.int64)
    np.cumsum(counts, out=offs[1:])
    flat = np.zeros(max(int(offs[-1]), 1), np.int64)
    lib().orc_neighbors(pm, h, n, float(kappa), int(mode), rr, k, counts,
                        offs.ctypes.data_as(C.c_void_p), flat.ctypes.data_as(C.c_void_p))
    return counts, [flat[offs[r]:offs[r + 1]] for r in range(k)]


def philox4x64(counter, key) -> np.ndarray:
    """Philox4x64-10 block for a 4-word counter and 2-word key (uint64)."""
    c = np.ascontiguousarray(counter, np.uint64)
    k = np.ascontiguousarray(key, np.uint64)
    out = np.zeros(4, np.uint64)
    lib().orc_philox4x64(c, k, out)
    return out


def leapfrog(pos_mass, vel, G: float = 1.0, eps: float = 0.0, dt: float = 1e-3,
             nsteps: int = 1):
    """fp64 kick-drift-kick leapfrog with brute-force forces.  Returns the
    final (positions+masses (n,4), velocities (n,3)) as fp64 copies."""
    pos = np.ascontiguousarray(pos_mass, np.float64).copy()
    v = np.ascontiguousarray(np.asarray(vel, np.float64)[:, :3]).copy()
    lib().orc_leapfrog(pos, v, pos.shape[0], float(G), float(eps), float(dt), int(nsteps))
    return pos, v


def rel_error(a, ref, floor_frac: float = 1e-3) -> np.ndarray:
    """|a - ref| / max(|ref|, floor_frac * median |ref|), row-wise on 3-vectors
    (or scalars).  The floor keeps near-zero net forces (symmetric centres)
    from dominating the statistics."""
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    if a.ndim == 2:
        num = np.linalg.norm(a - ref, axis=1)
        den = np.linalg.norm(ref, axis=1)
    else:
        num = np.abs(a - ref)
        den = np.abs(ref)
    floor = floor_frac * np.median(den) if den.size else 0.0
    return num / np.maximum(den, floor if floor > 0 else 1e-300)


def error_stats(e) -> dict:
    e = np.asarray(e, np.float64)
    return dict(median=float(np.median(e)), p99=float(np.percentile(e, 99)),
                max=float(e.max()), mean=float(e.mean()))
