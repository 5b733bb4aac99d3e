"""Second, independent restatements used to pin the oracle on tiny inputs.

Pure Python, written from the definitions rather than from the oracle's C:
the canonical octree by enumerating every key prefix at every level, centres
of mass by direct weighted means per cell, and a recursive Barnes-Hut walk.
Only for N <= ~64.
"""
from __future__ import annotations

import math

import numpy as np


def brute_cells(skeys, bits, leaf_cap):
    """All cells of the canonical tree as {(level, prefix): (first, count)}.

    A cell at level l is the set of keys sharing their top 3*l bits.  It
    exists iff l == 0 or its parent exists and holds more than leaf_cap keys
    (and the parent's level is below bits).
    """
    n = len(skeys)
    cells = {}
    for lvl in range(bits + 1):
        sh = 3 * (bits - lvl)
        groups = {}
        for r, k in enumerate(skeys):
            p = int(k) >> sh
            f, c = groups.get(p, (r, 0))
            groups[p] = (min(f, r), c + 1)
        for p, (f, c) in groups.items():
            if lvl == 0:
                cells[(0, p)] = (f, c)
                continue
            par = cells.get((lvl - 1, p >> 3))
            if par is not None and par[1] > leaf_cap and lvl - 1 < bits:
                cells[(lvl, p)] = (f, c)
    if n == 0:
        return {}
    return cells


def is_internal(cells, key, bits, leaf_cap):
    lvl, _ = key
    return cells[key][1] > leaf_cap and lvl < bits


def cell_com(spm, first, count):
    p = spm[first:first + count].astype(np.float64)
    m = p[:, 3].sum()
    return (p[:, :3] * p[:, 3:4]).sum(axis=0) / m, m


def box_distance2(c, lo, hi, rule="box"):
    """Squared distance from point c to the axis-aligned box [lo, hi].

    rule "box" is the definition: the distance to the nearest point of the
    box, which is c itself clipped into the box axis by axis (0 on an axis
    where c lies between lo and hi).  The other rules are plausible mistakes,
    kept only so the tests can show that their inputs tell them apart:
    "far_corner" (distance to the farthest corner), "centre" (distance to the
    box centre) and "swapped" (the clip written with lo and hi exchanged).
    """
    c = np.asarray(c, np.float64)
    lo = np.asarray(lo, np.float64)
    hi = np.asarray(hi, np.float64)
    if rule == "box":
        d = c - np.clip(c, lo, hi)
    elif rule == "far_corner":
        d = c - np.where(np.abs(c - lo) > np.abs(c - hi), lo, hi)
    elif rule == "centre":
        d = c - 0.5 * (lo + hi)
    elif rule == "swapped":
        d = np.array([hi[a] - c[a] if c[a] < hi[a] else (c[a] - lo[a] if c[a] > lo[a] else 0.0)
                      for a in range(3)])
    else:
        raise ValueError(rule)
    return float(d @ d)


def recursive_bh(spm, skeys, bits, leaf_cap, L, theta, G, eps, x, self_j=-1,
                 group_x=None, group_rule="vote", log=None):
    """Barnes-Hut by recursion over brute_cells.

    group_x: optional (k,3) array.  With group_rule "vote" a cell is then
    accepted only if the test holds for every row (the warp-vote form); with
    a box rule ("box", or one of the planted mistakes of box_distance2) only
    if it holds at the distance from the centre of mass to the bounding box
    of the rows.  The returned value is for x.  log: optional list that
    receives (level, com, accepted) for every cell the walk decides.
    """
    cells = brute_cells(skeys, bits, leaf_cap)
    xs = np.asarray(x, np.float64)
    acc = np.zeros(4)
    terms = [0]
    if group_x is not None:
        gx = np.asarray(group_x, np.float64).reshape(-1, 3)
        glo, ghi = gx.min(axis=0), gx.max(axis=0)

    def term(src_pos, m):
        d = np.asarray(src_pos, np.float64) - xs
        r2 = float(d @ d) + eps * eps
        if r2 == 0.0:
            return
        inv = 1.0 / math.sqrt(r2)
        acc[:3] += m * d * inv ** 3
        acc[3] -= m * inv
        terms[0] += 1

    def visit(key):
        lvl, p = key
        f, c = cells[key]
        com, m = cell_com(spm, f, c)
        w = L / (2.0 ** lvl)
        ropen2 = (w * w) / (theta * theta) if theta > 0 else math.inf
        if group_x is not None and group_rule != "vote":
            ok = ropen2 < box_distance2(com, glo, ghi, group_rule)
        else:
            pts = [xs] if group_x is None else list(gx)
            ok = all(ropen2 < float((com - q) @ (com - q)) for q in pts)
        if log is not None:
            log.append((lvl, com, ok))
        if ok:
            term(com, m)
        elif not is_internal(cells, key, bits, leaf_cap):
            for j in range(f, f + c):
                if j != self_j:
                    term(spm[j, :3], float(spm[j, 3]))
        else:
            for d in range(8):
                ck = (lvl + 1, (p << 3) | d)
                if ck in cells:
                    visit(ck)

    if len(skeys):
        visit((0, 0))
    return G * acc, terms[0]


def decode(key, bits):
    q = [0, 0, 0]
    for k in range(bits):
        for a in range(3):
            q[a] |= ((int(key) >> (3 * k + a)) & 1) << k
    return tuple(q)
