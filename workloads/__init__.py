"""Seeded synthetic inputs for the Barnes-Hut gravity path.

This module only draws random numbers and lays them out as fp32 ``(x, y, z, m)``
rows.  It holds none of the method's arithmetic (no keys, no tree, no forces),
so both the CPU oracle and the CUDA path can consume the same bytes.

Every generator draws in float64 from ``numpy.random.Generator(PCG64(seed))``
and casts to float32 at the end.  The five workloads follow the problem set of
the Barnes-Hut gravity study this library implements:

* ``uniform_cube``  -- N i.i.d. points in [0,1)^3, equal masses 1/N.
* ``lattice``       -- a regular n^3 lattice of cell centres filling the unit
  cube (the 1M-particle "regular arrangement" test of the GASPHiA tree-code
  page, section "性能测试与对比"), optionally shuffled to reproduce that page's
  "打乱后" (shuffled) run.
* ``ellipsoid_surfaces`` + ``query_grid`` -- sources sampled uniformly by area
  on random ellipsoid surfaces with a 100^3 query grid of targets; stands in for
  the 116-mesh dataset of the stochastic Barnes-Hut notes (section "实验结果"),
  which is not available here.
* ``galaxy_pair``   -- two Hernquist halo + exponential disk galaxies; stands in
  for the 5M-particle DICE galaxy-collision run shown at the top of the
  GASPHiA page.
* ``plummer``       -- a truncated Plummer sphere for the scaling sweep.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng", "uniform_cube", "lattice", "ellipsoid_surfaces", "query_grid",
    "galaxy_pair", "plummer", "uniform_ball", "sph_plummer", "uniform_sph",
    "error_sample", "WORKLOADS", "make",
]


def rng(seed: int) -> np.random.Generator:
    """The one generator every workload uses: PCG64 with a fixed seed."""
    return np.random.Generator(np.random.PCG64(seed))


def _pack(pos: np.ndarray, mass) -> np.ndarray:
    out = np.empty((pos.shape[0], 4), dtype=np.float64)
    out[:, :3] = pos
    out[:, 3] = mass
    return np.ascontiguousarray(out.astype(np.float32))


def _unit_vectors(g: np.random.Generator, n: int) -> np.ndarray:
    """Isotropic directions: cos(polar) uniform in [-1,1], azimuth uniform."""
    cz = 2.0 * g.random(n) - 1.0
    ph = 2.0 * np.pi * g.random(n)
    sz = np.sqrt(np.maximum(0.0, 1.0 - cz * cz))
    return np.stack([sz * np.cos(ph), sz * np.sin(ph), cz], axis=1)


def uniform_cube(n: int = 4096, seed: int = 0) -> np.ndarray:
    """N points i.i.d. uniform in [0,1)^3, each of mass 1/N."""
    g = rng(seed)
    return _pack(g.random((n, 3)), 1.0 / n)


def lattice(side: int = 100, spacing: float = 0.01, mass: float | None = None,
            permute_seed: int | None = None) -> np.ndarray:
    """side^3 particles at the cell centres (i+0.5)*spacing, x fastest.

    Index = i + side*j + side^2*k.  ``permute_seed`` shuffles the particle order
    with ``rng(permute_seed).permutation``.
    """
    n = side ** 3
    t = (np.arange(side, dtype=np.float64) + 0.5) * spacing
    z, y, x = np.meshgrid(t, t, t, indexing="ij")
    pos = np.stack([x.ravel(), y.ravel(), z.ravel()], axis=1)
    if mass is None:
        mass = 1.0 / n
    out = _pack(pos, mass)
    if permute_seed is not None:
        out = np.ascontiguousarray(out[rng(permute_seed).permutation(n)])
    return out


def ellipsoid_surfaces(m: int = 1 << 20, seed: int = 2, n_ell: int = 8,
                       area_samples: int = 1_000_000) -> np.ndarray:
    """M points uniform by area on the surfaces of ``n_ell`` random ellipsoids.

    Semi-axes U[0.05,0.3]^3 and centres U[0.2,0.8]^3, axis aligned.  The
    ellipsoid of each point is chosen by area share (area by a Monte-Carlo mean
    of the area element over the unit sphere), then the point by rejection:
    a unit direction u maps to c + diag(a,b,c) u and is kept with probability
    g(u)/g_max, g(u) = abc*sqrt(ux^2/a^2 + uy^2/b^2 + uz^2/c^2),
    g_max = abc/min(a,b,c).  Masses are equal area weights summing to 1.
    """
    g = rng(seed)
    axes = g.uniform(0.05, 0.3, size=(n_ell, 3))
    centres = g.uniform(0.2, 0.8, size=(n_ell, 3))
    u = _unit_vectors(g, area_samples)
    areas = np.empty(n_ell)
    for e in range(n_ell):
        a, b, c = axes[e]
        gu = a * b * c * np.sqrt((u[:, 0] / a) ** 2 + (u[:, 1] / b) ** 2 + (u[:, 2] / c) ** 2)
        areas[e] = 4.0 * np.pi * gu.mean()
    which = g.choice(n_ell, size=m, p=areas / areas.sum())
    pos = np.empty((m, 3))
    for e in range(n_ell):
        idx = np.nonzero(which == e)[0]
        need = idx.size
        a, b, c = axes[e]
        gmax = a * b * c / min(a, b, c)
        got = []
        while need > 0:
            k = max(1024, int(need * 1.6))
            d = _unit_vectors(g, k)
            gu = a * b * c * np.sqrt((d[:, 0] / a) ** 2 + (d[:, 1] / b) ** 2 + (d[:, 2] / c) ** 2)
            keep = d[g.random(k) < gu / gmax][:need]
            got.append(keep)
            need -= keep.shape[0]
        d = np.concatenate(got, axis=0)
        pos[idx] = centres[e] + d * axes[e]
    return _pack(pos, 1.0 / m)


def query_grid(sources: np.ndarray, side: int = 100) -> np.ndarray:
    """A side^3 grid of query points over the sources' bounding box.

    Endpoints included (coordinate lo + (hi-lo)*t/(side-1)), x fastest.  The
    fourth column is 0 (targets carry no mass).
    """
    p = sources[:, :3].astype(np.float64)
    lo, hi = p.min(axis=0), p.max(axis=0)
    t = np.arange(side, dtype=np.float64) / (side - 1)
    gx = lo[0] + (hi[0] - lo[0]) * t
    gy = lo[1] + (hi[1] - lo[1]) * t
    gz = lo[2] + (hi[2] - lo[2]) * t
    z, y, x = np.meshgrid(gz, gy, gx, indexing="ij")
    pos = np.stack([x.ravel(), y.ravel(), z.ravel()], axis=1)
    return _pack(pos, 0.0)


def _hernquist(g, n, a, rmax_over_a):
    smax = rmax_over_a / (1.0 + rmax_over_a)
    u = g.uniform(0.0, smax * smax, size=n)
    s = np.sqrt(u)
    r = a * s / (1.0 - s)
    return r[:, None] * _unit_vectors(g, n)


def _exp_disk(g, n, rd, z0, xmax):
    umax = 1.0 - (1.0 + xmax) * np.exp(-xmax)
    u = g.uniform(0.0, umax, size=n)
    x = np.full(n, 2.0)
    for _ in range(60):                      # Newton on 1-(1+x)e^-x = u
        ex = np.exp(-x)
        f = 1.0 - (1.0 + x) * ex - u
        x = np.clip(x - f / np.maximum(x * ex, 1e-300), 0.0, xmax)
        if np.max(np.abs(f)) < 1e-15:
            break
    ph = 2.0 * np.pi * g.random(n)
    w = 2.0 * g.random(n) - 1.0
    w = np.clip(w, -1.0 + 1e-15, 1.0 - 1e-15)
    z = z0 * np.arctanh(w)
    R = x * rd
    return np.stack([R * np.cos(ph), R * np.sin(ph), z], axis=1)


def galaxy_pair(n_total: int = 5_000_000, seed: int = 3) -> np.ndarray:
    """Two galaxies, each 60% Hernquist halo + 40% exponential disk by number.

    Halo: M_h = 1, scale a = 0.1, truncated at 10a (radius from the inverse of
    the enclosed-mass fraction (r/(r+a))^2).  Disk: M_d = 0.05, R_d = 0.02,
    radius from the inverse of 1-(1+x)e^-x truncated at x < 10, sech^2 vertical
    profile z = z0*atanh(2u-1), z0 = 0.002.  Centres (-0.25,0,0) and
    (+0.25,0,0); the second disk is tilted 45 degrees about the x axis.  Order:
    halo 1, disk 1, halo 2, disk 2.  At 5M this is 1.5M + 1M per galaxy.
    """
    g = rng(seed)
    per = n_total // 2
    nh = (per * 3) // 5
    nd = per - nh
    parts, masses = [], []
    c, s = np.cos(np.pi / 4), np.sin(np.pi / 4)
    rot_x = np.array([[1, 0, 0], [0, c, -s], [0, s, c]])
    for gi, cx in enumerate((-0.25, 0.25)):
        h = _hernquist(g, nh, 0.1, 10.0)
        d = _exp_disk(g, nd, 0.02, 0.002, 10.0)
        if gi == 1:
            d = d @ rot_x.T
        off = np.array([cx, 0.0, 0.0])
        parts += [h + off, d + off]
        masses += [np.full(nh, 1.0 / nh), np.full(nd, 0.05 / nd)]
    return _pack(np.concatenate(parts), np.concatenate(masses))


def plummer(n: int = 1 << 16, seed: int = 4, a: float = 0.1,
            trunc: float = 20.0) -> np.ndarray:
    """Plummer sphere of scale a truncated at trunc*a, total mass 1.

    r = a / sqrt(u^(-2/3) - 1) with u uniform in (0, u_max],
    u_max = (trunc^2/(trunc^2+1))^(3/2) (the enclosed-mass fraction at the
    truncation radius); isotropic directions; masses 1/N.
    """
    g = rng(seed)
    umax = (trunc * trunc / (trunc * trunc + 1.0)) ** 1.5
    u = umax * (1.0 - g.random(n))
    r = a / np.sqrt(u ** (-2.0 / 3.0) - 1.0)
    return _pack(r[:, None] * _unit_vectors(g, n), 1.0 / n)


def uniform_ball(n: int = 1 << 16, seed: int = 6, radius: float = 1.0,
                 total_mass: float = 1.0) -> np.ndarray:
    """N points uniform in a ball (r = R u^(1/3)), equal masses."""
    g = rng(seed)
    r = radius * np.cbrt(g.random(n))
    return _pack(r[:, None] * _unit_vectors(g, n), total_mass / n)


def sph_plummer(n: int = 1 << 20, seed: int = 4, a: float = 0.1,
                trunc: float = 20.0, n_ngb: float = 64.0):
    """Plummer sphere (as ``plummer``) with SPH smoothing lengths.

    h_i = eta * (m / rho(r_i))^(1/3) from the analytic Plummer density
    rho(r) = 3 M / (4 pi a^3) (1 + r^2/a^2)^(-5/2) (M = 1, m = 1/N), with
    eta chosen so that a sphere of radius 2 h holds n_ngb particles on
    average: (4/3) pi (2 h)^3 rho / m = n_ngb, i.e. eta^3 = 3 n_ngb / (32 pi).
    Returns (pos_mass float32 (n, 4), h float32 (n,)).
    """
    pm = plummer(n, seed=seed, a=a, trunc=trunc)
    r = np.linalg.norm(pm[:, :3].astype(np.float64), axis=1)
    rho = 3.0 / (4.0 * np.pi * a ** 3) * (1.0 + (r / a) ** 2) ** -2.5
    eta = (3.0 * n_ngb / (32.0 * np.pi)) ** (1.0 / 3.0)
    h = eta * np.cbrt((1.0 / n) / rho)
    return pm, h.astype(np.float32)


def uniform_sph(n: int = 1 << 20, seed: int = 0, n_ngb: float = 64.0):
    """Uniform cube [0,1)^3 with one smoothing length for all particles,
    chosen as in ``sph_plummer``: (4/3) pi (2 h)^3 n = n_ngb."""
    pm = uniform_cube(n, seed)
    h = (3.0 * n_ngb / (32.0 * np.pi * n)) ** (1.0 / 3.0)
    return pm, np.full(n, h, np.float32)


def error_sample(n: int, s: int = 16384, seed: int = 5) -> np.ndarray:
    """Sorted sample of min(s, n) distinct target indices (PCG64 seed 5)."""
    if n <= s:
        return np.arange(n, dtype=np.int64)
    return np.sort(rng(seed).choice(n, size=s, replace=False)).astype(np.int64)


# name -> (builder, G, eps, theta, mode).  mode "self" = targets are the sources.
WORKLOADS = {
    "uniform4096": (lambda: uniform_cube(4096, 0), 1.0, 1e-3, 0.5, "self"),
    "lattice1m": (lambda: lattice(100), 1.0, 5e-3, 0.5, "self"),
    "lattice1m_shuffled": (lambda: lattice(100, permute_seed=1), 1.0, 5e-3, 0.5, "self"),
    "surface2e15": (lambda: ellipsoid_surfaces(1 << 15), 1.0, 1e-4, 0.5, "grid"),
    "surface2e17": (lambda: ellipsoid_surfaces(1 << 17), 1.0, 1e-4, 0.5, "grid"),
    "surface2e20": (lambda: ellipsoid_surfaces(1 << 20), 1.0, 1e-4, 0.5, "grid"),
    "galaxy5m": (lambda: galaxy_pair(5_000_000), 1.0, 1e-3, 0.5, "self"),
}
for _e in (16, 18, 20, 22, 24):
    WORKLOADS[f"plummer2e{_e}"] = ((lambda e=_e: plummer(1 << e)), 1.0, 1e-3, 0.5, "self")


def make(name: str):
    """Return (sources, targets_or_None, G, eps, theta) for a named workload."""
    build, G, eps, theta, mode = WORKLOADS[name]
    src = build()
    tgt = query_grid(src) if mode == "grid" else None
    return src, tgt, G, eps, theta
