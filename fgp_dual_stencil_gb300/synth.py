"""Seeded synthetic inputs for the FGP step: the volumes b that the oracle and
the GPU path are both fed.

This module holds none of the method's arithmetic; it only draws random
phantoms and noise.  It imports nothing but numpy, so the oracle's tests and
the GPU path's tests can share it without sharing any code of the method.

The page "TV solver: the FGP step on the GPU" measures on a phantom that is
not available here ("Result at 256³", the README phantom).  These generators
stand in for it with the same shapes and value ranges: a refractive-index
contrast in [0, 1] made of ellipsoids, plus Gaussian noise, fp32, x fastest.

Conventions: shapes are given as (nx, ny, nz); arrays come back C-ordered as
(nz, ny, nx) float32.  Every draw comes from ``numpy.random.default_rng`` on a
seed sequence ``[seed, stream]``: stream 0 is the phantom, stream 1000 + k the
noise of outer iteration k.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: volume shape, lambda and the step schedule."""
    key: str
    nx: int
    ny: int
    nz: int
    lam: float
    outers: int          # outer iterations (fresh b per outer when > 1)
    steps: int           # FGP steps per outer
    t0: float
    seed: int
    phantom_seed: int
    description: str

    @property
    def shape(self):
        return (self.nx, self.ny, self.nz)

    @property
    def nvox(self) -> int:
        return self.nx * self.ny * self.nz

    @property
    def total_steps(self) -> int:
        return self.outers * self.steps


WORKLOADS = {
    "c1": Workload("c1", 32, 32, 32, 0.05, 1, 10, 1.0, BASE_SEED + 0, BASE_SEED + 0,
                   "32x32x32: 4 painted axis-aligned ellipsoids U[0.2,1] + N(0,0.05^2); "
                   "lambda 0.05; 10 steps"),
    "c2": Workload("c2", 128, 128, 128, 0.03, 1, 50, 1.0, BASE_SEED + 1, BASE_SEED + 1,
                   "128^3: 12 additive ellipsoids U[0,1] + N(0,0.05^2); lambda 0.03; 50 steps"),
    "c3": Workload("c3", 256, 256, 256, 0.02, 20, 10, 1.0, BASE_SEED + 2, BASE_SEED + 2,
                   "256^3: fixed 10-ellipsoid phantom in [0,1] + fresh N(0,0.02^2) per outer; "
                   "20 outers x 10 steps, warm p/r, t0=1 each outer; lambda 0.02"),
    # The 512^3 phantom is the 256^3 one scaled: same phantom seed, relative
    # coordinates; its noise streams use its own seed.
    "c4": Workload("c4", 512, 512, 512, 0.02, 20, 10, 1.0, BASE_SEED + 3, BASE_SEED + 2,
                   "512^3: the 256^3 phantom scaled + fresh N(0,0.02^2) per outer; "
                   "20 outers x 10 steps, warm p/r, t0=1 each outer; lambda 0.02"),
    "c5": Workload("c5", 1000, 600, 300, 0.1, 1, 100, 1.0, BASE_SEED + 4, BASE_SEED + 4,
                   "1000x600x300: 200 Gaussian blobs (sigma U[3,15], peak U[0.5,2], cut at "
                   "2.5 sigma) + N(0,0.01^2), clamped >= 0; lambda 0.1; 100 steps"),
}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def ellipsoids(shape, count, rng, *, value_range, semi_range, centre_range=(0.2, 0.8),
               additive=False) -> np.ndarray:
    """Axis-aligned ellipsoids painted (later ones overwrite) or added.
    Centres, semi-axes are fractions of each axis length."""
    nx, ny, nz = shape
    vol = np.zeros((nz, ny, nx), dtype=np.float32)
    n = np.array([nx, ny, nz], dtype=np.float64)
    for _ in range(count):
        c = rng.uniform(centre_range[0], centre_range[1], size=3) * n
        a = rng.uniform(semi_range[0], semi_range[1], size=3) * n
        v = np.float32(rng.uniform(value_range[0], value_range[1]))
        lo = np.maximum(np.floor(c - a).astype(np.int64), 0)
        hi = np.minimum(np.ceil(c + a).astype(np.int64) + 1, n.astype(np.int64))
        if np.any(hi <= lo):
            continue
        xs = ((np.arange(lo[0], hi[0]) - c[0]) / a[0]) ** 2
        ys = ((np.arange(lo[1], hi[1]) - c[1]) / a[1]) ** 2
        zs = ((np.arange(lo[2], hi[2]) - c[2]) / a[2]) ** 2
        inside = (zs[:, None, None] + ys[None, :, None] + xs[None, None, :]) <= 1.0
        view = vol[lo[2]:hi[2], lo[1]:hi[1], lo[0]:hi[0]]
        if additive:
            view[inside] += v
        else:
            view[inside] = v
    return vol


def gaussian_blobs(shape, count, rng, *, sigma_range, peak_range, cut=2.5) -> np.ndarray:
    """Isotropic Gaussian blobs with uniform centres, truncated at cut*sigma, added."""
    nx, ny, nz = shape
    vol = np.zeros((nz, ny, nx), dtype=np.float32)
    n = np.array([nx, ny, nz], dtype=np.float64)
    for _ in range(count):
        c = rng.uniform(0.0, 1.0, size=3) * n
        s = rng.uniform(sigma_range[0], sigma_range[1])
        pk = rng.uniform(peak_range[0], peak_range[1])
        rad = cut * s
        lo = np.maximum(np.floor(c - rad).astype(np.int64), 0)
        hi = np.minimum(np.ceil(c + rad).astype(np.int64) + 1, n.astype(np.int64))
        if np.any(hi <= lo):
            continue
        dx = (np.arange(lo[0], hi[0]) - c[0]) ** 2
        dy = (np.arange(lo[1], hi[1]) - c[1]) ** 2
        dz = (np.arange(lo[2], hi[2]) - c[2]) ** 2
        d2 = dz[:, None, None] + dy[None, :, None] + dx[None, None, :]
        blob = pk * np.exp(-d2 / (2.0 * s * s))
        blob[d2 > rad * rad] = 0.0
        vol[lo[2]:hi[2], lo[1]:hi[1], lo[0]:hi[0]] += blob.astype(np.float32)
    return vol


def noise(shape, sigma, rng) -> np.ndarray:
    nx, ny, nz = shape
    out = rng.standard_normal((nz, ny, nx), dtype=np.float32)
    out *= np.float32(sigma)
    return out


def phantom(w: Workload) -> np.ndarray:
    """The noise-free part of b for workload w."""
    rng = _rng(w.phantom_seed, 0)
    if w.key == "c1":
        return ellipsoids(w.shape, 4, rng, value_range=(0.2, 1.0), semi_range=(0.1, 0.35))
    if w.key == "c2":
        return ellipsoids(w.shape, 12, rng, value_range=(0.0, 1.0), semi_range=(0.1, 0.35),
                          additive=True)
    if w.key in ("c3", "c4"):
        return ellipsoids(w.shape, 10, rng, value_range=(0.0, 1.0), semi_range=(0.05, 0.4))
    if w.key == "c5":
        return gaussian_blobs(w.shape, 200, rng, sigma_range=(3.0, 15.0), peak_range=(0.5, 2.0))
    raise KeyError(w.key)


_SIGMA = {"c1": 0.05, "c2": 0.05, "c3": 0.02, "c4": 0.02, "c5": 0.01}


def make_b(w: Workload, outer: int = 0, base: np.ndarray | None = None) -> np.ndarray:
    """b for outer iteration `outer` of workload w: phantom + fresh noise
    (clamped at 0 for the blob workload).  Pass `base` = phantom(w) to avoid
    redrawing the phantom for every outer."""
    if base is None:
        base = phantom(w)
    b = noise(w.shape, _SIGMA[w.key], _rng(w.seed, 1000 + outer))
    b += base
    if w.key == "c5":
        np.maximum(b, np.float32(0.0), out=b)
    return b


def random_case(shape, seed, *, lo=-0.5, hi=1.5) -> np.ndarray:
    """A small uniform random b for edge-case shapes (values may be negative,
    so that the clamp at 0 is exercised)."""
    nx, ny, nz = shape
    return _rng(seed, 7).uniform(lo, hi, size=(nz, ny, nx)).astype(np.float32)


def random_dual(shape, seed, *, scale=0.5) -> np.ndarray:
    """A random dual field (3, nz, ny, nx) float32, for warm-start cases."""
    nx, ny, nz = shape
    return (_rng(seed, 11).uniform(-scale, scale, size=(3, nz, ny, nx))).astype(np.float32)
