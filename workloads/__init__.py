"""Seeded synthetic body sets for the all-pairs gravity workloads.

This module is shared by the CPU oracle checks, the GPU parity tests and the
benchmark.  It holds only initial conditions (positions, masses, velocities)
and the seeded choice of sampled bodies; it contains no part of the force law
or of the integrator.

Every array is drawn in float64 with NumPy's PCG64 ``default_rng(seed)`` and
cast to float32 once, so both the oracle and the CUDA library read the very
same float32 bodies.  Bodies are float4 rows ``(x, y, z, m)``; velocities are
float4 rows ``(vx, vy, vz, 0)``.

Workloads (sizes and parameters as the benchmark definition states them):

* ``uniform-cube-1024``      N=1024, uniform in [-1,1]^3, m=1/N, v=0, seed 0,
                             eps2=1e-2, one evaluation + one step of dt=1e-3.
* ``plummer-16384``          N=16384 Plummer sphere (a=1, M=1, equal masses,
                             isotropic equilibrium velocities), seed 1,
                             eps2=1e-4, 10 steps of dt=1e-3.
* ``two-plummer-131072``     two Plummer spheres of 65536 bodies each (a=1,
                             mass 1/2 each) centred at x=+-3, closing at
                             relative speed 0.5, seed 2, eps2=1e-4, 10 steps of
                             dt=5e-4.
* ``ball-lognormal-1048576`` N=2^20 uniform in the unit ball, log-normal
                             (mu=0, sigma=1) masses normalised to total 1,
                             seed 3, eps2=1e-3, one evaluation; 4096 sampled
                             bodies for the oracle check.
* ``cube-sweep-<N>``         N in {1000, 4097, 65537, 500000, 4194304}, uniform
                             in [0,1]^3, m=1/N, seed 4, eps2=1e-3, one
                             evaluation; 4096 sampled bodies above N=65537.
* ``points2d-<N>``           2-D points for the cutoff neighbour list: uniform in
                             a square of side sqrt(N / 0.4) (0.4 points per unit
                             area, so ~4.5 neighbours within the cutoff 1.9 and
                             a thin tail above 10), seed 5, float32.  Stands in
                             for the coordinate file of the neighbour-list
                             example, which is not available here.
"""
from __future__ import annotations

import dataclasses

import numpy as np

SWEEP_SIZES = (1000, 4097, 65537, 500000, 4194304)
SAMPLE_COUNT = 4096
SAMPLE_SEED_OFFSET = 1000


@dataclasses.dataclass
class Workload:
    """One synthetic problem: float32 bodies and velocities plus run parameters."""

    name: str
    pos_mass: np.ndarray  # (n, 4) float32: x, y, z, m
    vel: np.ndarray  # (n, 4) float32: vx, vy, vz, 0
    eps2: float
    dt: float
    steps: int  # 0 means: one acceleration evaluation only
    sample: np.ndarray | None  # int64 indices the oracle checks, or None for all
    seed: int

    @property
    def n(self) -> int:
        return int(self.pos_mass.shape[0])


# --------------------------------------------------------------------------
# primitive draws
# --------------------------------------------------------------------------


def unit_vectors(rng: np.random.Generator, n: int) -> np.ndarray:
    """Isotropic unit vectors: three normals, normalised (float64, (n, 3))."""
    v = rng.standard_normal((n, 3))
    norm = np.linalg.norm(v, axis=1, keepdims=True)
    bad = norm[:, 0] == 0.0
    if np.any(bad):  # probability ~0; keep the draw count fixed anyway
        v[bad] = (1.0, 0.0, 0.0)
        norm[bad] = 1.0
    return v / norm


def uniform_box(rng: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    return lo + (hi - lo) * rng.random((n, 3))


def uniform_ball(rng: np.random.Generator, n: int, radius: float = 1.0) -> np.ndarray:
    """Uniform in a ball: isotropic direction times radius * u^(1/3)."""
    d = unit_vectors(rng, n)
    r = radius * np.cbrt(rng.random(n))
    return d * r[:, None]


def lognormal_masses(rng: np.random.Generator, n: int, total: float = 1.0) -> np.ndarray:
    """exp(N(0, 1)) masses divided by their float64 sum (times ``total``)."""
    m = np.exp(rng.standard_normal(n))
    return m * (total / m.sum())


def plummer(rng: np.random.Generator, n: int, total_mass: float = 1.0,
            scale: float = 1.0) -> tuple[np.ndarray, np.ndarray]:
    """Plummer sphere by the Aarseth-Henon-Wielen (1974) recipe, G = 1.

    Radius: invert the enclosed-mass fraction M(<r)/M = r^3/(r^2+a^2)^(3/2) at
    a uniform deviate.  Speed: q drawn by rejection from q^2 (1-q^2)^(7/2) on
    [0, 1] (bound 0.1 > max 0.0923), times the local escape speed
    sqrt(2 M / a) (1 + r^2/a^2)^(-1/4).  Directions isotropic.  No radial
    cut-off and no virial rescaling; the centre of mass and its velocity are
    subtracted.  Returns float64 positions and velocities, each (n, 3).
    """
    x1 = rng.random(n)
    x1 = np.maximum(x1, np.finfo(np.float64).tiny)
    r = scale / np.sqrt(x1 ** (-2.0 / 3.0) - 1.0)
    pos = unit_vectors(rng, n) * r[:, None]

    q = np.empty(n)
    filled = 0
    while filled < n:
        want = n - filled
        cand = rng.random(want)
        y = 0.1 * rng.random(want)
        ok = cand[y < cand * cand * (1.0 - cand * cand) ** 3.5]
        take = ok[: n - filled]
        q[filled:filled + take.size] = take
        filled += take.size
    vesc = np.sqrt(2.0 * total_mass / scale) * (1.0 + (r / scale) ** 2) ** (-0.25)
    vel = unit_vectors(rng, n) * (q * vesc)[:, None]

    pos -= pos.mean(axis=0)
    vel -= vel.mean(axis=0)
    return pos, vel


def sample_indices(n: int, seed: int, count: int = SAMPLE_COUNT) -> np.ndarray:
    """Seeded sorted subset of ``count`` distinct body indices (no replacement)."""
    rng = np.random.default_rng(seed + SAMPLE_SEED_OFFSET)
    idx = rng.choice(n, size=min(count, n), replace=False)
    return np.sort(idx).astype(np.int64)


def pack(pos: np.ndarray, mass: np.ndarray, vel: np.ndarray | None) -> tuple[np.ndarray, np.ndarray]:
    """float64 (n,3) positions, (n,) masses, (n,3) velocities -> float32 float4 rows."""
    n = pos.shape[0]
    pm = np.empty((n, 4), dtype=np.float64)
    pm[:, :3] = pos
    pm[:, 3] = mass
    v = np.zeros((n, 4), dtype=np.float64)
    if vel is not None:
        v[:, :3] = vel
    return np.ascontiguousarray(pm.astype(np.float32)), np.ascontiguousarray(v.astype(np.float32))


# --------------------------------------------------------------------------
# the named workloads
# --------------------------------------------------------------------------


def uniform_cube_1024() -> Workload:
    n, seed = 1024, 0
    rng = np.random.default_rng(seed)
    pos = uniform_box(rng, n, -1.0, 1.0)
    pm, v = pack(pos, np.full(n, 1.0 / n), None)
    return Workload("uniform-cube-1024", pm, v, 1e-2, 1e-3, 1, None, seed)


def plummer_16384() -> Workload:
    n, seed = 16384, 1
    rng = np.random.default_rng(seed)
    pos, vel = plummer(rng, n)
    pm, v = pack(pos, np.full(n, 1.0 / n), vel)
    return Workload("plummer-16384", pm, v, 1e-4, 1e-3, 10, None, seed)


def two_plummer_131072(n: int = 131072) -> Workload:
    """Two equal Plummer spheres (mass 1/2 each, a=1) at x=+-3 closing at 0.5.

    Each sphere is drawn as a unit-mass Plummer model and its velocities are
    scaled by sqrt(1/2) so that a half-mass sphere stays in equilibrium.  The
    sphere at +3 moves with vx -= 0.25, the one at -3 with vx += 0.25.
    """
    seed = 2
    half = n // 2
    rng = np.random.default_rng(seed)
    pa, va = plummer(rng, half)
    pb, vb = plummer(rng, n - half)
    s = np.sqrt(0.5)
    pa[:, 0] += 3.0
    pb[:, 0] -= 3.0
    va *= s
    vb *= s
    va[:, 0] -= 0.25
    vb[:, 0] += 0.25
    pos = np.concatenate([pa, pb])
    vel = np.concatenate([va, vb])
    pm, v = pack(pos, np.full(n, 1.0 / n), vel)
    return Workload(f"two-plummer-{n}", pm, v, 1e-4, 5e-4, 10, None, seed)


def ball_lognormal_1048576(n: int = 1048576) -> Workload:
    seed = 3
    rng = np.random.default_rng(seed)
    pos = uniform_ball(rng, n)
    m = lognormal_masses(rng, n)
    pm, v = pack(pos, m, None)
    return Workload(f"ball-lognormal-{n}", pm, v, 1e-3, 1e-3, 0,
                    sample_indices(n, seed), seed)


def cube_sweep(n: int) -> Workload:
    seed = 4
    rng = np.random.default_rng(seed)
    pos = uniform_box(rng, n, 0.0, 1.0)
    pm, v = pack(pos, np.full(n, 1.0 / n), None)
    sample = sample_indices(n, seed) if n > 65537 else None
    return Workload(f"cube-sweep-{n}", pm, v, 1e-3, 1e-3, 0, sample, seed)


def by_name(name: str) -> Workload:
    if name == "uniform-cube-1024":
        return uniform_cube_1024()
    if name == "plummer-16384":
        return plummer_16384()
    if name.startswith("two-plummer-"):
        return two_plummer_131072(int(name.rsplit("-", 1)[1]))
    if name.startswith("ball-lognormal-"):
        return ball_lognormal_1048576(int(name.rsplit("-", 1)[1]))
    if name.startswith("cube-sweep-"):
        return cube_sweep(int(name.rsplit("-", 1)[1]))
    if name.startswith("points2d-"):
        return points_2d(int(name.rsplit("-", 1)[1]))
    raise KeyError(name)


WORKLOAD_NAMES = (
    "uniform-cube-1024",
    "plummer-16384",
    "two-plummer-131072",
    "ball-lognormal-1048576",
) + tuple(f"cube-sweep-{n}" for n in SWEEP_SIZES)


def random_bodies(n: int, seed: int, spread: float = 1.0,
                  mass_lo: float = 0.5, mass_hi: float = 1.5) -> np.ndarray:
    """Generic float32 bodies for edge-case tests: uniform box, uniform masses."""
    rng = np.random.default_rng(seed)
    pos = uniform_box(rng, n, -spread, spread)
    m = mass_lo + (mass_hi - mass_lo) * rng.random(n)
    pm, _ = pack(pos, m / n, None)
    return pm


def random_velocities(n: int, seed: int, scale: float = 0.1) -> np.ndarray:
    rng = np.random.default_rng(seed + 7919)
    v = np.zeros((n, 4), dtype=np.float64)
    v[:, :3] = scale * rng.standard_normal((n, 3))
    v[:, 3] = rng.random(n)  # arbitrary w: the library must leave it untouched
    return np.ascontiguousarray(v.astype(np.float32))


NEIGHBOR_CUTOFF = 1.9
NEIGHBOR_MAX = 10


@dataclasses.dataclass
class Points2D:
    name: str
    x: np.ndarray  # (n,) float32
    y: np.ndarray  # (n,) float32
    cutoff: float
    max_neighbors: int

    @property
    def n(self) -> int:
        return int(self.x.shape[0])


def points_2d(n: int, seed: int = 5, density: float = 0.4) -> Points2D:
    rng = np.random.default_rng(seed)
    side = float(np.sqrt(n / density))
    xy = side * rng.random((n, 2))
    return Points2D(f"points2d-{n}", np.ascontiguousarray(xy[:, 0].astype(np.float32)),
                    np.ascontiguousarray(xy[:, 1].astype(np.float32)), NEIGHBOR_CUTOFF,
                    NEIGHBOR_MAX)
