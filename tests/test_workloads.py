"""The seeded input generators: determinism, layout and distribution checks.

The exact draws are fixed only by the seed (nothing external prints them);
what is pinned here is their structure and their distributions: uniform
boxes and balls, log-normal masses, and the Plummer model's enclosed-mass
profile M(<r) = r^3/(1+r^2)^{3/2}, its virial equilibrium and its mean field
-r/(1+r^2)^{3/2} (G = M = a = 1).
"""
import numpy as np
import pytest
from scipy import stats
from scipy.spatial.distance import pdist

import oracle
import workloads as W


def test_deterministic_by_seed():
    a = W.plummer_16384()
    b = W.plummer_16384()
    assert np.array_equal(a.pos_mass, b.pos_mass) and np.array_equal(a.vel, b.vel)
    c = W.cube_sweep(4097)
    d = W.cube_sweep(4097)
    assert np.array_equal(c.pos_mass, d.pos_mass)


@pytest.mark.parametrize("name", ["uniform-cube-1024", "plummer-16384", "cube-sweep-1000",
                                  "cube-sweep-4097", "cube-sweep-65537"])
def test_layout(name):
    w = W.by_name(name)
    assert w.pos_mass.dtype == np.float32 and w.pos_mass.shape == (w.n, 4)
    assert w.vel.dtype == np.float32 and w.vel.shape == (w.n, 4)
    assert w.pos_mass.flags.c_contiguous and w.vel.flags.c_contiguous
    assert np.all(w.vel[:, 3] == 0.0)
    assert np.all(w.pos_mass[:, 3] > 0.0)
    assert abs(float(np.sum(w.pos_mass[:, 3], dtype=np.float64)) - 1.0) < 1e-5
    assert w.eps2 > 0.0


def test_uniform_cube_1024():
    w = W.uniform_cube_1024()
    assert w.n == 1024 and w.eps2 == 1e-2 and w.dt == 1e-3 and w.steps == 1
    p = w.pos_mass[:, :3]
    assert p.min() >= -1.0 and p.max() <= 1.0
    assert np.all(w.vel == 0.0)
    assert np.all(w.pos_mass[:, 3] == np.float32(1.0 / 1024))
    for c in range(3):
        assert stats.kstest((p[:, c] + 1.0) / 2.0, "uniform").pvalue > 1e-3


def test_cube_sweep_bounds_and_sampling():
    w = W.cube_sweep(65537)
    p = w.pos_mass[:, :3]
    assert p.min() >= 0.0 and p.max() <= 1.0 and w.sample is None
    idx = W.sample_indices(500000, 4)
    assert idx.shape == (4096,) and np.all(np.diff(idx) > 0)
    assert idx.min() >= 0 and idx.max() < 500000
    assert np.array_equal(idx, W.sample_indices(500000, 4))


def test_unit_ball_lognormal():
    w = W.ball_lognormal_1048576(n=65536)  # same recipe, smaller n for speed
    r = np.linalg.norm(w.pos_mass[:, :3].astype(np.float64), axis=1)
    assert r.max() <= 1.0 + 1e-6
    assert stats.kstest(r ** 3, "uniform").pvalue > 1e-3
    m = w.pos_mass[:, 3].astype(np.float64)
    lm = np.log(m)
    assert abs(np.std(lm) - 1.0) < 0.02
    assert abs(m.sum() - 1.0) < 1e-4


def test_plummer_enclosed_mass_profile():
    w = W.plummer_16384()
    r = np.linalg.norm(w.pos_mass[:, :3].astype(np.float64), axis=1)
    frac = r ** 3 / (1.0 + r * r) ** 1.5
    assert stats.kstest(frac, "uniform").pvalue > 1e-3


def test_plummer_virial_equilibrium():
    """Kinetic energy 3 pi/64 and potential -3 pi/32 for G = M = a = 1."""
    w = W.plummer_16384()
    m = w.pos_mass[:, 3].astype(np.float64)
    v = w.vel[:, :3].astype(np.float64)
    T = 0.5 * float(np.sum(m * np.sum(v * v, axis=1)))
    assert abs(T / (3 * np.pi / 64) - 1.0) < 0.05
    rng = np.random.default_rng(0)
    sub = rng.choice(w.n, 4096, replace=False)
    x = w.pos_mass[sub, :3].astype(np.float64)
    d = pdist(x)  # the len(sub) * (len(sub) - 1) / 2 pair distances
    pair_sum = float(np.sum(1.0 / d))
    n_pairs_all = w.n * (w.n - 1) / 2
    Wpot = -(1.0 / w.n) ** 2 * pair_sum * n_pairs_all / d.size
    assert abs(Wpot / (-3 * np.pi / 32) - 1.0) < 0.06
    assert abs(2 * T / abs(Wpot) - 1.0) < 0.1


def test_plummer_mean_field_through_oracle():
    """Binned mean radial acceleration approaches -r/(1+r^2)^{3/2}."""
    w = W.plummer_16384()
    rng = np.random.default_rng(1)
    tgt = np.sort(rng.choice(w.n, 2048, replace=False))
    a = oracle.accel(w.pos_mass, w.eps2, idx=tgt)
    x = w.pos_mass[tgt, :3].astype(np.float64)
    r = np.linalg.norm(x, axis=1)
    ar = np.sum(a * x, axis=1) / r
    for lo, hi in [(0.3, 0.6), (0.6, 1.0), (1.0, 1.6), (1.6, 3.0)]:
        sel = (r >= lo) & (r < hi)
        assert sel.sum() > 100
        want = np.mean(-r[sel] / (1.0 + r[sel] ** 2) ** 1.5)
        got = np.mean(ar[sel])
        assert abs(got / want - 1.0) < 0.05, (lo, hi, got, want)


def test_two_plummer_layout():
    w = W.two_plummer_131072(n=8192)  # same recipe at a smaller n
    p = w.pos_mass[:, :3].astype(np.float64)
    v = w.vel[:, :3].astype(np.float64)
    h = w.n // 2
    assert abs(p[:h, 0].mean() - 3.0) < 1e-5 and abs(p[h:, 0].mean() + 3.0) < 1e-5
    assert abs(v[:h, 0].mean() + 0.25) < 1e-6 and abs(v[h:, 0].mean() - 0.25) < 1e-6
    assert abs(float(w.pos_mass[:, 3].astype(np.float64).sum()) - 1.0) < 1e-5
    assert w.eps2 == 1e-4 and w.dt == 5e-4 and w.steps == 10


def test_names_resolve():
    for name in W.WORKLOAD_NAMES[:3]:
        assert W.by_name(name).name == name
    with pytest.raises(KeyError):
        W.by_name("nope")
