"""Checks that pin the FP64 oracle to facts outside itself.

Each ``pin_*`` function takes a loaded oracle (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with a closed form, an invariant, a
special case or a correctly rounded brute-force sum.  The same functions run
against the real oracle (``test_oracle_pins.py``) and against deliberately
broken copies of it (``test_oracle_mutants.py``), where at least one of them
must fail.

Sources: "CUDA N-Body Simulation" (LienoPC/N-BodySimulation README) §1.2
(softened sum, G = 1, zero self term) and §1.3 (half-kick with a(x(t)), then
drift with the kicked velocity).
"""
from __future__ import annotations

import math

import numpy as np


def _close(got, want, tol, scale=None, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if scale is None:
        scale = max(float(np.max(np.abs(want))), 1e-300)
    err = float(np.max(np.abs(got - want))) / scale
    assert np.all(np.isfinite(got)), f"{what}: non-finite result {got}"
    assert err <= tol, f"{what}: relative error {err:.3e} > {tol:.1e}\n got={got}\nwant={want}"


def _two_body_expected(x0, x1, m0, m1, eps2):
    """Closed form: a_0 = m_1 r/(|r|^2+eps2)^{3/2}, a_1 = -m_0 r/(...), r = x_1 - x_0."""
    r = np.asarray(x1, float) - np.asarray(x0, float)
    d = float(r @ r) + eps2
    f = d ** -1.5
    return m1 * f * r, -m0 * f * r


# ---------------------------------------------------------------------------
# acceleration pins
# ---------------------------------------------------------------------------


def pin_two_body_closed_form(o):
    cases = [
        ((0.0, 0.0, 0.0), (1.0, 0.0, 0.0), 2.0, 3.0, 0.01),
        ((0.0, 0.0, 0.0), (0.0, -2.0, 0.0), 0.5, 4.0, 0.25),
        ((1.0, 1.0, 1.0), (1.0, 1.0, 3.0), 1.0, 7.0, 1e-4),
        ((0.3, -0.2, 0.1), (-0.4, 0.5, 0.9), 1.5, 0.25, 0.09),
    ]
    for x0, x1, m0, m1, eps2 in cases:
        pm = np.array([[*x0, m0], [*x1, m1]])
        a = o.accel(pm, eps2)
        e0, e1 = _two_body_expected(x0, x1, m0, m1, eps2)
        _close(a[0], e0, 1e-14, what=f"two-body a0 {x0}->{x1}")
        _close(a[1], e1, 1e-14, what=f"two-body a1 {x0}->{x1}")


def _ring(n, radius, total_mass):
    th = 2.0 * np.pi * np.arange(n) / n
    pm = np.zeros((n, 4))
    pm[:, 0] = radius * np.cos(th)
    pm[:, 1] = radius * np.sin(th)
    pm[:, 3] = total_mass / n
    return pm


def pin_ring_axis_closed_form(o):
    """A point on the axis of a ring of mass M, radius R, at height z:
    every ring body is at distance sqrt(R^2 + z^2), the in-plane parts cancel,
    so a = -M z / (R^2 + z^2 + eps2)^{3/2} along the axis."""
    for n, R, M, eps2 in [(16, 1.0, 1.0, 0.01), (37, 2.0, 3.0, 1.0), (64, 0.5, 0.2, 0.3)]:
        for z in (0.0, 0.2, -0.7, 1.5, 4.0):
            pm = np.vstack([_ring(n, R, M), [[0.0, 0.0, z, 0.8]]])
            a = o.accel(pm, eps2)[-1]
            az = -M * z / (R * R + z * z + eps2) ** 1.5
            scale = M / (R * R + eps2)
            _close(a, [0.0, 0.0, az], 1e-13, scale=scale, what=f"ring n={n} z={z}")


def pin_cube_centre_zero(o):
    """Equal masses on the 8 corners of a cube: zero acceleration at the centre,
    and each corner's pull points at the centre with equal magnitude."""
    c = np.array([[sx, sy, sz] for sx in (-1, 1) for sy in (-1, 1) for sz in (-1, 1)], float)
    pm = np.zeros((9, 4))
    pm[:8, :3] = 0.5 * c
    pm[:8, 3] = 0.125
    pm[8] = (0.0, 0.0, 0.0, 2.0)
    a = o.accel(pm, 0.05)
    term = 0.125 / (0.75 + 0.05) ** 1.5
    _close(a[8], np.zeros(3), 1e-14, scale=term, what="cube centre")
    mags = np.linalg.norm(a[:8], axis=1)
    assert np.max(np.abs(mags - mags[0])) <= 1e-14 * mags[0], "cube corners differ"
    cosines = np.sum(a[:8] * (-c), axis=1) / (mags * math.sqrt(3.0))
    assert np.all(np.abs(cosines - 1.0) < 1e-14), "corner pull not toward centre"


def pin_single_body_and_coincident_zero(o):
    a = o.accel(np.array([[0.3, -1.2, 5.0, 7.0]]), 1e-3)
    assert np.all(a == 0.0), f"single body accelerates: {a}"
    pm = np.array([[0.3, -1.2, 5.0, 7.0], [0.3, -1.2, 5.0, 2.0]])
    a = o.accel(pm, 1e-3)
    assert np.all(a == 0.0), f"coincident pair accelerates: {a}"


def pin_momentum_antisymmetry(o):
    """sum_i m_i a_i = 0: each pair's terms are equal and opposite."""
    rng = np.random.default_rng(12)
    pm = np.zeros((300, 4))
    pm[:, :3] = rng.normal(size=(300, 3))
    pm[:, 3] = rng.uniform(0.1, 3.0, size=300)
    a = o.accel(pm, 1e-2)
    net = np.sum(pm[:, 3:4] * a, axis=0)
    scale = float(np.sum(pm[:, 3] * np.linalg.norm(a, axis=1)))
    assert np.max(np.abs(net)) <= 1e-13 * scale, f"net force {net} vs scale {scale}"


def pin_scaling_homogeneity(o):
    """a(lambda x, lambda^2 eps2) = a(x, eps2) / lambda^2.  For lambda = 2 every
    operation is scaled by a power of two, so the equality is bitwise."""
    rng = np.random.default_rng(3)
    pm = np.zeros((50, 4))
    pm[:, :3] = rng.uniform(-1, 1, size=(50, 3))
    pm[:, 3] = rng.uniform(0.5, 1.5, size=50)
    eps2 = 0.02
    a1 = o.accel(pm, eps2)
    s = pm.copy()
    s[:, :3] *= 2.0
    a2 = o.accel(s, 4.0 * eps2)
    assert np.array_equal(a2 * 4.0, a1), "lambda=2 scaling not exact"
    s = pm.copy()
    s[:, :3] *= 3.0
    a3 = o.accel(s, 9.0 * eps2)
    _close(a3 * 9.0, a1, 1e-13, what="lambda=3 scaling")


def pin_mass_linearity(o):
    """a is linear in the source masses: doubling all masses doubles a, and a
    from masses m1 + m2 is a(m1) + a(m2)."""
    rng = np.random.default_rng(4)
    pm = np.zeros((60, 4))
    pm[:, :3] = rng.uniform(-1, 1, size=(60, 3))
    m1 = rng.uniform(0.1, 1.0, size=60)
    m2 = rng.uniform(0.1, 1.0, size=60)
    pm[:, 3] = m1
    a1 = o.accel(pm, 0.01)
    p2 = pm.copy()
    p2[:, 3] = 2.0 * m1
    assert np.array_equal(o.accel(p2, 0.01), 2.0 * a1), "mass doubling not exact"
    p2[:, 3] = m2
    a2 = o.accel(p2, 0.01)
    p2[:, 3] = m1 + m2
    _close(o.accel(p2, 0.01), a1 + a2, 1e-13, what="mass superposition")


def pin_translation_invariance(o):
    rng = np.random.default_rng(5)
    pm = np.zeros((40, 4))
    pm[:, :3] = rng.uniform(-1, 1, size=(40, 3))
    pm[:, 3] = rng.uniform(0.5, 1.5, size=40)
    a = o.accel(pm, 0.01)
    sh = pm.copy()
    sh[:, :3] += (0.25, -0.5, 1.0)
    _close(o.accel(sh, 0.01), a, 1e-13, what="translation")


def pin_bruteforce_fsum(o):
    """Tiny N: every component against a correctly rounded sum (math.fsum) of
    the terms over j != i, written independently here in pure Python."""
    rng = np.random.default_rng(6)
    for n, eps2 in [(2, 0.1), (7, 1e-3), (40, 1e-2)]:
        pm = np.zeros((n, 4))
        pm[:, :3] = rng.normal(size=(n, 3))
        pm[:, 3] = rng.uniform(0.1, 2.0, size=n)
        a = o.accel(pm, eps2)
        for i in range(n):
            terms = [[], [], []]
            for j in range(n):
                if j == i:
                    continue
                r = [pm[j, c] - pm[i, c] for c in range(3)]
                d = r[0] * r[0] + r[1] * r[1] + r[2] * r[2] + eps2
                w = pm[j, 3] / (d * math.sqrt(d))
                for c in range(3):
                    terms[c].append(w * r[c])
            for c in range(3):
                want = math.fsum(terms[c])
                scale = math.fsum(abs(t) for t in terms[c])
                assert abs(a[i, c] - want) <= 1e-13 * scale, (
                    f"n={n} i={i} c={c}: {a[i, c]} vs fsum {want}")


def pin_sampled_rows_match_full(o):
    rng = np.random.default_rng(7)
    pm = np.zeros((200, 4))
    pm[:, :3] = rng.normal(size=(200, 3))
    pm[:, 3] = rng.uniform(0.1, 2.0, size=200)
    full = o.accel(pm, 1e-3)
    idx = np.array([199, 0, 17, 17, 123, 5])
    part = o.accel(pm, 1e-3, idx=idx)
    assert np.array_equal(part, full[idx]), "sampled rows differ from full rows"


# ---------------------------------------------------------------------------
# leapfrog pins
# ---------------------------------------------------------------------------


def pin_leapfrog_zero_steps(o):
    pm = np.array([[0.0, 0.0, 0.0, 1.0], [1.0, 0.0, 0.0, 1.0]])
    v = np.array([[0.1, 0.2, 0.3], [0.0, 0.0, 0.0]])
    p2, v2, a2 = o.leapfrog(pm, v, 0.01, 0.1, 0)
    assert np.array_equal(p2, pm) and np.array_equal(v2, v) and np.all(a2 == 0)


def pin_leapfrog_single_body_drift(o):
    """A lone body feels no force: v is constant and x_n = x_0 + n dt v_0."""
    pm = np.array([[0.5, -1.0, 2.0, 3.0]])
    v0 = np.array([[0.25, 0.5, -0.75]])
    dt, n = 0.125, 8  # dyadic values: every step is exact
    p, v, a = o.leapfrog(pm, v0, 1e-2, dt, n)
    assert np.all(a == 0.0)
    assert np.array_equal(v, v0)
    assert np.array_equal(p[0, :3], pm[0, :3] + n * dt * v0[0])
    assert p[0, 3] == 3.0


def pin_leapfrog_two_body_by_hand(o):
    """Three steps of the half-kick + drift rule integrated here by hand with
    the closed-form two-body accelerations from the start-of-step positions."""
    x = [np.array([0.0, 0.0, 0.0]), np.array([1.0, 0.5, -0.25])]
    v = [np.array([0.0, 0.1, 0.0]), np.array([-0.2, 0.0, 0.05])]
    m = [2.0, 0.5]
    eps2, dt, steps = 0.04, 0.05, 3
    pm = np.array([[*x[0], m[0]], [*x[1], m[1]]])
    vv = np.array([v[0], v[1]])
    a = [None, None]
    for _ in range(steps):
        a = list(_two_body_expected(x[0], x[1], m[0], m[1], eps2))
        for k in range(2):
            v[k] = v[k] + 0.5 * dt * a[k]
            x[k] = x[k] + dt * v[k]
    p2, v2, a2 = o.leapfrog(pm, vv, eps2, dt, steps)
    _close(p2[:, :3], np.array(x), 1e-14, what="two-body positions")
    _close(v2, np.array(v), 1e-14, what="two-body velocities")
    _close(a2, np.array(a), 1e-14, what="two-body last-step accelerations")
    assert np.array_equal(p2[:, 3], pm[:, 3]), "masses changed"


def pin_leapfrog_from_rest_one_step(o):
    """From rest: v_1 = (dt/2) a_0 and x_1 = x_0 + (dt^2/2) a_0."""
    rng = np.random.default_rng(8)
    pm = np.zeros((30, 4))
    pm[:, :3] = rng.uniform(-1, 1, size=(30, 3))
    pm[:, 3] = rng.uniform(0.5, 1.5, size=30) / 30
    dt = 0.01
    a0 = o.accel(pm, 0.01)
    p1, v1, a1 = o.leapfrog(pm, np.zeros((30, 3)), 0.01, dt, 1)
    assert np.array_equal(a1, a0), "step acceleration differs from accel()"
    _close(v1, 0.5 * dt * a0, 1e-15, what="v1")
    _close(p1[:, :3] - pm[:, :3], 0.5 * dt * dt * a0, 1e-12, what="x1 - x0")


def pin_leapfrog_momentum_and_com(o):
    """sum m a = 0, so sum m v is constant and the centre of mass moves by
    dt * (sum m v) / M per step."""
    rng = np.random.default_rng(9)
    n = 64
    pm = np.zeros((n, 4))
    pm[:, :3] = rng.normal(size=(n, 3))
    pm[:, 3] = rng.uniform(0.5, 1.5, size=n)
    v0 = rng.normal(scale=0.3, size=(n, 3))
    dt, steps = 0.01, 5
    p, v, _ = o.leapfrog(pm, v0, 0.05, dt, steps)
    m = pm[:, 3:4]
    P0 = np.sum(m * v0, axis=0)
    scale = float(np.sum(m * np.abs(v)))
    assert np.max(np.abs(np.sum(m * v, axis=0) - P0)) <= 1e-13 * scale, "momentum drift"
    com0 = np.sum(m * pm[:, :3], axis=0) / m.sum()
    com = np.sum(m * p[:, :3], axis=0) / m.sum()
    _close(com - com0, steps * dt * P0 / m.sum(), 1e-10, what="centre-of-mass motion")


def pin_leapfrog_composition(o):
    """State lives entirely in (x, v): 4 steps then 6 steps equals 10 steps."""
    rng = np.random.default_rng(10)
    pm = np.zeros((25, 4))
    pm[:, :3] = rng.normal(size=(25, 3))
    pm[:, 3] = rng.uniform(0.5, 1.5, size=25)
    v0 = rng.normal(scale=0.1, size=(25, 3))
    pa, va, aa = o.leapfrog(pm, v0, 0.01, 0.02, 10)
    pb, vb, _ = o.leapfrog(pm, v0, 0.01, 0.02, 4)
    pc, vc, ac = o.leapfrog(pb, vb, 0.01, 0.02, 6)
    assert np.array_equal(pa, pc) and np.array_equal(va, vc) and np.array_equal(aa, ac)


# ---------------------------------------------------------------------------
# kick-drift-kick leapfrog pins
# ---------------------------------------------------------------------------


def pin_kdk_zero_steps(o):
    pm = np.array([[0.0, 0.0, 0.0, 1.0], [1.0, 0.0, 0.0, 1.0]])
    v = np.array([[0.1, 0.2, 0.3], [0.0, 0.0, 0.0]])
    p2, v2, a2 = o.leapfrog_kdk(pm, v, 0.01, 0.1, 0)
    assert np.array_equal(p2, pm) and np.array_equal(v2, v) and np.all(a2 == 0)


def pin_kdk_single_body_drift(o):
    pm = np.array([[0.5, -1.0, 2.0, 3.0]])
    v0 = np.array([[0.25, 0.5, -0.75]])
    p, v, a = o.leapfrog_kdk(pm, v0, 1e-2, 0.125, 8)
    assert np.all(a == 0.0) and np.array_equal(v, v0)
    assert np.array_equal(p[0, :3], pm[0, :3] + 8 * 0.125 * v0[0])


def pin_kdk_two_body_by_hand(o):
    """Three kick-drift-kick steps integrated here from the closed-form
    two-body accelerations."""
    x = [np.array([0.0, 0.0, 0.0]), np.array([1.0, 0.5, -0.25])]
    v = [np.array([0.0, 0.1, 0.0]), np.array([-0.2, 0.0, 0.05])]
    m = [2.0, 0.5]
    eps2, dt, steps = 0.04, 0.05, 3
    pm = np.array([[*x[0], m[0]], [*x[1], m[1]]])
    vv = np.array([v[0], v[1]])
    a = list(_two_body_expected(x[0], x[1], m[0], m[1], eps2))
    for _ in range(steps):
        for k in range(2):
            v[k] = v[k] + 0.5 * dt * a[k]
            x[k] = x[k] + dt * v[k]
        a = list(_two_body_expected(x[0], x[1], m[0], m[1], eps2))
        for k in range(2):
            v[k] = v[k] + 0.5 * dt * a[k]
    p2, v2, a2 = o.leapfrog_kdk(pm, vv, eps2, dt, steps)
    _close(p2[:, :3], np.array(x), 1e-14, what="kdk two-body positions")
    _close(v2, np.array(v), 1e-14, what="kdk two-body velocities")
    _close(a2, np.array(a), 1e-14, what="kdk two-body final accelerations")


def pin_kdk_time_reversible(o):
    """Kick-drift-kick is time-symmetric: run forward, reverse the velocities,
    run the same number of steps, reverse again: the start comes back."""
    rng = np.random.default_rng(11)
    n = 24
    pm = np.zeros((n, 4))
    pm[:, :3] = rng.normal(size=(n, 3))
    pm[:, 3] = rng.uniform(0.5, 1.5, size=n) / n
    v0 = rng.normal(scale=0.2, size=(n, 3))
    p1, v1, _ = o.leapfrog_kdk(pm, v0, 0.02, 0.01, 40)
    p2, v2, _ = o.leapfrog_kdk(p1, -v1, 0.02, 0.01, 40)
    _close(p2[:, :3], pm[:, :3], 1e-11, what="reversed positions")
    _close(-v2, v0, 1e-10, what="reversed velocities")


def _circular_pair(eps2):
    """Two masses 1/2 at separation 1 on a circular orbit of the softened
    force: omega^2 = 2 m / (D^2 + eps2)^{3/2}, radius D/2."""
    m, D = 0.5, 1.0
    R = D / 2
    w = math.sqrt(2 * m / (D * D + eps2) ** 1.5)
    pm = np.array([[R, 0.0, 0.0, m], [-R, 0.0, 0.0, m]])
    v = np.array([[0.0, w * R, 0.0], [0.0, -w * R, 0.0]])
    return pm, v, w, R


def pin_kdk_second_order(o):
    """Global error on a circular orbit falls 4x per halving of dt."""
    eps2, T = 0.01, 2.0
    pm, v, w, R = _circular_pair(eps2)
    exact = np.array([R * math.cos(w * T), R * math.sin(w * T), 0.0])
    errs = []
    for steps in (50, 100, 200):
        p, _, _ = o.leapfrog_kdk(pm, v, eps2, T / steps, steps)
        errs.append(float(np.linalg.norm(p[0, :3] - exact)))
    r1, r2 = errs[0] / errs[1], errs[1] / errs[2]
    assert 3.6 < r1 < 4.4 and 3.6 < r2 < 4.4, (errs, r1, r2)


def pin_kdk_matches_half_kick_drift_then_kick(o):
    """One KDK step = the half-kick + drift step, then a half kick with the
    acceleration at the new positions."""
    rng = np.random.default_rng(12)
    pm = np.zeros((30, 4))
    pm[:, :3] = rng.normal(size=(30, 3))
    pm[:, 3] = rng.uniform(0.5, 1.5, size=30)
    v0 = rng.normal(scale=0.1, size=(30, 3))
    pk, vk, ak = o.leapfrog_kdk(pm, v0, 0.01, 0.02, 1)
    ph, vh, _ = o.leapfrog(pm, v0, 0.01, 0.02, 1)
    assert np.array_equal(pk, ph), "KDK drift differs from the half-kick + drift step"
    a1 = o.accel(ph, 0.01)
    assert np.array_equal(ak, a1)
    _close(vk, vh + 0.5 * 0.02 * a1, 1e-15, what="closing half kick")


def pin_kdk_momentum(o):
    rng = np.random.default_rng(13)
    n = 40
    pm = np.zeros((n, 4))
    pm[:, :3] = rng.normal(size=(n, 3))
    pm[:, 3] = rng.uniform(0.5, 1.5, size=n)
    v0 = rng.normal(scale=0.3, size=(n, 3))
    _, v, _ = o.leapfrog_kdk(pm, v0, 0.05, 0.01, 6)
    m = pm[:, 3:4]
    P0 = np.sum(m * v0, axis=0)
    assert np.max(np.abs(np.sum(m * v, axis=0) - P0)) <= 1e-13 * float(np.sum(m * np.abs(v)))


KDK_PINS = [
    pin_kdk_zero_steps,
    pin_kdk_single_body_drift,
    pin_kdk_two_body_by_hand,
    pin_kdk_time_reversible,
    pin_kdk_second_order,
    pin_kdk_matches_half_kick_drift_then_kick,
    pin_kdk_momentum,
]

# ---------------------------------------------------------------------------
# point-shader pins ("CUDA N-Body Simulation" §4.3)
# ---------------------------------------------------------------------------


def pin_render_ndc_equals_x_over_limit(o):
    """The section states the affine map as x_NDC = x / X; the shader writes
    2 (x + X) / (2 X) - 1.  The two agree, and the box corners map to +-1."""
    rng = np.random.default_rng(14)
    pm = np.zeros((100, 4))
    lim = (2.0, 0.5, 300.0)
    for c in range(3):
        pm[:, c] = rng.uniform(-1.5, 1.5, size=100) * lim[c]
    pm[:, 3] = rng.uniform(1.0, 2.0, size=100)
    ndc, _ = o.render_points(pm, lim, 1.0, 2.0)
    _close(ndc[:, :3], pm[:, :3] / np.array(lim), 1e-15, what="ndc = x / X")
    assert np.all(ndc[:, 3] == 1.0)
    corners = np.array([[2.0, -0.5, 300.0, 1.0], [-2.0, 0.5, -300.0, 1.0], [0, 0, 0, 1.0]])
    ndc, _ = o.render_points(corners, lim, 1.0, 2.0)
    assert np.array_equal(ndc[:, :3], [[1, -1, 1], [-1, 1, -1], [0, 0, 0]])


def pin_render_colour_ramp(o):
    """Lightest mass is green, heaviest red, the midpoint half of each, and
    the colour is affine in the mass (GLSL mix)."""
    pm = np.zeros((5, 4))
    pm[:, 3] = [1e5, 1e9, 0.5 * (1e5 + 1e9), 1e5 + 0.25 * (1e9 - 1e5), 2e9]
    _, rgba = o.render_points(pm, (1.0, 1.0, 1.0), 1e5, 1e9)
    _close(rgba[0], [0, 1, 0, 1], 1e-15, what="min mass")
    _close(rgba[1], [1, 0, 0, 1], 1e-15, what="max mass")
    _close(rgba[2], [0.5, 0.5, 0, 1], 1e-15, what="mid mass")
    _close(rgba[3], [0.25, 0.75, 0, 1], 1e-15, what="quarter mass")
    w = (2e9 - 1e5) / (1e9 - 1e5)  # no clamp: extrapolates beyond red
    _close(rgba[4], [w, 1 - w, 0, 1], 1e-15, what="beyond max mass")


RENDER_PINS = [pin_render_ndc_equals_x_over_limit, pin_render_colour_ramp]


# ---------------------------------------------------------------------------
# 2-D cutoff neighbour-list pins ("CUDA编程（九）原子函数的合理使用" §3)
# ---------------------------------------------------------------------------


def _lattice(k):
    """k x k unit square lattice, row-major indices, integer coordinates."""
    ix, iy = np.meshgrid(np.arange(k), np.arange(k), indexing="xy")
    return ix.ravel().astype(np.float32), iy.ravel().astype(np.float32)


def _lattice_neighbours(k, offsets):
    out = []
    for y in range(k):
        for x in range(k):
            nb = [(y + dy) * k + (x + dx) for dx, dy in offsets
                  if 0 <= x + dx < k and 0 <= y + dy < k]
            out.append(sorted(nb))
    return out


def pin_neighbors_square_lattice(o):
    """Unit lattice: cutoff 1.2 keeps the 4 edge neighbours, cutoff 1.5 adds
    the 4 diagonals (sqrt 2), cutoff exactly 2 adds nothing more because the
    test is strict (d^2 = 4 is not < 4).  Lists come in ascending order."""
    k = 7
    x, y = _lattice(k)
    four = [(1, 0), (-1, 0), (0, 1), (0, -1)]
    eight = four + [(1, 1), (1, -1), (-1, 1), (-1, -1)]
    for cutoff, offs in [(1.2, four), (1.5, eight), (2.0, eight)]:
        nn, nl = o.neighbors_2d(x, y, cutoff, 12)
        want = _lattice_neighbours(k, offs)
        for i in range(k * k):
            assert nn[i] == len(want[i]), (cutoff, i, nn[i], want[i])
            assert list(nl[:nn[i], i]) == want[i], (cutoff, i)
            assert np.all(nl[nn[i]:, i] == -1)


def pin_neighbors_symmetric(o):
    rng = np.random.default_rng(15)
    x = (8 * rng.random(300)).astype(np.float32)
    y = (8 * rng.random(300)).astype(np.float32)
    nn, nl = o.neighbors_2d(x, y, 1.1, 64)
    assert nn.max() < 64
    pairs = {(i, int(j)) for i in range(300) for j in nl[:nn[i], i]}
    assert all((j, i) in pairs for i, j in pairs), "neighbour relation not symmetric"
    assert all(i != j for i, j in pairs), "a point is its own neighbour"


def _half_loop_lists(x, y, cutoff, mn):
    """The page's CPU algorithm, restated in pure Python with float32 scalars:
    n2 > n1 only, and every hit is appended to both lists."""
    n = len(x)
    c2 = np.float32(cutoff) * np.float32(cutoff)
    lists = [[] for _ in range(n)]
    for n1 in range(n):
        for n2 in range(n1 + 1, n):
            x12 = np.float32(x[n2] - x[n1])
            y12 = np.float32(y[n2] - y[n1])
            d2 = np.float32(np.float32(x12 * x12) + np.float32(y12 * y12))
            if d2 < c2:
                lists[n1].append(n2)
                lists[n2].append(n1)
    nn = np.array([len(l) for l in lists], dtype=np.int32)
    nl = np.full((mn, n), -1, dtype=np.int32)
    for i, l in enumerate(lists):
        for k, j in enumerate(l[:mn]):
            nl[k, i] = j
    return nn, nl


def pin_neighbors_match_half_loop_algorithm(o):
    rng = np.random.default_rng(16)
    for n, cutoff, mn in [(2, 5.0, 3), (60, 1.9, 10), (150, 1.9, 4)]:
        x = (6 * rng.random(n)).astype(np.float32)
        y = (6 * rng.random(n)).astype(np.float32)
        nn, nl = o.neighbors_2d(x, y, cutoff, mn)
        wn, wl = _half_loop_lists(x, y, cutoff, mn)
        assert np.array_equal(nn, wn) and np.array_equal(nl, wl), (n, cutoff, mn)


def pin_neighbors_truncation_and_duplicates(o):
    """20 points packed in a small circle: each has 19 neighbours (two of them
    coincide and are each other's neighbour, never their own); the list keeps
    the 10 lowest indices."""
    th = np.linspace(0.0, 2 * np.pi, 19, endpoint=False)
    x = np.concatenate([0.1 * np.cos(th), [0.1]]).astype(np.float32)
    y = np.concatenate([0.1 * np.sin(th), [0.0]]).astype(np.float32)  # last = copy of point 0
    nn, nl = o.neighbors_2d(x, y, 1.0, 10)
    assert np.all(nn == 19)
    for i in range(20):
        assert list(nl[:, i]) == [j for j in range(20) if j != i][:10]
    far = np.array([0.0, 100.0], dtype=np.float32)
    nn, nl = o.neighbors_2d(far, far, 1.0, 3)
    assert np.all(nn == 0) and np.all(nl == -1)


def pin_neighbors_sampled_rows_match_full(o):
    rng = np.random.default_rng(17)
    x = (10 * rng.random(400)).astype(np.float32)
    y = (10 * rng.random(400)).astype(np.float32)
    nn, nl = o.neighbors_2d(x, y, 1.9, 6)
    idx = np.array([399, 0, 17, 17, 200])
    sn, sl = o.neighbors_2d(x, y, 1.9, 6, idx=idx)
    assert np.array_equal(sn, nn[idx]) and np.array_equal(sl, nl[:, idx])


NEIGHBOR_PINS = [pin_neighbors_sampled_rows_match_full, pin_neighbors_square_lattice, pin_neighbors_symmetric,
                 pin_neighbors_match_half_loop_algorithm, pin_neighbors_truncation_and_duplicates]

ACCEL_PINS = [
    pin_two_body_closed_form,
    pin_ring_axis_closed_form,
    pin_cube_centre_zero,
    pin_single_body_and_coincident_zero,
    pin_momentum_antisymmetry,
    pin_scaling_homogeneity,
    pin_mass_linearity,
    pin_translation_invariance,
    pin_bruteforce_fsum,
    pin_sampled_rows_match_full,
]
def pin_step_sampled_rows_match_full(o):
    """The sampled step's rows are the full one-step leapfrog's rows, bit for
    bit, in any order and with repeats; masses are carried unchanged."""
    rng = np.random.default_rng(11)
    pm = np.zeros((150, 4))
    pm[:, :3] = rng.normal(size=(150, 3))
    pm[:, 3] = rng.uniform(0.1, 2.0, size=150)
    v = rng.normal(size=(150, 3))
    fp, fv, fa = o.leapfrog(pm, v, 1e-2, 0.01, 1)
    idx = np.array([149, 3, 3, 0, 77])
    sp, sv, sa = o.step_sampled(pm, v, 1e-2, 0.01, idx)
    assert np.array_equal(sp, fp[idx]) and np.array_equal(sv, fv[idx])
    assert np.array_equal(sa, fa[idx])
    assert np.array_equal(sp[:, 3], pm[idx, 3])


LEAPFROG_PINS = [
    pin_step_sampled_rows_match_full,
    pin_leapfrog_zero_steps,
    pin_leapfrog_single_body_drift,
    pin_leapfrog_two_body_by_hand,
    pin_leapfrog_from_rest_one_step,
    pin_leapfrog_momentum_and_com,
    pin_leapfrog_composition,
]
ALL_PINS = ACCEL_PINS + LEAPFROG_PINS + KDK_PINS + RENDER_PINS + NEIGHBOR_PINS


def failing_pins(o) -> list[str]:
    """Names of the pins this oracle fails (any exception counts as a failure)."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception:  # noqa: BLE001 - a crash is as good as a failure here
            bad.append(pin.__name__)
    return bad
