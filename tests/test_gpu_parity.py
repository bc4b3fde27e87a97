"""CUDA path against the FP64 oracle, element by element, through the C ABI.

Workloads: the five benchmark configurations (full oracle up to 131072
bodies, 4096 seeded sampled bodies above), every force-pass path forced on
the same inputs, ragged sizes around every tile and block width, the
degenerate cases (one body, coincident bodies, zero steps), determinism and
step composition.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import (ACC_TOL, EPS32, POS_TOL, VEL_TOL, displacement_err, gpu_accel, gpu_leapfrog,
                    rel_err)

pytestmark = pytest.mark.gpu

PATHS = [(0, 0), (1, 0), (2, 0), (2, 1), (2, 3), (2, 7), (3, 0), (3, 1), (3, 5), (4, 0)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    from all_pairs_body_gb300 import build as nbuild
    nbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()


_REF = {}


def oracle_accel_cached(w):
    key = (w.name, w.n)
    if key not in _REF:
        _REF[key] = oracle.accel(w.pos_mass, w.eps2, idx=w.sample)
    return _REF[key]


def check_accel(w, path=0, split=0, tol=ACC_TOL):
    a = gpu_accel(w.pos_mass, w.eps2, path, split)
    assert np.all(np.isfinite(a))
    assert np.all(a[:, 3] == 0.0), "accel.w must be 0"
    ref = oracle_accel_cached(w)
    got = a if w.sample is None else a[w.sample]
    err = rel_err(got, ref)
    assert err <= tol, f"{w.name} path={path} split={split}: err {err:.3e}"
    return a, err


# ---------------------------------------------------------------------------
# the benchmark workloads
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("name", ["uniform-cube-1024", "plummer-16384", "two-plummer-131072",
                                  "ball-lognormal-1048576", "cube-sweep-1000",
                                  "cube-sweep-4097", "cube-sweep-65537", "cube-sweep-500000",
                                  "cube-sweep-4194304"])
def test_accel_workload(name):
    check_accel(W.by_name(name))


def test_uniform_cube_1024_step():
    w = W.uniform_cube_1024()
    p, v, a = gpu_leapfrog(w.pos_mass, w.vel, w.eps2, w.dt, w.steps)
    rp, rv, ra = oracle.leapfrog(w.pos_mass, w.vel, w.eps2, w.dt, w.steps)
    assert rel_err(a, ra) <= ACC_TOL
    assert rel_err(v, rv) <= VEL_TOL
    assert rel_err(p, rp) <= POS_TOL
    # from rest: v_1 = (dt/2) a_0 exactly in the oracle's arithmetic
    assert rel_err(v, 0.5 * w.dt * ra) <= VEL_TOL


@pytest.mark.parametrize("name,moving", [("ball-lognormal-1048576", False),
                                         ("ball-lognormal-1048576", True),
                                         ("cube-sweep-4194304", True)])
def test_full_size_step_sampled(name, moving):
    """One leapfrog step at the full sizes, through the default plan (the pair
    kernel in chunks of reaction rows, the chunked accumulation and the fused
    half-kick and drift), checked on the workload's 4096 sampled bodies against
    the oracle's step of those rows.  The bodies start at rest, as the benchmark
    runs them, or with seeded velocities so that the drift moves them."""
    import all_pairs_body_gb300 as nb
    w = W.by_name(name)
    v0 = W.random_velocities(w.n, 4100) if moving else w.vel
    p, v, a = gpu_leapfrog(w.pos_mass, v0, w.eps2, w.dt, 1)
    plan = nb.last_plan()
    assert plan["path"] == nb.PATH_PAIRS and plan["chunks"] > 1
    rp, rv, ra = oracle.step_sampled(w.pos_mass, v0, w.eps2, w.dt, w.sample)
    s = w.sample
    assert rel_err(a[s], ra) <= ACC_TOL
    assert rel_err(v[s], rv) <= VEL_TOL
    assert rel_err(p[s], rp) <= POS_TOL
    assert displacement_err(p[s], rp, w.pos_mass[s], 1) <= 1e-3
    # the kick alone: v - v0 = (dt/2) a, beyond one float32 ulp of |v|
    dv = v[s, :3].astype(np.float64) - v0[s, :3]
    dv_ref = rv - v0[s, :3]
    floor = EPS32 * np.sqrt(3.0) * np.linalg.norm(rv, axis=1)
    excess = np.maximum(np.linalg.norm(dv - dv_ref, axis=1) - floor, 0.0)
    assert excess.max() <= 1e-3 * np.sqrt(np.mean(np.sum(dv_ref * dv_ref, axis=1)))
    assert np.array_equal(p[:, 3], w.pos_mass[:, 3]), "masses changed"
    assert np.array_equal(v[:, 3], v0[:, 3]), "vel.w changed"


@pytest.mark.parametrize("name", ["plummer-16384", "two-plummer-131072"])
def test_trajectory_10_steps(name):
    w = W.by_name(name)
    p, v, a = gpu_leapfrog(w.pos_mass, w.vel, w.eps2, w.dt, w.steps)
    rp, rv, ra = oracle.leapfrog(w.pos_mass, w.vel, w.eps2, w.dt, w.steps)
    assert rel_err(p, rp) <= POS_TOL
    assert rel_err(v, rv) <= VEL_TOL
    assert rel_err(a, ra) <= ACC_TOL
    # displacement over the run (a far stricter view of the positions), beyond
    # the float32 storage floor of one ulp of |x| per step
    assert displacement_err(p, rp, w.pos_mass, w.steps) <= 1e-3
    assert np.array_equal(p[:, 3], w.pos_mass[:, 3]), "masses changed"
    assert np.array_equal(v[:, 3], w.vel[:, 3]), "vel.w changed"


@pytest.mark.parametrize("path", [0, 3])
def test_trajectory_100_steps(path):
    """C2's bodies for 100 steps in one call (200 kernels chained as
    programmatic dependents on the pair path, 100 one-kernel passes and a copy
    on the warp path), against the oracle's trajectory."""
    w = W.plummer_16384()
    p, v, a = gpu_leapfrog(w.pos_mass, w.vel, w.eps2, w.dt, 100, path)
    if "trajectory_100" not in _REF:
        _REF["trajectory_100"] = oracle.leapfrog(w.pos_mass, w.vel, w.eps2, w.dt, 100)
    rp, rv, ra = _REF["trajectory_100"]
    assert rel_err(p, rp) <= POS_TOL
    assert rel_err(v, rv) <= VEL_TOL
    assert rel_err(a, ra) <= ACC_TOL
    assert displacement_err(p, rp, w.pos_mass, 100) <= 1e-3


# ---------------------------------------------------------------------------
# every path on the same inputs
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("path,split", PATHS)
@pytest.mark.parametrize("n", [1000, 4097, 16384, 20000])
def test_paths_accel(n, path, split):
    w = W.cube_sweep(n) if n != 16384 else W.plummer_16384()
    check_accel(w, path, split)


@pytest.mark.parametrize("path,split", PATHS)
def test_paths_leapfrog(path, split):
    n = 5000
    pm = W.random_bodies(n, 21)
    v = W.random_velocities(n, 21)
    p, vv, a = gpu_leapfrog(pm, v, 1e-3, 1e-3, 3, path, split)
    rp, rv, ra = oracle.leapfrog(pm, v, 1e-3, 1e-3, 3)
    assert rel_err(a, ra) <= ACC_TOL
    assert rel_err(vv, rv) <= VEL_TOL
    assert rel_err(p, rp) <= POS_TOL
    assert np.array_equal(vv[:, 3], v[:, 3]) and np.array_equal(p[:, 3], pm[:, 3])


RAGGED = [1, 2, 3, 7, 8, 9, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 513,
          1023, 1025, 2047, 2049, 4095, 4097]


@pytest.mark.parametrize("n", RAGGED)
@pytest.mark.parametrize("path,split", [(0, 0), (1, 0), (2, 0), (2, 3), (3, 0), (3, 2), (4, 0)])
def test_ragged_sizes(n, path, split):
    pm = W.random_bodies(n, 1000 + n)
    a = gpu_accel(pm, 1e-2, path, split)
    ref = oracle.accel(pm, 1e-2)
    if n == 1:
        assert np.all(a == 0.0)
    else:
        assert rel_err(a, ref) <= ACC_TOL, (n, path, split)


# ---------------------------------------------------------------------------
# closed forms and invariants on the GPU
# ---------------------------------------------------------------------------


def test_two_body_closed_form():
    pm = np.array([[0.0, 0.0, 0.0, 2.0], [1.0, 0.5, -0.25, 3.0]], dtype=np.float32)
    a = gpu_accel(pm, 0.01).astype(np.float64)
    r = pm[1, :3].astype(np.float64) - pm[0, :3]
    f = (r @ r + 0.01) ** -1.5
    assert np.allclose(a[0, :3], 3.0 * f * r, rtol=2e-6, atol=0)
    assert np.allclose(a[1, :3], -2.0 * f * r, rtol=2e-6, atol=0)


def test_coincident_and_single_bodies():
    pm = np.array([[0.5, 0.5, 0.5, 1.0]] * 5, dtype=np.float32)
    for path, split in [(0, 0), (1, 0), (3, 0), (4, 0)]:
        assert np.all(gpu_accel(pm, 1e-3, path, split)[:, :3] == 0.0)


def test_momentum_invariant():
    w = W.plummer_16384()
    a = gpu_accel(w.pos_mass, w.eps2).astype(np.float64)
    m = w.pos_mass[:, 3:4].astype(np.float64)
    net = np.abs(np.sum(m * a[:, :3], axis=0)).max()
    assert net <= 1e-5 * float(np.sum(m[:, 0] * np.linalg.norm(a[:, :3], axis=1)))


# ---------------------------------------------------------------------------
# determinism, composition, streams
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("path,split", [(0, 0), (1, 0), (2, 5), (3, 0), (4, 0)])
def test_bitwise_deterministic(path, split):
    pm = W.cube_sweep(65537).pos_mass
    a1 = gpu_accel(pm, 1e-3, path, split)
    a2 = gpu_accel(pm, 1e-3, path, split)
    assert np.array_equal(a1, a2)


@pytest.mark.parametrize("n", [3000, 40000])
def test_steps_compose(n):
    pm = W.random_bodies(n, 5)
    v = W.random_velocities(n, 5)
    p10, v10, a10 = gpu_leapfrog(pm, v, 1e-3, 1e-3, 10)
    p4, v4, _ = gpu_leapfrog(pm, v, 1e-3, 1e-3, 4)
    p46, v46, a46 = gpu_leapfrog(p4, v4, 1e-3, 1e-3, 6)
    assert np.array_equal(p10, p46) and np.array_equal(v10, v46) and np.array_equal(a10, a46)


# (n, path, split): the one-kernel warp pass and the one-sided paths
# (ping-pong, and a copy into the caller's buffer after an odd number of
# drifts), the warp pass with slices and the pair path (drift in place in the
# finishing kernel)
DRIFT_CASES = [(1024, 0, 0, "warp", 0), (4097, 3, 1, "warp", 0), (3000, 3, 5, "warp", 1),
               (20000, 4, 0, "pairs", 1), (20000, 1, 0, "tiled", 0), (20000, 2, 3, "tiled", 1)]


@pytest.mark.parametrize("n,path,split,kind,second", DRIFT_CASES)
def test_drift_buffers_by_path(n, path, split, kind, second):
    """One, two and three steps per call on every way the new positions reach
    the caller's buffer, against the oracle; three one-step calls give the
    bits of one three-step call; the kick-drift-kick form the same."""
    import all_pairs_body_gb300 as nb
    pm = W.random_bodies(n, 8100 + n)
    v = W.random_velocities(n, 8100 + n)
    for steps in (1, 2, 3):
        p, vv, a = gpu_leapfrog(pm, v, 1e-3, 1e-3, steps, path, split)
        plan = nb.last_plan()
        assert plan["path"] == {"warp": nb.PATH_WARP, "pairs": nb.PATH_PAIRS}.get(
            kind, plan["path"]) and plan["second_pass"] == second
        rp, rv, ra = oracle.leapfrog(pm, v, 1e-3, 1e-3, steps)
        assert rel_err(a, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL
        assert rel_err(p, rp) <= POS_TOL
        assert displacement_err(p, rp, pm, steps) <= 1e-3
        assert np.array_equal(p[:, 3], pm[:, 3]) and np.array_equal(vv[:, 3], v[:, 3])
    p1, v1, a1 = pm, v, None
    for _ in range(3):
        p1, v1, a1 = gpu_leapfrog(p1, v1, 1e-3, 1e-3, 1, path, split)
    assert np.array_equal(p1, p) and np.array_equal(v1, vv) and np.array_equal(a1, a)
    for steps in (1, 3):
        p, vv, a = gpu_kdk(pm, v, 1e-3, 1e-3, steps, path, split)
        rp, rv, ra = oracle.leapfrog_kdk(pm, v, 1e-3, 1e-3, steps)
        assert rel_err(a, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL
        assert displacement_err(p, rp, pm, steps) <= 1e-3


def test_zero_steps_is_noop():
    pm = W.random_bodies(100, 2)
    v = W.random_velocities(100, 2)
    p, vv, a = gpu_leapfrog(pm, v, 1e-3, 1e-3, 0)
    assert np.array_equal(p, pm) and np.array_equal(vv, v) and np.all(np.isnan(a))


def test_side_stream_matches_default_stream():
    import torch
    import all_pairs_body_gb300 as nb
    pm = torch.from_numpy(W.cube_sweep(4097).pos_mass).cuda()
    ref = nb.accel(pm, 1e-3)
    nb.sync()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = nb.accel(pm, 1e-3)
        nb.sync()
    assert torch.equal(out, ref)


def test_plan_is_consistent():
    import all_pairs_body_gb300 as nb
    for n in (1000, 16384, 1048576):
        p = nb.plan(n)
        assert p["sms"] > 0 and p["grid"] >= 1 and p["threads"] % 32 == 0
        assert p["launches_accel"] >= 1
    p = nb.plan(1048576, path=nb.PATH_TILED)
    assert p["second_pass"] == 0 and p["grid"] * p["bodies_per_cta"] >= 1048576
    # the warp kernel: 8 targets per CTA up to 4096 bodies, 6 above
    for n, kw in ((1000, 8), (4096, 8), (4097, 6), (16383, 6)):
        p = nb.plan(n)
        assert p["path"] == nb.PATH_WARP and p["bodies_per_cta"] == kw, (n, p)
        assert p["grid"] == -(-n // kw) and p["second_pass"] == 0


def test_plan_shape_follows_streamk_model():
    """Above the warp kernel the one-sided stream-K plan takes the 512- or the
    256-source shape, whichever gives the slowest CTA less work:
    ceil(units / grid) tiles of tj sources at the shape's relative speed (1
    and 0.973)."""
    import all_pairs_body_gb300 as nb
    shapes = ((512, 1.0), (256, 0.973))
    for n in list(range(24577, 140000, 4099)) + [262144, 500000, 1048576, 4194304]:
        p = nb.plan(n, path=nb.PATH_SPLIT)
        assert p["bodies_per_cta"] == 2560
        cost = []
        for tj, speed in shapes:
            units = -(-n // 2560) * -(-n // tj)
            grid = min(units, p["sms"])
            cost.append(-(-units // grid) * tj / speed)
        want = shapes[0][0] if cost[0] <= cost[1] else shapes[1][0]
        assert p["tile"] == want, (n, cost, p)
        assert p["grid"] == min(p["units"], p["sms"])
    if nb.plan(32768)["sms"] == 152:  # the measured cases on a 152-SM GPU
        assert [nb.plan(n, path=nb.PATH_SPLIT)["tile"]
                for n in (32768, 49152, 65537, 81920, 1048576)] == [256, 512, 256, 512, 512]


def pair_units(n, block, tj=512):
    """Units of the pair path: block I meets the tiles of itself and of every
    later block."""
    nb_, nt = -(-n // block), -(-n // tj)
    return sum(nt - (block // tj) * i for i in range(nb_))


PAIR_SHAPES = ((4096, 512, 1.0), (3584, 512, 0.9977), (3072, 512, 0.9726), (2560, 512, 0.9736),
               (2048, 512, 0.9539), (2048, 256, 0.9602))  # targets per CTA, tile, speed


def test_plan_pairs_path(monkeypatch):
    """Above the warp kernel the pair path, with the shape whose slowest CTA
    has the least work: ceil(units / grid) units of B x TJ pairs at the
    shape's relative speed."""
    import all_pairs_body_gb300 as nb
    assert nb.plan(16383)["path"] == nb.PATH_WARP
    for n in list(range(16384, 140000, 5003)) + [262144, 1048576, 2000000]:
        p = nb.plan(n)
        assert p["path"] == nb.PATH_PAIRS and p["second_pass"] == 1
        cost = []
        for block, tj, speed in PAIR_SHAPES:
            units = pair_units(n, block, tj)
            cost.append(-(-units // min(units, p["sms"])) * block * tj / speed)
        block, tj, _ = PAIR_SHAPES[cost.index(min(cost))]
        assert p["bodies_per_cta"] == block and p["tile"] == tj, (n, cost, p)
        assert p["units"] == pair_units(n, block, tj)
        assert p["grid"] == min(p["units"], p["sms"])
        chunks = pair_chunks(n, block, 1 << 30, tj)
        assert p["launches_accel"] == (2 if chunks == 1 else 2 * chunks + 1)
        assert p["chunks"] == chunks and p["react_bytes"] <= 1 << 30
    if nb.plan(32768)["sms"] == 152:
        assert nb.plan(1048576)["bodies_per_cta"] == 4096
    # 4M bodies need ~39 GB of reaction rows: the pass runs in chunks of
    # i-blocks whose rows fit 1 GiB, one accumulation pass per chunk
    p = nb.plan(4194304)
    assert p["path"] == nb.PATH_PAIRS
    assert p["launches_accel"] == 2 * pair_chunks(4194304, p["bodies_per_cta"], 1 << 30,
                                                  p["tile"]) + 1
    monkeypatch.setenv("NBODY_PAIRS_MAX_BYTES", "1000")
    p = nb.plan(65537)
    assert p["path"] == nb.PATH_PAIRS
    assert p["launches_accel"] == 2 * -(-65537 // p["bodies_per_cta"]) + 1  # a block per chunk


def pair_chunks(n, block, cap, tj=512):
    """Chunks of consecutive i-blocks whose reaction rows (TJ float4 per
    unit) fit `cap` bytes, one block at least."""
    nb_, nt, tb = -(-n // block), -(-n // tj), block // tj
    chunks, acc = 1, 0
    for i in range(nb_):
        u = nt - tb * i
        if acc > 0 and (acc + u) * tj * 16 > cap:
            chunks, acc = chunks + 1, 0
        acc += u
    return chunks


@pytest.mark.parametrize("n,cap", [(20000, 1), (30001, 300000), (65537, 2000000),
                                   (65537, 50000000)])
def test_pair_path_in_chunks(n, cap, monkeypatch):
    """The pair path with its reaction rows split into chunks of i-blocks
    (forced by a small scratch cap) against the oracle, for accelerations, a
    leapfrog step and a kick-drift-kick step; chunked runs are deterministic."""
    import all_pairs_body_gb300 as nb
    monkeypatch.setenv("NBODY_PAIRS_MAX_BYTES", str(cap))
    p = nb.plan(n, path=nb.PATH_PAIRS)
    chunks = pair_chunks(n, p["bodies_per_cta"], max(cap, p["tile"] * 16), p["tile"])
    assert p["launches_accel"] == (2 * chunks + 1 if chunks > 1 else 2)
    pm = W.random_bodies(n, 6000 + n)
    a = gpu_accel(pm, 1e-3, path=4)
    assert rel_err(a, oracle.accel(pm, 1e-3)) <= ACC_TOL
    assert np.array_equal(a, gpu_accel(pm, 1e-3, path=4))
    v = W.random_velocities(n, 6000 + n)
    pp, vv, aa = gpu_leapfrog(pm, v, 1e-3, 1e-3, 2, path=4)
    rp, rv, ra = oracle.leapfrog(pm, v, 1e-3, 1e-3, 2)
    assert rel_err(aa, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL and rel_err(pp, rp) <= POS_TOL


# block edges of the pair shapes (2048, 2560, 3072 or 3584 targets, 512-source
# tiles): one block, a block and one body, ragged tiles, several blocks
@pytest.mark.parametrize("n", [511, 512, 513, 2047, 2048, 2049, 2559, 2560, 2561, 3071, 3072,
                               3073, 3583, 3584, 3585, 4095, 4096, 4097, 5121, 6145, 7169,
                               7681, 9217, 12801, 30001])
def test_pair_path_block_edges(n):
    pm = W.random_bodies(n, 4000 + n)
    a = gpu_accel(pm, 1e-3, path=4)
    assert np.all(a[:, 3] == 0.0)
    assert rel_err(a, oracle.accel(pm, 1e-3)) <= ACC_TOL, n


def test_every_path_gives_zero_for_coincident_bodies():
    """All bodies at one point: every term is m_j * 0 * d^(-3/2), exactly zero,
    across and inside i-blocks, on every path (the pair path's reactions too)."""
    pm = np.zeros((20000, 4), dtype=np.float32)
    pm[:, :3] = (0.25, -0.5, 0.75)
    pm[:, 3] = np.linspace(0.5, 1.5, 20000, dtype=np.float32) / 20000
    for path, split in [(0, 0), (2, 0), (3, 0), (4, 0)]:
        assert np.all(gpu_accel(pm, 1e-3, path, split)[:, :3] == 0.0), (path, split)


def test_pair_path_two_distant_clusters():
    """Two clusters of half the mass, 5 apart: each body's field is dominated
    by its own cluster (RMS ~50), the other adds a pull of ~0.02 along x. The
    forces inside a cluster cancel in its mean (action = -reaction), so the
    near cluster's mean acceleration is the far cluster's pull, 0.5 / 5^2 to
    within the clusters' size — a figure far below each body's own field that
    the pair path must keep as the oracle does."""
    rng = np.random.default_rng(31)
    n = 30000
    pos = rng.normal(scale=0.05, size=(n, 3))
    pos[n // 2:, 0] += 5.0
    pm = np.empty((n, 4), dtype=np.float32)
    pm[:, :3] = pos
    pm[:, 3] = 1.0 / n
    a = gpu_accel(pm, 1e-4, path=4).astype(np.float64)
    ref = oracle.accel(pm, 1e-4)
    assert rel_err(a, ref) <= ACC_TOL
    pull = 0.5 / 5.0 ** 2
    near, far = slice(0, n // 2), slice(n // 2, n)
    assert abs(ref[near, 0].mean() / pull - 1.0) < 1e-2  # the oracle's own mean
    assert abs(a[near, 0].mean() - ref[near, 0].mean()) < 1e-3 * pull
    assert abs(a[far, 0].mean() - ref[far, 0].mean()) < 1e-3 * pull


def test_pair_path_masses():
    """Zero, negative and one dominant mass: the reaction uses the target's
    own mass, so a massless target must pull on nothing."""
    pm = W.random_bodies(20000, 9)
    pm[::7, 3] = 0.0
    pm[1::11, 3] *= -1.0
    a = gpu_accel(pm, 1e-3, path=4)
    assert rel_err(a, oracle.accel(pm, 1e-3)) <= ACC_TOL
    lone = np.zeros((20000, 4), dtype=np.float32)
    lone[:, :3] = pm[:, :3]
    lone[15000, 3] = 1.0  # the only mass sits in the last block: reactions only
    a = gpu_accel(lone, 1e-3, path=4)
    assert rel_err(a, oracle.accel(lone, 1e-3)) <= ACC_TOL


# ---------------------------------------------------------------------------
# errors seen from the GPU side
# ---------------------------------------------------------------------------


def test_rejects_host_and_misaligned_pointers():
    import ctypes
    import torch
    import all_pairs_body_gb300 as nb
    L = nb.lib()
    dev = torch.zeros((64, 4), device="cuda")
    host = torch.zeros((64, 4))
    pinned = torch.zeros((64, 4)).pin_memory()
    out = torch.zeros((64, 4), device="cuda")
    P = ctypes.c_void_p
    s = P(torch.cuda.current_stream().cuda_stream)
    assert L.nbody_accel_with(P(host.data_ptr()), P(out.data_ptr()), 64, 0.1, 0, 0, s) == nb.EINVAL
    assert L.nbody_accel_with(P(pinned.data_ptr()), P(out.data_ptr()), 64, 0.1, 0, 0, s) == nb.EINVAL
    flat = torch.zeros(64 * 4 + 1, device="cuda")
    assert L.nbody_accel_with(P(flat.data_ptr() + 4), P(out.data_ptr()), 64, 0.1, 0, 0, s) == nb.EINVAL
    assert L.nbody_accel_with(P(dev.data_ptr()), P(out.data_ptr()), 64, 0.1, 0, 0, s) == nb.OK
    nb.sync()


def test_allocation_failure_is_enomem(monkeypatch):
    import torch
    import all_pairs_body_gb300 as nb
    nb.release()
    pm = torch.from_numpy(W.cube_sweep(40000).pos_mass).cuda()  # tiled plan: needs scratch
    monkeypatch.setenv("NBODY_FAULT_ALLOC", "1")
    with pytest.raises(nb.NBodyError) as ei:
        nb.accel(pm, 1e-3)
    assert ei.value.status == nb.ENOMEM
    monkeypatch.delenv("NBODY_FAULT_ALLOC")
    out = nb.accel(pm, 1e-3)
    nb.sync()
    assert torch.isfinite(out).all()


def test_bounded_wait_times_out_and_context_survives():
    import torch
    import all_pairs_body_gb300 as nb
    assert nb.selftest_timeout(50) == nb.ETIMEOUT
    nb.sync()  # status was cleared by the self test
    pm = W.cube_sweep(4097)
    a = gpu_accel(pm.pos_mass, pm.eps2)
    assert rel_err(a, oracle.accel(pm.pos_mass, pm.eps2)) <= ACC_TOL
    assert torch.cuda.is_available()


def test_status_is_per_stream():
    """An expired wait on one stream is reported by nbody_sync on that stream
    only: a clean call on a second stream syncs clean, the first stream's
    sync returns ETIMEOUT once, and both streams keep working."""
    import torch
    import all_pairs_body_gb300 as nb
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    w = W.cube_sweep(4097)
    with torch.cuda.stream(sb):
        pm = torch.from_numpy(w.pos_mass).cuda()
    torch.cuda.synchronize()
    assert nb.selftest_timeout_enqueue(50, stream=sa) == nb.OK
    out = nb.accel(pm, w.eps2, stream=sb)
    torch.cuda.synchronize()  # both streams' kernels have finished
    assert nb.lib().nbody_sync(nb._stream(sb)) == nb.OK
    assert nb.lib().nbody_sync(nb._stream(sa)) == nb.ETIMEOUT
    assert nb.lib().nbody_sync(nb._stream(sa)) == nb.OK  # read and cleared
    assert rel_err(out.cpu().numpy(), oracle.accel(w.pos_mass, w.eps2)) <= ACC_TOL
    again = nb.accel(pm, w.eps2, stream=sa)
    nb.sync(sa)
    assert torch.equal(again, out)


def test_pair_scratch_failure_falls_back_visibly(monkeypatch):
    """Where the automatic plan's pair path cannot get its reaction rows the
    call runs the one-sided plan instead, and nbody_last_plan says so."""
    import torch
    import all_pairs_body_gb300 as nb
    nb.release()
    w = W.cube_sweep(20000)
    pm = torch.from_numpy(w.pos_mass).cuda()
    ref = oracle.accel(w.pos_mass, w.eps2)
    assert nb.plan(w.n)["path"] == nb.PATH_PAIRS
    out = nb.accel(pm, w.eps2)
    nb.sync()
    assert nb.last_plan()["path"] == nb.PATH_PAIRS
    nb.release()
    monkeypatch.setenv("NBODY_FAULT_ALLOC", "pairs")
    out2 = nb.accel(pm, w.eps2)
    nb.sync()
    assert nb.plan(w.n)["path"] == nb.PATH_PAIRS  # the plan before allocation
    last = nb.last_plan()
    assert last["path"] == nb.PATH_SPLIT and last["react_bytes"] == 0
    for got in (out, out2):
        assert rel_err(got.cpu().numpy(), ref) <= ACC_TOL
    monkeypatch.delenv("NBODY_FAULT_ALLOC")
    nb.release()
    with pytest.raises(nb.NBodyError):
        nb.last_plan()  # nothing ran since the release


@pytest.mark.parametrize("n", [9000, 20000])
def test_pair_and_one_sided_terms_agree_bitwise(n):
    """Every path forms the term m_j (q q) q r of a pair the same way, and the
    pair kernel's reaction -m_i q^3 r is the exact negative of the term the
    one-sided kernels form from the other body's side.  With only two massive
    bodies (in different i-blocks) every acceleration is one term, or the sum
    of two, whatever the order of the additions, so all paths must agree bit
    for bit."""
    pm = W.random_bodies(n, 7100 + n)
    pm[:, 3] = 0.0
    pm[5, 3] = 0.7
    pm[n - 3, 3] = 1.3
    ref = oracle.accel(pm, 1e-3)
    outs = {name: gpu_accel(pm, 1e-3, path, split) for name, path, split in
            (("pairs", 4, 0), ("split", 2, 0), ("split3", 2, 3), ("tiled", 1, 0), ("warp", 3, 0),
             ("warp5", 3, 5))}
    assert rel_err(outs["pairs"], ref) <= ACC_TOL
    for name, a in outs.items():
        assert np.array_equal(a, outs["pairs"]), name


@pytest.mark.parametrize("n", [16384, 65537, 262144, 1048576, 4194304, 16777216])
def test_default_pair_scratch_is_at_most_1_gib(n):
    import all_pairs_body_gb300 as nb
    p = nb.plan(n)
    assert p["path"] == nb.PATH_PAIRS and 0 < p["react_bytes"] <= 1 << 30


# ---------------------------------------------------------------------------
# kick-drift-kick leapfrog
# ---------------------------------------------------------------------------


def gpu_kdk(pos_mass_np, vel_np, eps2, dt, steps, path=0, split=0):
    import torch
    import all_pairs_body_gb300 as nb
    pm = torch.from_numpy(np.ascontiguousarray(pos_mass_np, dtype=np.float32)).cuda()
    v = torch.from_numpy(np.ascontiguousarray(vel_np, dtype=np.float32)).cuda()
    a = torch.full_like(pm, float("nan"))
    nb.leapfrog_kdk(pm, v, a, eps2, dt, steps, path=path, split=split)
    nb.sync()
    return pm.cpu().numpy(), v.cpu().numpy(), a.cpu().numpy()


@pytest.mark.parametrize("name", ["uniform-cube-1024", "plummer-16384", "two-plummer-131072"])
def test_kdk_trajectory(name):
    w = W.by_name(name)
    steps = max(w.steps, 1)
    p, v, a = gpu_kdk(w.pos_mass, w.vel, w.eps2, w.dt, steps)
    rp, rv, ra = oracle.leapfrog_kdk(w.pos_mass, w.vel, w.eps2, w.dt, steps)
    assert rel_err(p, rp) <= POS_TOL
    assert rel_err(v, rv) <= VEL_TOL
    assert rel_err(a, ra) <= ACC_TOL
    assert displacement_err(p, rp, w.pos_mass, steps) <= 1e-3
    assert np.array_equal(p[:, 3], w.pos_mass[:, 3]) and np.array_equal(v[:, 3], w.vel[:, 3])


@pytest.mark.parametrize("path,split", PATHS)
def test_kdk_paths(path, split):
    n = 5000
    pm = W.random_bodies(n, 23)
    v = W.random_velocities(n, 23)
    p, vv, a = gpu_kdk(pm, v, 1e-3, 1e-3, 3, path, split)
    rp, rv, ra = oracle.leapfrog_kdk(pm, v, 1e-3, 1e-3, 3)
    assert rel_err(a, ra) <= ACC_TOL
    assert rel_err(vv, rv) <= VEL_TOL
    assert rel_err(p, rp) <= POS_TOL


def test_kdk_first_drift_is_the_pages_step():
    pm = W.random_bodies(3000, 24)
    v = W.random_velocities(3000, 24)
    pk, vk, ak = gpu_kdk(pm, v, 1e-3, 1e-3, 1)
    ph, vh, _ = gpu_leapfrog(pm, v, 1e-3, 1e-3, 1)
    assert np.array_equal(pk, ph)
    # the closing half kick uses the acceleration at the new positions
    assert rel_err(vk[:, :3] - vh[:, :3], 0.5e-3 * oracle.accel(ph, 1e-3)) <= 1e-3


def test_kdk_time_reversible():
    pm = W.random_bodies(4000, 25)
    v = W.random_velocities(4000, 25, scale=0.3)
    p1, v1, _ = gpu_kdk(pm, v, 1e-3, 1e-3, 20)
    back = v1.copy()
    back[:, :3] *= -1.0
    p2, v2, _ = gpu_kdk(p1, back, 1e-3, 1e-3, 20)
    moved = float(np.abs(p1[:, :3] - pm[:, :3]).max())
    assert float(np.abs(p2[:, :3] - pm[:, :3]).max()) <= 1e-3 * moved
    assert float(np.abs(-v2[:, :3] - v[:, :3]).max()) <= 1e-4 * float(np.abs(v[:, :3]).max())


# ---------------------------------------------------------------------------
# point shaders as a kernel
# ---------------------------------------------------------------------------

RENDER_TOL = 2e-6  # float32 arithmetic on values of order one


def gpu_render(pm_np, lim, min_w, max_w):
    import torch
    import all_pairs_body_gb300 as nb
    pm = torch.from_numpy(np.ascontiguousarray(pm_np, dtype=np.float32)).cuda()
    ndc, rgba = nb.render_points(pm, lim, min_w, max_w)
    nb.sync()
    return ndc.cpu().numpy(), rgba.cpu().numpy()


def render_err(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got.astype(np.float64) - ref) / np.maximum(1.0, np.abs(ref))))


@pytest.mark.parametrize("n", [1, 7, 1000, 65537, 1048576])
def test_render_points(n):
    w = W.ball_lognormal_1048576(n) if n > 1 else W.random_bodies(1, 3)
    pm = w.pos_mass if hasattr(w, "pos_mass") else w
    m = pm[:, 3].astype(np.float64)
    lim = (1.25, 0.75, 1.5)  # some bodies fall outside the box: no clamping
    min_w, max_w = float(m.min()), float(m.max()) if n > 1 else float(m.min()) + 1.0
    ndc, rgba = gpu_render(pm, lim, min_w, max_w)
    rn, rc = oracle.render_points(pm, lim, np.float32(min_w), np.float32(max_w))
    assert render_err(ndc, rn) <= RENDER_TOL and render_err(rgba, rc) <= RENDER_TOL
    assert np.all(ndc[:, 3] == 1.0) and np.all(rgba[:, 3] == 1.0) and np.all(rgba[:, 2] == 0.0)


def test_render_after_steps():
    """The intended use: colour and place the bodies after each step."""
    w = W.plummer_16384()
    p, _, _ = gpu_leapfrog(w.pos_mass, w.vel, w.eps2, w.dt, 3)
    ndc, rgba = gpu_render(p, (4.0, 4.0, 4.0), 0.0, 2.0 / w.n)
    rn, rc = oracle.render_points(p, (4.0, 4.0, 4.0), 0.0, np.float32(2.0 / w.n))
    assert render_err(ndc, rn) <= RENDER_TOL and render_err(rgba, rc) <= RENDER_TOL


# ---------------------------------------------------------------------------
# 2-D cutoff neighbour list: counts and lists bit-exact against the oracle
# ---------------------------------------------------------------------------


def gpu_neighbors(x, y, cutoff, mn):
    import torch
    import all_pairs_body_gb300 as nb
    tx = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    ty = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).cuda()
    nn = torch.full((len(x),), -7, dtype=torch.int32, device="cuda")
    nl = torch.full((mn, len(x)), -7, dtype=torch.int32, device="cuda")
    nb.neighbors_2d(tx, ty, cutoff, mn, nn=nn, nl=nl)
    nb.sync()
    return nn.cpu().numpy(), nl.cpu().numpy()


@pytest.mark.parametrize("n", [1, 2, 3, 127, 128, 129, 511, 512, 513, 1000, 20000, 65537])
def test_neighbors_match_oracle(n):
    p = W.points_2d(n)
    nn, nl = gpu_neighbors(p.x, p.y, p.cutoff, p.max_neighbors)
    rn, rl = oracle.neighbors_2d(p.x, p.y, p.cutoff, p.max_neighbors)
    assert np.array_equal(nn, rn) and np.array_equal(nl, rl)


def test_neighbors_lattice_boundary_cases():
    k = 37
    ix, iy = np.meshgrid(np.arange(k), np.arange(k), indexing="xy")
    x, y = ix.ravel().astype(np.float32), iy.ravel().astype(np.float32)
    for cutoff in (1.0, 1.2, np.sqrt(2.0), 1.5, 2.0, 2.5):  # exact-distance ties included
        nn, nl = gpu_neighbors(x, y, cutoff, 24)
        rn, rl = oracle.neighbors_2d(x, y, cutoff, 24)
        assert np.array_equal(nn, rn) and np.array_equal(nl, rl), cutoff


def test_neighbors_truncated_and_empty_lists():
    p = W.points_2d(30000)
    for mn in (0, 1, 3, 64):
        nn, nl = gpu_neighbors(p.x, p.y, p.cutoff, mn)
        rn, rl = oracle.neighbors_2d(p.x, p.y, p.cutoff, mn)
        assert np.array_equal(nn, rn) and np.array_equal(nl, rl), mn
    assert (rn > 3).any()


def test_neighbors_large_sampled():
    """2^20 points: 4096 seeded sampled targets against the oracle, plus the
    symmetry of the relation (the sum of all counts is even)."""
    p = W.points_2d(1048576)
    nn, nl = gpu_neighbors(p.x, p.y, p.cutoff, p.max_neighbors)
    assert int(nn.astype(np.int64).sum()) % 2 == 0
    idx = W.sample_indices(p.n, 5)
    rn, rl = oracle.neighbors_2d(p.x, p.y, p.cutoff, p.max_neighbors, idx=idx)
    assert np.array_equal(nn[idx], rn) and np.array_equal(nl[:, idx], rl)


# ---------------------------------------------------------------------------
# velocity / acceleration layouts: same bits as the float4 rows
# ---------------------------------------------------------------------------


def _to_layout(v4, layout):
    v = np.ascontiguousarray(v4[:, :3])
    return v if layout == 1 else np.ascontiguousarray(v.T)


@pytest.mark.parametrize("layout", [0, 1, 2])
@pytest.mark.parametrize("n", [3000, 40000, 200000])  # warp, medium tiled, large tiled kernels
def test_layouts_match_rows4(layout, n):
    import torch
    import all_pairs_body_gb300 as nb
    pm = W.random_bodies(n, 40 + layout)
    v = W.random_velocities(n, 40 + layout)
    ref_a = gpu_accel(pm, 1e-3)
    rp, rv, ra = gpu_leapfrog(pm, v, 1e-3, 1e-3, 3)
    shape = (n, 4) if layout == 0 else ((n, 3) if layout == 1 else (3, n))
    out = torch.empty(shape, device="cuda")
    nb.accel_layout(torch.from_numpy(pm).cuda(), out, 1e-3, layout)
    nb.sync()
    want = ref_a if layout == 0 else _to_layout(ref_a, layout)
    assert np.array_equal(out.cpu().numpy(), want)
    tv = torch.from_numpy(v if layout == 0 else _to_layout(v, layout)).cuda()
    ta = torch.empty_like(tv)
    tp = torch.from_numpy(pm).cuda()
    nb.leapfrog_step_layout(tp, tv, ta, 1e-3, 1e-3, 3, layout)
    nb.sync()
    assert np.array_equal(tp.cpu().numpy(), rp)
    wantv = rv if layout == 0 else _to_layout(rv, layout)
    wanta = ra if layout == 0 else _to_layout(ra, layout)
    assert np.array_equal(tv.cpu().numpy(), wantv) and np.array_equal(ta.cpu().numpy(), wanta)


def _from_layout(a, layout):
    """(n, 3) rows of a velocity or acceleration array in `layout`."""
    a = np.asarray(a, dtype=np.float64)
    return a[:, :3] if layout != 2 else a.T


_LAYOUT_REF = {}


@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("n", [3000, 40000, 200000])  # warp kernel, pair path, pair path
def test_layout_steps_match_oracle(layout, n):
    """Three leapfrog steps with velocities and accelerations as float3 rows or
    x/y/z blocks, against the FP64 oracle at the trajectory tolerances."""
    import torch
    import all_pairs_body_gb300 as nb
    pm = W.random_bodies(n, 8000 + n)
    v = W.random_velocities(n, 8000 + n)
    if n not in _LAYOUT_REF:
        _LAYOUT_REF[n] = oracle.leapfrog(pm, v, 1e-3, 1e-3, 3)
    rp, rv, ra = _LAYOUT_REF[n]
    tp = torch.from_numpy(pm).cuda()
    tv = torch.from_numpy(_to_layout(v, layout)).cuda()
    ta = torch.full_like(tv, float("nan"))
    nb.leapfrog_step_layout(tp, tv, ta, 1e-3, 1e-3, 3, layout)
    nb.sync()
    got_p = tp.cpu().numpy()
    assert np.array_equal(got_p[:, 3], pm[:, 3]), "masses must not change"
    assert rel_err(got_p, rp) <= POS_TOL
    assert rel_err(_from_layout(tv.cpu().numpy(), layout), rv) <= VEL_TOL
    assert rel_err(_from_layout(ta.cpu().numpy(), layout), ra) <= ACC_TOL
    assert displacement_err(got_p, rp, pm, 3) <= POS_TOL


# ---------------------------------------------------------------------------
# seeded random configurations
# ---------------------------------------------------------------------------


def _random_cases(count, seed):
    """Seeded draws over the call space: n log-uniform in [1, 60000], the
    entry point (accelerations, steps, kick-drift-kick steps, steps with
    float3 or block velocity layouts), the forced path and split, 1-4 steps
    and eps2 in {1e-2, 1e-3, 1e-4}."""
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(count):
        n = int(round(float(np.exp(rng.uniform(0.0, np.log(60000.0))))))
        mode = ("accel", "step", "kdk", "layout")[int(rng.integers(4))]
        path, split = PATHS[int(rng.integers(len(PATHS)))]
        cases.append((k, n, mode, path, split, int(rng.integers(1, 5)), int(rng.integers(1, 3)),
                      (1e-2, 1e-3, 1e-4)[int(rng.integers(3))]))
    return cases


@pytest.mark.parametrize("k,n,mode,path,split,steps,layout,eps2", _random_cases(24, 2026))
def test_random_configurations(k, n, mode, path, split, steps, layout, eps2):
    import torch
    import all_pairs_body_gb300 as nb
    pm = W.random_bodies(n, 8500 + k)
    v = W.random_velocities(n, 8500 + k)
    if mode == "accel":
        a = gpu_accel(pm, eps2, path, split)
        assert rel_err(a, oracle.accel(pm, eps2)) <= ACC_TOL
        assert np.all(a[:, 3] == 0.0)
        return
    if mode == "layout":
        tp = torch.from_numpy(pm).cuda()
        tv = torch.from_numpy(_to_layout(v, layout)).cuda()
        ta = torch.full_like(tv, float("nan"))
        nb.leapfrog_step_layout(tp, tv, ta, eps2, 1e-3, steps, layout)
        nb.sync()
        p, vv, a = tp.cpu().numpy(), _from_layout(tv.cpu().numpy(), layout), \
            _from_layout(ta.cpu().numpy(), layout)
        rp, rv, ra = oracle.leapfrog(pm, v, eps2, 1e-3, steps)
    elif mode == "kdk":
        p, vv, a = gpu_kdk(pm, v, eps2, 1e-3, steps, path, split)
        rp, rv, ra = oracle.leapfrog_kdk(pm, v, eps2, 1e-3, steps)
        assert np.array_equal(vv[:, 3], v[:, 3])
    else:
        p, vv, a = gpu_leapfrog(pm, v, eps2, 1e-3, steps, path, split)
        rp, rv, ra = oracle.leapfrog(pm, v, eps2, 1e-3, steps)
        assert np.array_equal(vv[:, 3], v[:, 3])
    assert rel_err(a, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL
    assert rel_err(p, rp) <= POS_TOL and displacement_err(p, rp, pm, steps) <= 1e-3
    assert np.array_equal(p[:, 3], pm[:, 3])


# ---------------------------------------------------------------------------
# plain entry points (legacy default stream) and concurrent streams
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("n", [1000, 3000, 20000])
def test_caller_kernels_around_calls_are_ordered(n):
    """The library's kernels are programmatic dependents of one another; the
    caller's own kernels enqueued right before and after a call, with no host
    synchronisation, still see the call's inputs and outputs in stream order:
    a step on positions a torch kernel just shifted, then a torch kernel that
    reads the step's outputs."""
    import torch
    import all_pairs_body_gb300 as nb
    pm0 = W.random_bodies(n, 9100 + n)
    v0 = W.random_velocities(n, 9100 + n)
    shift = np.array([0.25, -0.5, 0.125, 0.0], dtype=np.float32)
    pm = torch.from_numpy(pm0).cuda()
    v = torch.from_numpy(v0).cuda()
    a = torch.empty_like(pm)
    torch.cuda.synchronize()
    for _ in range(2):
        pm.add_(torch.from_numpy(shift).cuda())  # a caller kernel before the call
        nb.leapfrog_step(pm, v, a, 1e-3, 1e-3, 3)
        doubled = a * 2.0  # a caller kernel after it
    nb.sync()
    p_ref, v_ref = pm0.copy(), v0.copy()
    for _ in range(2):
        p_ref[:, :3] += shift[:3]
        p_ref, v_ref, a_ref = oracle.leapfrog(p_ref.astype(np.float32), v_ref.astype(np.float32),
                                              1e-3, 1e-3, 3)
        v_ref = np.concatenate([v_ref, v0[:, 3:4]], axis=1)
    assert rel_err(pm.cpu().numpy(), p_ref) <= POS_TOL
    assert rel_err(v.cpu().numpy(), v_ref) <= VEL_TOL
    assert rel_err(doubled.cpu().numpy(), 2.0 * a_ref) <= ACC_TOL
    assert np.array_equal(doubled.cpu().numpy(), 2.0 * a.cpu().numpy())


def test_plain_entry_points_on_the_legacy_stream():
    import ctypes
    import torch
    import all_pairs_body_gb300 as nb
    L = nb.lib()
    P = ctypes.c_void_p
    w = W.cube_sweep(4097)
    pm = torch.from_numpy(w.pos_mass).cuda()
    out = torch.full_like(pm, float("nan"))
    torch.cuda.synchronize()
    assert L.nbody_accel(P(pm.data_ptr()), P(out.data_ptr()), w.n, ctypes.c_float(w.eps2)) == nb.OK
    assert L.nbody_sync(P(0)) == nb.OK
    assert rel_err(out.cpu().numpy(), oracle.accel(w.pos_mass, w.eps2)) <= ACC_TOL
    v = torch.from_numpy(W.random_velocities(w.n, 9)).cuda()
    a = torch.full_like(pm, float("nan"))
    assert L.nbody_leapfrog_step(P(pm.data_ptr()), P(v.data_ptr()), P(a.data_ptr()), w.n,
                                 ctypes.c_float(w.eps2), ctypes.c_float(1e-3), 2) == nb.OK
    assert L.nbody_sync(P(0)) == nb.OK
    rp, rv, ra = oracle.leapfrog(w.pos_mass, W.random_velocities(w.n, 9), w.eps2, 1e-3, 2)
    assert rel_err(a.cpu().numpy(), ra) <= ACC_TOL and rel_err(pm.cpu().numpy(), rp) <= POS_TOL


@pytest.mark.parametrize("n", [4000, 40000])
def test_concurrent_streams_use_separate_scratch(n):
    """Two multi-step calls in flight at once on two streams (each with its
    own cached scratch and grid counter) give the same bits as the same calls
    run alone: the one-kernel warp pass and the pair path."""
    import torch
    import all_pairs_body_gb300 as nb
    inputs = [(W.random_bodies(n, s), W.random_velocities(n, s)) for s in (51, 52)]
    alone = [gpu_leapfrog(pm, v, 1e-3, 1e-3, 3) for pm, v in inputs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    bufs = []
    for (pm, v), st in zip(inputs, streams):
        with torch.cuda.stream(st):
            tp = torch.from_numpy(pm).to("cuda", non_blocking=False)
            tv = torch.from_numpy(v).to("cuda", non_blocking=False)
            ta = torch.empty_like(tp)
            bufs.append((tp, tv, ta))
    torch.cuda.synchronize()
    for (tp, tv, ta), st in zip(bufs, streams):
        with torch.cuda.stream(st):
            nb.leapfrog_step(tp, tv, ta, 1e-3, 1e-3, 3)
    for st in streams:
        nb.sync(st)
    for (tp, tv, ta), (rp, rv, ra) in zip(bufs, alone):
        assert np.array_equal(tp.cpu().numpy(), rp) and np.array_equal(tv.cpu().numpy(), rv)
        assert np.array_equal(ta.cpu().numpy(), ra)
