"""Every row of the tuning build's kernel tables against the FP64 oracle.

The release library holds only the kernel shapes its plans choose between.
The tuning build (compiled with NBODY_TUNING_TABLE) appends every other shape
and reaction scheme that was measured while choosing them: the one-sided
tiled kernel with other tiles, unrolls and the mixed rsqrt/logarithmic inner
loop, and the pair-symmetric kernel with the warp-butterfly reduction and
the plain lane rotation, and the small-n warp kernel with other target
counts and load-ahead depths.  NBODY_TILED_CONFIG / NBODY_PAIRS_CONFIG /
NBODY_WARP_CONFIG select a row by index; these tests route the binding
through that build and hold each row to the same tolerances as the release
paths.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import ACC_TOL, POS_TOL, VEL_TOL, gpu_accel, gpu_leapfrog, rel_err

pytestmark = pytest.mark.gpu

# rows of the tuning build's tables (the release rows come first)
N_TILED_ROWS = 22
N_PAIR_ROWS = 90
N_WARP_ROWS = 16
N_TILED_RELEASE = 4
N_PAIR_RELEASE = 6
N_WARP_RELEASE = 2


@pytest.fixture(scope="module", autouse=True)
def tuning_lib():
    """Route the binding through the tuning build for this module."""
    import torch
    import all_pairs_body_gb300 as nb
    from all_pairs_body_gb300 import build as nbuild
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()
    path = nbuild.build(tuning=True)
    saved = nb._lib
    nb._lib = nb.load(path)
    try:
        assert nb.table_row(0, 0)["rows"] == N_TILED_ROWS
        assert nb.table_row(1, 0)["rows"] == N_PAIR_ROWS
        assert nb.table_row(2, 0)["rows"] == N_WARP_ROWS
        yield nb._lib
    finally:
        nb.release()
        nb._lib = saved


def test_release_rows_lead_the_tuning_tables():
    """The tuning build's first rows are the release build's rows, so a row
    index means the same kernel in both builds."""
    import all_pairs_body_gb300 as nb
    release = nb.load(nb.LIB_PATH)
    for which, count in ((0, N_TILED_RELEASE), (1, N_PAIR_RELEASE), (2, N_WARP_RELEASE)):
        for r in range(count):
            out = (nb.ctypes.c_int64 * 6)()
            assert release.nbody_table(which, r, out, 6) == nb.OK
            got = nb.table_row(which, r)
            assert [got[k] for k in nb.TABLE_FIELDS[1:]] == list(out)[1:], (which, r)


@pytest.mark.parametrize("cfg", range(N_PAIR_ROWS))
def test_every_pair_variant(cfg, monkeypatch):
    monkeypatch.setenv("NBODY_PAIRS_CONFIG", str(cfg))
    w = W.cube_sweep(20000)
    a = gpu_accel(w.pos_mass, w.eps2, path=4)
    assert np.all(a[:, 3] == 0.0)
    assert rel_err(a, oracle.accel(w.pos_mass, w.eps2)) <= ACC_TOL
    pm = W.random_bodies(9000, 78)
    v = W.random_velocities(9000, 78)
    p, vv, a = gpu_leapfrog(pm, v, 1e-3, 1e-3, 3, path=4)
    rp, rv, ra = oracle.leapfrog(pm, v, 1e-3, 1e-3, 3)
    assert rel_err(a, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL and rel_err(p, rp) <= POS_TOL


@pytest.mark.parametrize("cfg", range(N_WARP_ROWS))
@pytest.mark.parametrize("n", [1000, 4097, 9000])
def test_every_warp_variant(cfg, n, monkeypatch):
    monkeypatch.setenv("NBODY_WARP_CONFIG", str(cfg))
    pm = W.random_bodies(n, 79 + n)
    a = gpu_accel(pm, 1e-3, path=3)
    assert np.all(a[:, 3] == 0.0)
    assert rel_err(a, oracle.accel(pm, 1e-3)) <= ACC_TOL
    a5 = gpu_accel(pm, 1e-3, path=3, split=5)  # five j slices and the second pass
    assert rel_err(a5, oracle.accel(pm, 1e-3)) <= ACC_TOL
    v = W.random_velocities(n, 79 + n)
    p, vv, a = gpu_leapfrog(pm, v, 1e-3, 1e-3, 2, path=3)
    rp, rv, ra = oracle.leapfrog(pm, v, 1e-3, 1e-3, 2)
    assert rel_err(a, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL and rel_err(p, rp) <= POS_TOL


@pytest.mark.parametrize("cfg", range(N_TILED_ROWS))
def test_every_tiled_variant(cfg, monkeypatch):
    monkeypatch.setenv("NBODY_TILED_CONFIG", str(cfg))
    w = W.cube_sweep(20000)
    a = gpu_accel(w.pos_mass, w.eps2, path=2)
    assert rel_err(a, oracle.accel(w.pos_mass, w.eps2)) <= ACC_TOL
    pm = W.random_bodies(9000, 77)
    v = W.random_velocities(9000, 77)
    p, vv, a = gpu_leapfrog(pm, v, 1e-3, 1e-3, 3, path=2)
    rp, rv, ra = oracle.leapfrog(pm, v, 1e-3, 1e-3, 3)
    assert rel_err(a, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL and rel_err(p, rp) <= POS_TOL


def special_masses(n, seed):
    pm = W.random_bodies(n, seed)
    pm[::7, 3] = 0.0  # massless bodies
    return pm


# one rsqrt-form row and three rows of the mixed rsqrt/logarithmic loop
@pytest.mark.parametrize("cfg,form", [(9, 0), (14, 1), (16, 1), (19, 1)])
def test_zero_masses(cfg, form, monkeypatch):
    import all_pairs_body_gb300 as nb
    assert nb.table_row(0, cfg)["form_or_acc"] == form
    monkeypatch.setenv("NBODY_TILED_CONFIG", str(cfg))
    pm = special_masses(20000, 5)
    a = gpu_accel(pm, 1e-3, path=2)
    assert rel_err(a, oracle.accel(pm, 1e-3)) <= ACC_TOL
    lone = np.zeros((20000, 4), dtype=np.float32)
    lone[:, :3] = pm[:, :3]
    lone[123, 3] = 1.0  # one massive body among massless ones
    a = gpu_accel(lone, 1e-3, path=2)
    assert rel_err(a, oracle.accel(lone, 1e-3)) <= ACC_TOL
    assert np.all(a[123, :3] == 0.0)


@pytest.mark.parametrize("cfg,form", [(9, 0), (14, 1), (16, 1)])
def test_negative_masses_take_the_exact_loop(cfg, form, monkeypatch):
    import all_pairs_body_gb300 as nb
    assert nb.table_row(0, cfg)["form_or_acc"] == form
    monkeypatch.setenv("NBODY_TILED_CONFIG", str(cfg))
    pm = W.random_bodies(20000, 6)
    pm[300:310, 3] *= -1.0  # a few negative masses inside one source tile
    pm[19990, 3] *= -1.0  # and one in the ragged last tile
    a = gpu_accel(pm, 1e-3, path=2)
    assert rel_err(a, oracle.accel(pm, 1e-3)) <= ACC_TOL
    v = W.random_velocities(20000, 6)
    p, vv, aa = gpu_leapfrog(pm, v, 1e-3, 1e-3, 2, path=2)
    rp, rv, ra = oracle.leapfrog(pm, v, 1e-3, 1e-3, 2)
    assert rel_err(aa, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL
