"""The C ABI without a GPU: exports, status texts and host-side argument checks.

Every check here happens before the library touches CUDA, so these tests run
on a machine with no GPU.  Pointers are plain integers that are never
dereferenced (validation rejects the call first).
"""
import ctypes
import math
import os
import re

import pytest

import all_pairs_body_gb300 as nb
from all_pairs_body_gb300 import build as nbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "nbody.h")
A, B, C = 0x10000, 0x20000, 0x30000  # 16-byte aligned fake addresses, far apart
S = ctypes.c_void_p(0)


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # noqa: BLE001
        return False


@pytest.fixture(scope="module")
def L():
    nbuild.build()
    return nb.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nbody_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_bound_functions():
    assert declared_functions() == sorted(nb.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_strerror(L):
    for code in (nb.OK, nb.EINVAL, nb.ENOMEM, nb.ECUDA, nb.ETIMEOUT):
        assert L.nbody_strerror(code)
    assert nb.strerror(nb.EINVAL) == "invalid argument"
    assert L.nbody_strerror(99) == b"unknown status"


def accel(L, pos, acc, n, eps2, path=0, split=0):
    return L.nbody_accel_with(ctypes.c_void_p(pos), ctypes.c_void_p(acc), n, eps2, path, split, S)


def step(L, pos, vel, acc, n, eps2, dt, steps, path=0, split=0):
    return L.nbody_leapfrog_step_with(ctypes.c_void_p(pos), ctypes.c_void_p(vel),
                                      ctypes.c_void_p(acc), n, eps2, dt, steps, path, split, S)


@pytest.mark.parametrize("n,eps2", [(-1, 0.1), (2 ** 31, 0.1), (10, 0.0), (10, -1e-3),
                                    (10, math.nan), (10, math.inf)])
def test_accel_bad_scalars(L, n, eps2):
    assert accel(L, A, B, n, eps2) == nb.EINVAL


@pytest.mark.parametrize("path,split", [(-1, 0), (5, 0), (0, -1)])
def test_accel_bad_path(L, path, split):
    assert accel(L, A, B, 10, 0.1, path, split) == nb.EINVAL


@pytest.mark.parametrize("pos,acc", [(0, B), (A, 0), (A + 4, B), (A, B + 8)])
def test_accel_bad_pointers(L, pos, acc):
    assert accel(L, pos, acc, 10, 0.1) == nb.EINVAL


def test_accel_overlap(L):
    assert accel(L, A, A, 10, 0.1) == nb.EINVAL
    assert accel(L, A, A + 16 * 9, 10, 0.1) == nb.EINVAL  # last row shared
    assert accel(L, A + 16 * 9, A, 10, 0.1) == nb.EINVAL


def test_accel_empty_is_noop(L):
    assert accel(L, 0, 0, 0, 0.1) == nb.OK
    assert L.nbody_accel(None, None, 0, ctypes.c_float(0.1)) == nb.OK


@pytest.mark.parametrize("n,eps2,dt,steps", [(-1, 0.1, 0.1, 1), (10, 0.0, 0.1, 1),
                                             (10, 0.1, math.nan, 1), (10, 0.1, math.inf, 1),
                                             (10, 0.1, 0.1, -1)])
def test_step_bad_scalars(L, n, eps2, dt, steps):
    assert step(L, A, B, C, n, eps2, dt, steps) == nb.EINVAL


def test_step_bad_pointers_and_overlap(L):
    assert step(L, 0, B, C, 10, 0.1, 0.1, 1) == nb.EINVAL
    assert step(L, A, B + 4, C, 10, 0.1, 0.1, 1) == nb.EINVAL
    assert step(L, A, A, C, 10, 0.1, 0.1, 1) == nb.EINVAL  # pos and vel alias
    assert step(L, A, B, B, 10, 0.1, 0.1, 1) == nb.EINVAL  # vel and accel alias
    assert step(L, A, B, A + 16, 10, 0.1, 0.1, 1) == nb.EINVAL  # pos and accel overlap


def test_step_noops(L):
    assert step(L, 0, 0, 0, 0, 0.1, 0.1, 3) == nb.OK
    assert step(L, A, B, C, 10, 0.1, 0.1, 0) == nb.OK
    assert step(L, 0, 0, 0, 10, 0.1, 0.1, 0) == nb.OK
    assert L.nbody_leapfrog_step(None, None, None, 0, ctypes.c_float(0.1),
                                 ctypes.c_float(0.1), 1) == nb.OK


def test_plan_rejects_bad_arguments(L):
    out = (ctypes.c_int64 * 4)()
    assert L.nbody_plan(-5, 0, 0, out, 4) == nb.EINVAL
    assert L.nbody_plan(10, 7, 0, out, 4) == nb.EINVAL
    assert L.nbody_plan(10, 0, 0, None, 4) == nb.EINVAL


@pytest.mark.skipif(_has_gpu(), reason="checks the no-device path")
def test_no_device_is_ecuda(L):
    assert accel(L, A, B, 10, 0.1) == nb.ECUDA
    assert step(L, A, B, C, 10, 0.1, 0.1, 1) == nb.ECUDA
    out = (ctypes.c_int64 * 4)()
    assert L.nbody_plan(10, 0, 0, out, 4) == nb.ECUDA
    assert L.nbody_selftest_timeout(10, S) in (nb.ENOMEM, nb.ECUDA)
    L.nbody_release()  # nothing cached: must not fail


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(nb, "_lib", None)
    monkeypatch.setattr(nb, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        nb.lib()


def render(L, pos, ndc, rgba, n, lim=(1.0, 1.0, 1.0), w=(0.0, 1.0)):
    return L.nbody_render_points(ctypes.c_void_p(pos), ctypes.c_void_p(ndc), ctypes.c_void_p(rgba),
                                 n, *lim, *w, S)


@pytest.mark.parametrize("lim,w", [((0.0, 1.0, 1.0), (0.0, 1.0)), ((1.0, -1.0, 1.0), (0.0, 1.0)),
                                   ((1.0, 1.0, math.nan), (0.0, 1.0)), ((1.0, 1.0, 1.0), (1.0, 1.0)),
                                   ((1.0, 1.0, 1.0), (2.0, 1.0)), ((1.0, 1.0, 1.0), (0.0, math.inf))])
def test_render_bad_parameters(L, lim, w):
    assert render(L, A, B, C, 10, lim, w) == nb.EINVAL


def test_render_bad_pointers(L):
    assert render(L, 0, B, C, 10) == nb.EINVAL
    assert render(L, A, B + 4, C, 10) == nb.EINVAL
    assert render(L, A, A + 16, C, 10) == nb.EINVAL
    assert render(L, A, B, B, 10) == nb.EINVAL
    assert render(L, A, B, C, -1) == nb.EINVAL
    assert render(L, 0, 0, 0, 0) == nb.OK


def neighbors(L, x, y, n, cutoff, mn, nn, nl):
    return L.nbody_neighbors_2d(ctypes.c_void_p(x), ctypes.c_void_p(y), n, cutoff, mn,
                                ctypes.c_void_p(nn), ctypes.c_void_p(nl), S)


def test_neighbors_bad_arguments(L):
    D = 0x40000
    assert neighbors(L, A, B, 10, 0.0, 4, C, D) == nb.EINVAL
    assert neighbors(L, A, B, 10, math.nan, 4, C, D) == nb.EINVAL
    assert neighbors(L, A, B, 10, 1e-30, 4, C, D) == nb.EINVAL  # cutoff^2 not a normal float
    assert neighbors(L, A, B, 10, 1.0, -1, C, D) == nb.EINVAL
    assert neighbors(L, A, B, -1, 1.0, 4, C, D) == nb.EINVAL
    assert neighbors(L, A, B, 10, 1.0, 4, C, 0) == nb.EINVAL
    assert neighbors(L, A + 2, B, 10, 1.0, 4, C, D) == nb.EINVAL
    assert neighbors(L, A, B, 10, 1.0, 4, A, D) == nb.EINVAL  # nn overlaps x
    assert neighbors(L, A, B, 10, 1.0, 4, C, C + 8) == nb.EINVAL  # nl overlaps nn
    assert neighbors(L, 0, 0, 0, 1.0, 4, 0, 0) == nb.OK


def test_layout_entry_points_validate(L):
    f = ctypes.c_float
    assert L.nbody_accel_layout(ctypes.c_void_p(A), ctypes.c_void_p(B), 10, f(0.1), 3, S) == nb.EINVAL
    assert L.nbody_accel_layout(ctypes.c_void_p(A), ctypes.c_void_p(B + 4), 10, f(0.1), 0, S) == nb.EINVAL
    assert L.nbody_accel_layout(ctypes.c_void_p(A), ctypes.c_void_p(B + 2), 10, f(0.1), 1, S) == nb.EINVAL
    # a three-float array of 10 rows is 120 bytes: it overlaps positions 16 bytes on
    assert L.nbody_accel_layout(ctypes.c_void_p(A), ctypes.c_void_p(A + 16 * 9), 10, f(0.1), 1,
                                S) == nb.EINVAL
    assert L.nbody_leapfrog_step_layout(ctypes.c_void_p(A), ctypes.c_void_p(B), ctypes.c_void_p(B + 100),
                                        10, f(0.1), f(0.1), 1, 2, S) == nb.EINVAL  # vel/accel overlap
    assert L.nbody_leapfrog_step_layout(ctypes.c_void_p(A), ctypes.c_void_p(B), ctypes.c_void_p(C),
                                        10, f(0.1), f(0.1), 1, -1, S) == nb.EINVAL


def test_strerror_covers_ebounds(L):
    assert L.nbody_strerror(nb.EBOUNDS) == b"a device-side index check failed (checked build)"


def test_checked_build_exports_every_declared_symbol():
    """The index-checked library builds without a GPU and exports the same C ABI."""
    Lc = nb.load(nbuild.build(checked=True))
    for name in declared_functions():
        assert hasattr(Lc, name), name
    assert Lc.nbody_strerror(nb.EBOUNDS).startswith(b"a device-side index check")
    # argument checks happen before any CUDA call, as in the release build
    assert Lc.nbody_accel_with(ctypes.c_void_p(A), ctypes.c_void_p(B), -1, 0.1, 0, 0, S) == nb.EINVAL


def test_binding_rejects_tensors_before_any_cuda_call():
    """The Python binding checks device, dtype, layout and shape first; these
    tensors live on the CPU or are malformed, so nothing reaches the library."""
    torch = pytest.importorskip("torch")
    good_shape = torch.zeros((8, 4), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        nb.accel(good_shape, 0.1, out=torch.zeros_like(good_shape))
    with pytest.raises(TypeError, match="must be a torch.Tensor"):
        nb.accel(good_shape.numpy(), 0.1, out=torch.zeros_like(good_shape))
    with pytest.raises(ValueError):
        nb.neighbors_2d(torch.zeros(8), torch.zeros(8), 0.5, 4)
    with pytest.raises(ValueError):
        nb.accel_layout(good_shape, torch.zeros(24), 0.1, nb.ROWS3)


def _table(L, which, row):
    out = (ctypes.c_int64 * 6)()
    rc = L.nbody_table(which, row, out, 6)
    return rc, list(out)


def test_release_table_holds_only_the_planned_kernels(L):
    """The release build compiles the rows its plans choose between: four
    one-sided tiled shapes (two large-n tiles, the no-allocation shape, the
    small-n shape), six pair-symmetric shapes (targets per thread, threads,
    tile, running sums in shared memory, reaction scheme) and two warp-kernel
    shapes (targets per CTA, threads, sources loaded ahead, lanes combined by
    a reduce-scatter): 12 force kernels."""
    rc, row = _table(L, 0, 0)
    assert rc == nb.OK and row[0] == 4
    tiled = [tuple(_table(L, 0, r)[1][1:5]) for r in range(4)]
    assert tiled == [(10, 256, 512, 0), (10, 256, 256, 0), (4, 128, 128, 0), (2, 128, 64, 0)]
    rc, row = _table(L, 1, 0)
    assert rc == nb.OK and row[0] == 6
    pairs = [tuple(_table(L, 1, r)[1][1:6]) for r in range(6)]
    assert pairs == [(16, 256, 512, 1, 3), (14, 256, 512, 0, 3), (12, 256, 512, 1, 3),
                     (10, 256, 512, 1, 4), (8, 256, 512, 1, 4), (8, 256, 256, 0, 4)]
    assert 4 + 6 + 2 <= 12
    rc, row = _table(L, 2, 0)
    assert rc == nb.OK and row[0] == 2
    warps = [tuple(_table(L, 2, r)[1][1:5]) for r in range(2)]
    assert warps == [(6, 128, 8, 1), (8, 128, 8, 1)]
    for which, row in ((0, 4), (1, 6), (2, 2), (0, -1), (3, 0)):
        assert _table(L, which, row)[0] == nb.EINVAL
    assert L.nbody_table(0, 0, None, 0) == nb.OK
    assert L.nbody_table(0, 0, None, 3) == nb.EINVAL


@pytest.mark.skipif(_has_gpu(), reason="checks the behaviour without a usable device")
def test_status_queries_without_a_device(L):
    out = (ctypes.c_int64 * 13)()
    assert L.nbody_last_plan(S, out, 13) in (nb.ECUDA, nb.EINVAL)
    assert L.nbody_last_plan(S, None, 13) == nb.EINVAL
    assert L.nbody_selftest_timeout_enqueue(0, S) == nb.EINVAL


def test_phase_clocks_only_in_the_profiling_build(L):
    """The release library has no phase stamps: nbody_phase_read says so
    without touching a device."""
    out = (ctypes.c_int64 * 7)()
    assert L.nbody_phase_read(out, 7) == nb.EINVAL
