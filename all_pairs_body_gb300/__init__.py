"""Python binding of the GB300 all-pairs softened-gravity library.

Argument marshalling only.  Every step of the computation (the all-pairs
acceleration sum, the second-pass reductions and the leapfrog kick/drift)
runs in the CUDA kernels of ``libnbody_gb300.so``, whose C ABI is declared in
``include/nbody.h``.  PyTorch supplies device memory and the current stream.
There is no CPU fallback: every call raises if the compiled library is
missing or no CUDA device is usable.

    a_i = sum_j m_j (x_j - x_i) / (|x_j - x_i|^2 + eps2)^(3/2),  G = 1
    step: v <- v + (dt/2) a(x);  x <- x + dt v

("CUDA N-Body Simulation" §1.2 and §1.3.)  Bodies are float32 (n, 4) rows
(x, y, z, m); velocities (vx, vy, vz, w); accelerations (ax, ay, az, 0).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnbody_gb300.so")

PATH_AUTO, PATH_TILED, PATH_SPLIT, PATH_WARP, PATH_PAIRS = 0, 1, 2, 3, 4
OK, EINVAL, ENOMEM, ECUDA, ETIMEOUT, EBOUNDS = 0, 1, 2, 3, 4, 5
PLAN_FIELDS = ("path", "grid", "threads", "bodies_per_cta", "tile", "tiles", "units",
               "second_pass", "launches_accel", "launches_step", "sms", "react_bytes", "chunks")

EXPORTS = ("nbody_accel", "nbody_accel_on_stream", "nbody_accel_with",
           "nbody_leapfrog_step", "nbody_leapfrog_step_on_stream",
           "nbody_leapfrog_step_with", "nbody_sync", "nbody_plan", "nbody_strerror",
           "nbody_release", "nbody_selftest_timeout", "nbody_profile_enable",
           "nbody_profile_read", "nbody_accel_noalloc", "nbody_leapfrog_kdk_on_stream",
           "nbody_leapfrog_kdk_with", "nbody_render_points", "nbody_neighbors_2d",
           "nbody_accel_layout", "nbody_leapfrog_step_layout", "nbody_table",
           "nbody_last_plan", "nbody_selftest_timeout_enqueue", "nbody_phase_read")
ROWS4, ROWS3, BLOCKS3 = 0, 1, 2
NOALLOC_MAX_N = 65536


class NBodyError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} (status {status})")


_lib = None


def load(path: str) -> ctypes.CDLL:
    """Load a build of the C library at ``path`` with its C signatures
    declared (the release build through lib(); tests also load the
    index-checked build this way)."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with all_pairs_body_gb300.build.build() "
            "(or __graft_entry__.build()); there is no CPU fallback")
    L = ctypes.CDLL(path)
    p, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    sig = {
        "nbody_accel": [p, p, i64, f32],
        "nbody_accel_on_stream": [p, p, i64, f32, p],
        "nbody_accel_with": [p, p, i64, f32, i32, i32, p],
        "nbody_accel_noalloc": [p, p, i64, f32, p],
        "nbody_leapfrog_step": [p, p, p, i64, f32, f32, i32],
        "nbody_leapfrog_step_on_stream": [p, p, p, i64, f32, f32, i32, p],
        "nbody_leapfrog_step_with": [p, p, p, i64, f32, f32, i32, i32, i32, p],
        "nbody_leapfrog_kdk_on_stream": [p, p, p, i64, f32, f32, i32, p],
        "nbody_leapfrog_kdk_with": [p, p, p, i64, f32, f32, i32, i32, i32, p],
        "nbody_render_points": [p, p, p, i64, f32, f32, f32, f32, f32, p],
        "nbody_neighbors_2d": [p, p, i64, f32, i32, p, p, p],
        "nbody_accel_layout": [p, p, i64, f32, i32, p],
        "nbody_leapfrog_step_layout": [p, p, p, i64, f32, f32, i32, i32, p],
        "nbody_sync": [p],
        "nbody_plan": [i64, i32, i32, ctypes.POINTER(i64), i32],
        "nbody_selftest_timeout": [i32, p],
        "nbody_selftest_timeout_enqueue": [i32, p],
        "nbody_last_plan": [p, ctypes.POINTER(i64), i32],
        "nbody_phase_read": [ctypes.POINTER(i64), i32],
        "nbody_table": [i32, i32, ctypes.POINTER(i64), i32],
        "nbody_profile_enable": [i32],
        "nbody_profile_read": [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64),
                               ctypes.POINTER(i64)],
        "nbody_strerror": [i32],
        "nbody_release": [],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = i32
    L.nbody_strerror.restype = ctypes.c_char_p
    L.nbody_release.restype = None
    return L


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def strerror(status: int) -> str:
    try:
        return lib().nbody_strerror(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _check(rc: int, where: str) -> None:
    if rc != OK:
        raise NBodyError(rc, where)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _rows(t, n: int | None, name: str):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if t.dim() != 2 or t.shape[1] != 4 or (n is not None and t.shape[0] != n):
        raise ValueError(f"{name} must have shape (n, 4)")
    return ctypes.c_void_p(t.data_ptr())


def accel(pos_mass, eps2: float, out=None, path: int = PATH_AUTO, split: int = 0,
          stream=None):
    """Accelerations of all bodies; returns ``out`` (allocated if None)."""
    import torch
    n = int(pos_mass.shape[0])
    if out is None:
        out = torch.empty_like(pos_mass)
    rc = lib().nbody_accel_with(_rows(pos_mass, None, "pos_mass"), _rows(out, n, "out"), n,
                                float(eps2), int(path), int(split), _stream(stream))
    _check(rc, "nbody_accel")
    return out


def accel_noalloc(pos_mass, out, eps2: float, stream=None):
    """Accelerations into ``out`` without any allocation by the library.

    For callers that must not allocate device memory when they ask for
    accelerations (a host whose own pool owns the device memory, a loop that
    bans allocation after start-up); the work memory is one fixed 6 MiB array
    per GPU that the library holds until exit.  n <= NOALLOC_MAX_N.  Calls
    must not overlap on the GPU (they share the array).  ``out`` must be
    allocated by the caller.
    """
    n = int(pos_mass.shape[0])
    rc = lib().nbody_accel_noalloc(_rows(pos_mass, None, "pos_mass"), _rows(out, n, "out"), n,
                                   float(eps2), _stream(stream))
    _check(rc, "nbody_accel_noalloc")
    return out


def leapfrog_step(pos_mass, vel, accel_out, eps2: float, dt: float, steps: int = 1,
                  path: int = PATH_AUTO, split: int = 0, stream=None) -> None:
    """``steps`` kick/drift steps in place on ``pos_mass`` and ``vel``; the last
    step's accelerations go to ``accel_out``."""
    n = int(pos_mass.shape[0])
    rc = lib().nbody_leapfrog_step_with(
        _rows(pos_mass, None, "pos_mass"), _rows(vel, n, "vel"), _rows(accel_out, n, "accel"),
        n, float(eps2), float(dt), int(steps), int(path), int(split), _stream(stream))
    _check(rc, "nbody_leapfrog_step")


def leapfrog_kdk(pos_mass, vel, accel_out, eps2: float, dt: float, steps: int = 1,
                 path: int = PATH_AUTO, split: int = 0, stream=None) -> None:
    """``steps`` kick-drift-kick steps in place; ``accel_out`` receives the
    accelerations at the final positions."""
    n = int(pos_mass.shape[0])
    rc = lib().nbody_leapfrog_kdk_with(
        _rows(pos_mass, None, "pos_mass"), _rows(vel, n, "vel"), _rows(accel_out, n, "accel"),
        n, float(eps2), float(dt), int(steps), int(path), int(split), _stream(stream))
    _check(rc, "nbody_leapfrog_kdk")


def render_points(pos_mass, max_xyz, min_w: float, max_w: float, ndc=None, rgba=None,
                  stream=None):
    """Normalised device coordinates and mass colours of all bodies (the
    pages' point shaders as a kernel); returns (ndc, rgba), (n, 4) each."""
    import torch
    n = int(pos_mass.shape[0])
    if ndc is None:
        ndc = torch.empty_like(pos_mass)
    if rgba is None:
        rgba = torch.empty_like(pos_mass)
    mx, my, mz = (float(v) for v in max_xyz)
    rc = lib().nbody_render_points(_rows(pos_mass, None, "pos_mass"), _rows(ndc, n, "ndc"),
                                   _rows(rgba, n, "rgba"), n, mx, my, mz, float(min_w),
                                   float(max_w), _stream(stream))
    _check(rc, "nbody_render_points")
    return ndc, rgba


def neighbors_2d(x, y, cutoff: float, max_neighbors: int, nn=None, nl=None, stream=None):
    """2-D cutoff neighbour list (all pairs, no atomics): returns (nn, nl),
    nn (n,) int32 counts and nl (max_neighbors, n) int32 ascending lists
    padded with -1."""
    import torch
    for name, t in (("x", x), ("y", y)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32
                and t.is_contiguous() and t.dim() == 1):
            raise ValueError(f"{name} must be a contiguous 1-D float32 CUDA tensor")
    n = int(x.shape[0])
    if int(y.shape[0]) != n:
        raise ValueError("x and y must have the same length")
    mn = int(max_neighbors)
    if nn is None:
        nn = torch.empty(n, dtype=torch.int32, device=x.device)
    if nl is None:
        nl = torch.empty((mn, n), dtype=torch.int32, device=x.device)
    rc = lib().nbody_neighbors_2d(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), n,
                                  float(cutoff), mn, ctypes.c_void_p(nn.data_ptr()),
                                  ctypes.c_void_p(nl.data_ptr() if mn > 0 else 0), _stream(stream))
    _check(rc, "nbody_neighbors_2d")
    return nn, nl


def _vec(t, n: int, layout: int, name: str):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    want = 4 * n if layout == ROWS4 else 3 * n
    if t.numel() != want:
        raise ValueError(f"{name} must hold {want} floats for layout {layout}")
    return ctypes.c_void_p(t.data_ptr())


def accel_layout(pos_mass, out, eps2: float, layout: int, stream=None):
    """Accelerations into ``out`` in ``layout`` (ROWS4: (n,4); ROWS3: (n,3);
    BLOCKS3: (3,n))."""
    n = int(pos_mass.shape[0])
    rc = lib().nbody_accel_layout(_rows(pos_mass, None, "pos_mass"), _vec(out, n, layout, "out"), n,
                                  float(eps2), int(layout), _stream(stream))
    _check(rc, "nbody_accel_layout")
    return out


def leapfrog_step_layout(pos_mass, vel, accel_out, eps2: float, dt: float, steps: int,
                         layout: int, stream=None) -> None:
    """``steps`` half-kick + drift steps with ``vel`` and ``accel_out`` in ``layout``."""
    n = int(pos_mass.shape[0])
    rc = lib().nbody_leapfrog_step_layout(_rows(pos_mass, None, "pos_mass"),
                                          _vec(vel, n, layout, "vel"),
                                          _vec(accel_out, n, layout, "accel"), n, float(eps2),
                                          float(dt), int(steps), int(layout), _stream(stream))
    _check(rc, "nbody_leapfrog_step_layout")


def sync(stream=None) -> None:
    """Wait for the stream and raise if a kernel this library enqueued on it
    reported a device-side failure."""
    _check(lib().nbody_sync(_stream(stream)), "nbody_sync")


def plan(n: int, path: int = PATH_AUTO, split: int = 0) -> dict:
    """Launch plan of a force pass over n bodies on the current device."""
    out = (ctypes.c_int64 * len(PLAN_FIELDS))()
    _check(lib().nbody_plan(int(n), int(path), int(split), out, len(PLAN_FIELDS)), "nbody_plan")
    return dict(zip(PLAN_FIELDS, (int(v) for v in out)))


TABLE_FIELDS = ("rows", "targets_per_thread", "threads", "tile", "form_or_acc", "rot")


def table_row(which: int, row: int) -> dict:
    """Shape of row ``row`` of this build's tiled (0), pair (1) or warp (2)
    kernel table; the fields as ``nbody_table`` in nbody.h describes them."""
    out = (ctypes.c_int64 * len(TABLE_FIELDS))()
    _check(lib().nbody_table(int(which), int(row), out, len(TABLE_FIELDS)), "nbody_table")
    return dict(zip(TABLE_FIELDS, (int(v) for v in out)))


def last_plan(stream=None) -> dict:
    """Plan of the last force pass enqueued on the stream (the one that ran,
    after any fallback when the pair path's scratch could not be allocated)."""
    out = (ctypes.c_int64 * len(PLAN_FIELDS))()
    _check(lib().nbody_last_plan(_stream(stream), out, len(PLAN_FIELDS)), "nbody_last_plan")
    return dict(zip(PLAN_FIELDS, (int(v) for v in out)))


PHASES = ("wait", "expand", "own_tiles", "cross_tiles", "reduce", "fold", "other")


def phase_read() -> dict:
    """SM cycles the pair kernel's warps spent in each phase since the last read
    (the profiling build only; others raise NBodyError(EINVAL))."""
    out = (ctypes.c_int64 * len(PHASES))()
    _check(lib().nbody_phase_read(out, len(PHASES)), "nbody_phase_read")
    return dict(zip(PHASES, (int(v) for v in out)))


def release() -> None:
    """Free the library's cached scratch on every device."""
    lib().nbody_release()


def profile_enable(on: bool = True) -> None:
    """Start (or stop) timing force-kernel launches and counting kernel launches."""
    _check(lib().nbody_profile_enable(1 if on else 0), "nbody_profile_enable")


def profile_read() -> tuple[float, int, int]:
    """(force-kernel ms, force-kernel launches, all kernel launches) since the last read."""
    ms = ctypes.c_double(0.0)
    fl = ctypes.c_int64(0)
    kl = ctypes.c_int64(0)
    _check(lib().nbody_profile_read(ctypes.byref(ms), ctypes.byref(fl), ctypes.byref(kl)),
           "nbody_profile_read")
    return float(ms.value), int(fl.value), int(kl.value)


def selftest_timeout(timeout_ms: int = 100, stream=None) -> int:
    """Run the bounded-wait check; a correct build returns ETIMEOUT."""
    return int(lib().nbody_selftest_timeout(int(timeout_ms), _stream(stream)))


def selftest_timeout_enqueue(timeout_ms: int = 100, stream=None) -> int:
    """Enqueue the bounded-wait check without waiting; its ETIMEOUT stays in
    the stream's status word for nbody_sync on that stream."""
    return int(lib().nbody_selftest_timeout_enqueue(int(timeout_ms), _stream(stream)))
