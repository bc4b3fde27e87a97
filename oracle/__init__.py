"""FP64 CPU oracle for the all-pairs softened-gravity sum and leapfrog step.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; the GPU library never uses it and
shares no code with it.  The arithmetic lives in ``nbody_oracle.c`` (plain
double loops, j ascending); this module only marshals NumPy arrays.

Sources: "CUDA N-Body Simulation" (LienoPC/N-BodySimulation README) §1.2 for
the softened sum with G = 1, §1.3 for the half-kick + drift step with
accelerations from the start-of-step coordinates, and for the staggered
leapfrog whose kick-drift-kick form ``leapfrog_kdk`` states.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bodies64(pos_mass) -> np.ndarray:
    pm = np.asarray(pos_mass)
    if pm.ndim != 2 or pm.shape[1] != 4:
        raise ValueError("pos_mass must be (n, 4) rows of x, y, z, m")
    return np.ascontiguousarray(pm, dtype=np.float64)


class Oracle:
    """A loaded copy of the oracle library (the default one, or a test build)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        d, i64, i32, p = ctypes.c_double, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_threads.argtypes = [i32]
        lib.oracle_threads.restype = i32
        lib.oracle_accel.argtypes = [p, i64, d, p, i64, p, i32]
        lib.oracle_accel.restype = i32
        lib.oracle_leapfrog.argtypes = [p, p, p, i64, d, d, i32, i32]
        lib.oracle_leapfrog.restype = i32
        lib.oracle_leapfrog_kdk.argtypes = [p, p, p, i64, d, d, i32, i32]
        lib.oracle_leapfrog_kdk.restype = i32
        lib.oracle_step_sampled.argtypes = [p, p, i64, d, d, p, i64, p, p, p, i32]
        lib.oracle_step_sampled.restype = i32
        lib.oracle_render_points.argtypes = [p, i64, d, d, d, d, d, p, p]
        lib.oracle_render_points.restype = i32
        lib.oracle_neighbors_2d.argtypes = [p, p, i64, ctypes.c_float, i32, p, i64, p, p, i32]
        lib.oracle_neighbors_2d.restype = i32
        self.lib = lib
        self.path = path

    def threads(self, requested: int = 0) -> int:
        """Threads a call with ``requested`` threads (0 = all cores) uses."""
        return int(self.lib.oracle_threads(int(requested)))

    def accel(self, pos_mass, eps2: float, idx=None, threads: int = 0) -> np.ndarray:
        """FP64 accelerations a_i = sum_j m_j r_ij / (|r_ij|^2 + eps2)^(3/2).

        ``pos_mass``: (n, 4) rows (x, y, z, m), any float dtype (widened to
        fp64).  ``idx``: optional indices of the target bodies; every source
        body is always summed.  Returns (len(idx) or n, 3) float64.
        """
        pm = _bodies64(pos_mass)
        n = pm.shape[0]
        if idx is None:
            idx_arr, n_idx = None, n
        else:
            idx_arr = np.ascontiguousarray(idx, dtype=np.int64)
            n_idx = idx_arr.shape[0]
        out = np.zeros((n_idx, 3), dtype=np.float64)
        rc = self.lib.oracle_accel(_ptr(pm), n, float(eps2),
                                   None if idx_arr is None else _ptr(idx_arr), n_idx,
                                   _ptr(out), int(threads))
        if rc < 0:
            raise ValueError("oracle_accel: bad argument")
        return out

    def leapfrog(self, pos_mass, vel, eps2: float, dt: float, steps: int,
                 threads: int = 0):
        """FP64 leapfrog: per step a = A(x) for all bodies, then v += dt/2 a, x += dt v.

        ``vel`` may be (n, 3) or (n, 4) (only xyz is used).  Returns
        ``(pos_mass (n,4), vel (n,3), acc (n,3))`` in float64; ``acc`` is the
        acceleration of the last step (zeros when ``steps`` is 0).
        """
        pm = _bodies64(pos_mass).copy()
        v = np.ascontiguousarray(np.asarray(vel, dtype=np.float64)[:, :3]).copy()
        n = pm.shape[0]
        if v.shape[0] != n:
            raise ValueError("vel must have one row per body")
        acc = np.zeros((n, 3), dtype=np.float64)
        rc = self.lib.oracle_leapfrog(_ptr(pm), _ptr(v), _ptr(acc), n, float(eps2),
                                      float(dt), int(steps), int(threads))
        if rc < 0:
            raise ValueError("oracle_leapfrog: bad argument")
        return pm, v, acc


    def step_sampled(self, pos_mass, vel, eps2: float, dt: float, idx, threads: int = 0):
        """One half-kick + drift step for the bodies ``idx`` only (their rows of
        ``leapfrog(..., steps=1)``): returns ``(pos_mass (k,4), vel (k,3), acc (k,3))``
        in float64."""
        pm = _bodies64(pos_mass)
        n = pm.shape[0]
        v = np.ascontiguousarray(np.asarray(vel, dtype=np.float64)[:, :3])
        if v.shape[0] != n:
            raise ValueError("vel must have one row per body")
        idx_arr = np.ascontiguousarray(idx, dtype=np.int64)
        m = idx_arr.shape[0]
        pos_out = np.empty((m, 4), dtype=np.float64)
        vel_out = np.empty((m, 3), dtype=np.float64)
        acc_out = np.empty((m, 3), dtype=np.float64)
        rc = self.lib.oracle_step_sampled(_ptr(pm), _ptr(v), n, float(eps2), float(dt),
                                          _ptr(idx_arr), m, _ptr(pos_out), _ptr(vel_out),
                                          _ptr(acc_out), int(threads))
        if rc < 0:
            raise ValueError("oracle_step_sampled: bad argument")
        return pos_out, vel_out, acc_out

    def leapfrog_kdk(self, pos_mass, vel, eps2: float, dt: float, steps: int,
                     threads: int = 0):
        """FP64 kick-drift-kick leapfrog (closing half-kick with a(x(t+dt))).

        Same arguments and returns as ``leapfrog``; ``acc`` is A at the final
        positions (zeros when ``steps`` is 0).
        """
        pm = _bodies64(pos_mass).copy()
        v = np.ascontiguousarray(np.asarray(vel, dtype=np.float64)[:, :3]).copy()
        n = pm.shape[0]
        if v.shape[0] != n:
            raise ValueError("vel must have one row per body")
        acc = np.zeros((n, 3), dtype=np.float64)
        rc = self.lib.oracle_leapfrog_kdk(_ptr(pm), _ptr(v), _ptr(acc), n, float(eps2),
                                          float(dt), int(steps), int(threads))
        if rc < 0:
            raise ValueError("oracle_leapfrog_kdk: bad argument")
        return pm, v, acc


    def render_points(self, pos_mass, max_xyz, min_w: float, max_w: float):
        """CPU restatement of the point shaders ("CUDA N-Body Simulation"
        §4.3): returns (ndc (n,4), rgba (n,4)) in float64."""
        pm = _bodies64(pos_mass)
        n = pm.shape[0]
        ndc = np.zeros((n, 4))
        rgba = np.zeros((n, 4))
        mx, my, mz = (float(v) for v in max_xyz)
        rc = self.lib.oracle_render_points(_ptr(pm), n, mx, my, mz, float(min_w), float(max_w),
                                           _ptr(ndc), _ptr(rgba))
        if rc < 0:
            raise ValueError("oracle_render_points: bad argument")
        return ndc, rgba


    def neighbors_2d(self, x, y, cutoff: float, max_neighbors: int, idx=None, threads: int = 0):
        """All-pairs 2-D cutoff neighbour list in float32 ("CUDA编程（九）" §3):
        returns (nn (m,) int32, nl (max_neighbors, m) int32, -1 = empty) for
        the m targets ``idx`` (all n points when None)."""
        xs = np.ascontiguousarray(x, dtype=np.float32)
        ys = np.ascontiguousarray(y, dtype=np.float32)
        n = xs.shape[0]
        if ys.shape[0] != n:
            raise ValueError("x and y must have the same length")
        idx_arr = None if idx is None else np.ascontiguousarray(idx, dtype=np.int64)
        m = n if idx_arr is None else idx_arr.shape[0]
        nn = np.zeros(m, dtype=np.int32)
        nl = np.zeros((max(int(max_neighbors), 0), m), dtype=np.int32)
        rc = self.lib.oracle_neighbors_2d(_ptr(xs), _ptr(ys), n, float(cutoff),
                                          int(max_neighbors),
                                          None if idx_arr is None else _ptr(idx_arr), m,
                                          _ptr(nn), _ptr(nl), int(threads))
        if rc < 0:
            raise ValueError("oracle_neighbors_2d: bad argument")
        return nn, nl


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def threads(requested: int = 0) -> int:
    return default().threads(requested)


def accel(pos_mass, eps2: float, idx=None, threads: int = 0) -> np.ndarray:
    return default().accel(pos_mass, eps2, idx, threads)


def leapfrog(pos_mass, vel, eps2: float, dt: float, steps: int, threads: int = 0):
    return default().leapfrog(pos_mass, vel, eps2, dt, steps, threads)


def leapfrog_kdk(pos_mass, vel, eps2: float, dt: float, steps: int, threads: int = 0):
    return default().leapfrog_kdk(pos_mass, vel, eps2, dt, steps, threads)


def step_sampled(pos_mass, vel, eps2: float, dt: float, idx, threads: int = 0):
    return default().step_sampled(pos_mass, vel, eps2, dt, idx, threads)


def render_points(pos_mass, max_xyz, min_w: float, max_w: float):
    return default().render_points(pos_mass, max_xyz, min_w, max_w)


def neighbors_2d(x, y, cutoff: float, max_neighbors: int, idx=None, threads: int = 0):
    return default().neighbors_2d(x, y, cutoff, max_neighbors, idx, threads)
