"""Error measures and GPU call helpers shared by the GPU parity tests.

Tolerances (float32 GPU against the float64 oracle on the same float32 bodies):
  accelerations  max_i |a_gpu,i - a_ref,i| / RMS_i |a_ref,i|  <= 1e-4
  positions      max_i |x_gpu,i - x_ref,i| / RMS_i |x_ref,i|  <= 1e-3
|.| is the Euclidean norm of the 3-vector and the RMS runs over the bodies
compared.  Velocities and last-step accelerations of a trajectory are also
held to 1e-4 of their RMS.
"""
from __future__ import annotations

import numpy as np

ACC_TOL = 1e-4
POS_TOL = 1e-3
VEL_TOL = 1e-4


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)[:, :3]
    ref = np.asarray(ref, dtype=np.float64)[:, :3]
    diff = np.linalg.norm(got - ref, axis=1)
    rms = float(np.sqrt(np.mean(np.sum(ref * ref, axis=1))))
    if rms == 0.0:
        return float(diff.max(initial=0.0))
    return float(diff.max(initial=0.0)) / rms


EPS32 = 2.0 ** -23  # one float32 ulp at 1.0


def displacement_err(p_gpu, p_ref, p0, steps: int) -> float:
    """Displacement error over a run, beyond the float32 storage floor.

    The GPU stores positions in float32 after every step, so even exact
    arithmetic leaves up to ~one ulp of |x| per step and component.  The
    excess of |dx_gpu - dx_ref| over steps * ulp(|x_ref|) is returned as a
    fraction of RMS |dx_ref|.
    """
    p0 = np.asarray(p0, dtype=np.float64)[:, :3]
    d_gpu = np.asarray(p_gpu, dtype=np.float64)[:, :3] - p0
    d_ref = np.asarray(p_ref, dtype=np.float64)[:, :3] - p0
    floor = steps * EPS32 * np.sqrt(3.0) * np.linalg.norm(np.asarray(p_ref)[:, :3], axis=1)
    excess = np.maximum(np.linalg.norm(d_gpu - d_ref, axis=1) - floor, 0.0)
    rms = float(np.sqrt(np.mean(np.sum(d_ref * d_ref, axis=1))))
    return float(excess.max(initial=0.0)) / rms


def gpu_accel(pos_mass_np, eps2, path=0, split=0):
    import torch
    import all_pairs_body_gb300 as nb
    pm = torch.from_numpy(np.ascontiguousarray(pos_mass_np, dtype=np.float32)).cuda()
    out = torch.full_like(pm, float("nan"))
    nb.accel(pm, eps2, out=out, path=path, split=split)
    nb.sync()
    return out.cpu().numpy()


def gpu_leapfrog(pos_mass_np, vel_np, eps2, dt, steps, path=0, split=0):
    import torch
    import all_pairs_body_gb300 as nb
    pm = torch.from_numpy(np.ascontiguousarray(pos_mass_np, dtype=np.float32)).cuda()
    v = torch.from_numpy(np.ascontiguousarray(vel_np, dtype=np.float32)).cuda()
    a = torch.full_like(pm, float("nan"))
    nb.leapfrog_step(pm, v, a, eps2, dt, steps, path=path, split=split)
    nb.sync()
    return pm.cpu().numpy(), v.cpu().numpy(), a.cpu().numpy()
