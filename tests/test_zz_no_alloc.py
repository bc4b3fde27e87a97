"""nbody_accel_noalloc: accelerations for callers that cannot allocate.

Some callers may not allocate GPU memory when they need accelerations (an
allocator that is off limits during stream capture, a host that owns all
device memory through its own pool, a real-time loop that bans allocation
after start-up).  nbody_accel_noalloc serves them from one fixed device array
that the library holds for the life of the process.  These tests call it
through the C ABI and compare it with the allocating entry point,
nbody_accel_on_stream, on two calls in a row: the second call is smaller, so
anything the first call left in the shared array must not leak into it.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from parity import ACC_TOL, rel_err

P = ctypes.c_void_p


def test_noalloc_rejects_sizes_beyond_the_array():
    import all_pairs_body_gb300 as nb
    from all_pairs_body_gb300 import build as nbuild
    nbuild.build()
    L = nb.lib()
    # host-side checks: nothing is touched on any device
    assert L.nbody_accel_noalloc(P(0x10000), P(0x20000), nb.NOALLOC_MAX_N + 1,
                                 ctypes.c_float(1e-3), P(0)) == nb.EINVAL
    assert L.nbody_accel_noalloc(P(0x10000), P(0x10000), 16, ctypes.c_float(1e-3), P(0)) == nb.EINVAL
    assert L.nbody_accel_noalloc(None, None, 0, ctypes.c_float(1e-3), P(0)) == nb.OK


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_two_calls_in_a_row():
    import torch

    import all_pairs_body_gb300 as nb
    from all_pairs_body_gb300 import build as nbuild
    nbuild.build()
    L = nb.lib()
    stream = torch.cuda.current_stream()
    s = P(stream.cuda_stream)
    for n, seed in [(nb.NOALLOC_MAX_N, 31), (4097, 32)]:
        pm = torch.from_numpy(W.random_bodies(n, seed)).cuda()
        out_noalloc = torch.full_like(pm, float("nan"))
        out_ref = torch.full_like(pm, float("nan"))
        assert L.nbody_accel_noalloc(P(pm.data_ptr()), P(out_noalloc.data_ptr()), n,
                                     ctypes.c_float(1e-3), s) == nb.OK
        assert L.nbody_accel_on_stream(P(pm.data_ptr()), P(out_ref.data_ptr()), n,
                                       ctypes.c_float(1e-3), s) == nb.OK
        nb.sync(stream)
        got = out_noalloc.cpu().numpy()
        ref = out_ref.cpu().numpy()
        assert np.all(np.isfinite(got)) and np.all(got[:, 3] == 0.0)
        assert rel_err(got, ref) <= ACC_TOL, (n, rel_err(got, ref))
