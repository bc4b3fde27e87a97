"""nbody_accel_noalloc: accelerations for callers that cannot allocate.

Some callers may not allocate GPU memory at the point where they need
accelerations: a host application that hands all device memory to its own
pool and forbids other allocations, or a real-time loop that bans allocation
after start-up because cudaMalloc may block or synchronise the device.
nbody_accel_noalloc serves them from one fixed device array that the library
holds for the life of the process.  These tests call it through the C ABI and
compare it with the allocating entry point, nbody_accel_on_stream, and with
the FP64 oracle, on calls in a row of decreasing size, so anything one call
left in the shared array must not leak into the next; the smallest size is
finished by the CTAs themselves, without the second pass.  Once the first
call has set up the device, the free device memory must not change across
further calls.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import oracle
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
def test_noalloc_matches_allocating_entry_point_calls_in_a_row():
    import torch

    import all_pairs_body_gb300 as nb
    from all_pairs_body_gb300 import build as nbuild
    nbuild.build()
    L = nb.lib()
    stream = torch.cuda.current_stream()
    s = P(stream.cuda_stream)
    cases = [(nb.NOALLOC_MAX_N, 31), (4097, 32), (100, 33)]
    bodies = [W.random_bodies(n, seed) for n, seed in cases]
    inputs = [torch.from_numpy(b).cuda() for b in bodies]
    outs = [torch.full_like(pm, float("nan")) for pm in inputs]
    refs = [torch.full_like(pm, float("nan")) for pm in inputs]
    # the first call on the device sets it up (and may load the library's
    # device code); every call after it must leave free memory unchanged
    assert L.nbody_accel_noalloc(P(inputs[2].data_ptr()), P(outs[2].data_ptr()), 100,
                                 ctypes.c_float(1e-3), s) == nb.OK
    nb.sync(stream)
    free_before = torch.cuda.mem_get_info()[0]
    for pm, out in zip(inputs, outs):
        n = pm.shape[0]
        assert L.nbody_accel_noalloc(P(pm.data_ptr()), P(out.data_ptr()), n,
                                     ctypes.c_float(1e-3), s) == nb.OK
        nb.sync(stream)
    assert torch.cuda.mem_get_info()[0] == free_before
    for pm, ref in zip(inputs, refs):
        assert L.nbody_accel_on_stream(P(pm.data_ptr()), P(ref.data_ptr()), pm.shape[0],
                                       ctypes.c_float(1e-3), s) == nb.OK
    nb.sync(stream)
    for (n, _), b, out, ref in zip(cases, bodies, outs, refs):
        got = out.cpu().numpy()
        want = ref.cpu().numpy()
        assert np.all(np.isfinite(got)) and np.all(got[:, 3] == 0.0)
        assert rel_err(got, want) <= ACC_TOL, (n, rel_err(got, want))
        idx = None if n <= 4097 else np.random.default_rng(n).choice(n, 4096, replace=False)
        exact = oracle.accel(b, 1e-3, idx=idx)
        assert rel_err(got if idx is None else got[idx], exact) <= ACC_TOL, n
