"""The index-checked build (NBODY_BOUNDS_CHECK) on every path.

In that build each computed index into the bodies' rows, the split sums
(`partial`), the pair kernel's reaction rows and the neighbour list is
compared on the device with the capacity the host allocated; an index
outside it is not used (the access is skipped) and NBODY_EBOUNDS is
recorded for nbody_sync.  These tests run every entry point of that build at
ragged sizes, chunked pair passes included, and require both a clean status
and oracle parity, so that no kernel computes an index beyond what its
caller allocated.  NBODY_BOUNDS_SHRINK sets one capacity to zero so that the
checks can be seen to fire; every access they stop is skipped, so the
shrunk runs stay inside their arrays too.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import ACC_TOL, POS_TOL, VEL_TOL, gpu_accel, gpu_leapfrog, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def checked_lib():
    """Route the binding through the checked build for this module."""
    import torch
    import all_pairs_body_gb300 as nb
    from all_pairs_body_gb300 import build as nbuild
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()
    path = nbuild.build(checked=True)
    saved = nb._lib
    nb._lib = nb.load(path)
    try:
        yield nb._lib
    finally:
        nb.release()
        nb._lib = saved


_REF = {}


@pytest.mark.parametrize("path,split", [(0, 0), (1, 0), (2, 0), (2, 3), (3, 0), (3, 5), (4, 0)])
@pytest.mark.parametrize("n", [1, 33, 513, 2049, 9000, 20000, 65537])
def test_checked_accel(n, path, split):
    pm = W.random_bodies(n, 9100 + n)
    a = gpu_accel(pm, 1e-2, path, split)  # gpu_accel syncs: EBOUNDS would raise
    if n == 1:
        assert np.all(a == 0.0)
        return
    if n not in _REF:
        _REF[n] = oracle.accel(pm, 1e-2)
    assert rel_err(a, _REF[n]) <= ACC_TOL


@pytest.mark.parametrize("path", [1, 4])
def test_checked_large_sampled(path):
    w = W.ball_lognormal_1048576()
    a = gpu_accel(w.pos_mass, w.eps2, path)
    ref = oracle.accel(w.pos_mass, w.eps2, idx=w.sample)
    assert rel_err(a[w.sample], ref) <= ACC_TOL


@pytest.mark.parametrize("n,cap", [(20000, 1), (30001, 300000)])
def test_checked_pair_chunks(n, cap, monkeypatch):
    import all_pairs_body_gb300 as nb
    monkeypatch.setenv("NBODY_PAIRS_MAX_BYTES", str(cap))
    assert nb.plan(n, path=nb.PATH_PAIRS)["launches_accel"] > 2
    pm = W.random_bodies(n, 9200 + n)
    a = gpu_accel(pm, 1e-3, path=4)
    assert rel_err(a, oracle.accel(pm, 1e-3)) <= ACC_TOL


# auto (the one-kernel warp pass and copy_rows), the one-sided paths (one
# kernel, and stream-K with its second pass), the sliced warp pass and the pair
# path (drift in place)
@pytest.mark.parametrize("path,split", [(0, 0), (1, 0), (2, 3), (3, 5), (4, 0)])
def test_checked_leapfrog_and_kdk(path, split):
    import torch
    import all_pairs_body_gb300 as nb
    n = 9000
    pm = W.random_bodies(n, 9300)
    v = W.random_velocities(n, 9300)
    p, vv, a = gpu_leapfrog(pm, v, 1e-3, 1e-3, 3, path, split)
    rp, rv, ra = oracle.leapfrog(pm, v, 1e-3, 1e-3, 3)
    assert rel_err(a, ra) <= ACC_TOL and rel_err(vv, rv) <= VEL_TOL and rel_err(p, rp) <= POS_TOL
    tp = torch.from_numpy(pm).cuda()
    tv = torch.from_numpy(v).cuda()
    ta = torch.empty_like(tp)
    nb.leapfrog_kdk(tp, tv, ta, 1e-3, 1e-3, 3, path=path, split=split)
    nb.sync()
    kp, kv, ka = oracle.leapfrog_kdk(pm, v, 1e-3, 1e-3, 3)
    assert rel_err(ta.cpu().numpy(), ka) <= ACC_TOL
    assert rel_err(tv.cpu().numpy(), kv) <= VEL_TOL
    assert rel_err(tp.cpu().numpy(), kp) <= POS_TOL


@pytest.mark.parametrize("n", [1, 1000, 65536])
def test_checked_noalloc(n):
    import torch
    import all_pairs_body_gb300 as nb
    pm = W.random_bodies(n, 9400 + n)
    out = torch.full((n, 4), float("nan"), device="cuda")
    nb.accel_noalloc(torch.from_numpy(pm).cuda(), out, 1e-2)
    nb.sync()
    a = out.cpu().numpy()
    if n == 1:
        assert np.all(a == 0.0)
    else:
        assert rel_err(a, oracle.accel(pm, 1e-2)) <= ACC_TOL


@pytest.mark.parametrize("layout", [1, 2])
def test_checked_layouts(layout):
    import torch
    import all_pairs_body_gb300 as nb
    n = 40000
    pm = W.random_bodies(n, 9500)
    tp = torch.from_numpy(pm).cuda()
    out = torch.empty(3 * n, device="cuda")
    nb.accel_layout(tp, out, 1e-2, layout)
    nb.sync()
    got = out.cpu().numpy().reshape(n, 3) if layout == 1 else out.cpu().numpy().reshape(3, n).T
    assert rel_err(got, oracle.accel(pm, 1e-2)) <= ACC_TOL


def test_checked_render():
    import torch
    import all_pairs_body_gb300 as nb
    n = 5000
    pm = W.random_bodies(n, 9600)
    ndc, rgba = nb.render_points(torch.from_numpy(pm).cuda(), (1.5, 1.5, 1.5), 0.0, 2.0)
    nb.sync()
    rn, rr = oracle.render_points(pm, (1.5, 1.5, 1.5), 0.0, np.float32(2.0))
    for got, ref in ((ndc, rn), (rgba, rr)):
        ref = np.asarray(ref, dtype=np.float64)
        err = np.abs(got.cpu().numpy().astype(np.float64) - ref) / np.maximum(1.0, np.abs(ref))
        assert float(err.max()) <= 2e-6


@pytest.mark.parametrize("n,mn", [(1, 4), (20000, 3), (20000, 64)])
def test_checked_neighbors(n, mn):
    import torch
    import all_pairs_body_gb300 as nb
    p = W.points_2d(n)
    nn, nl = nb.neighbors_2d(torch.from_numpy(p.x).cuda(), torch.from_numpy(p.y).cuda(),
                             p.cutoff, mn)
    nb.sync()
    rn, rl = oracle.neighbors_2d(p.x, p.y, p.cutoff, mn)
    assert np.array_equal(nn.cpu().numpy(), rn) and np.array_equal(nl.cpu().numpy(), rl)


def _accel_call(path, split):
    def run():
        pm = W.random_bodies(20000, 9700)
        return gpu_accel(pm, 1e-2, path, split)
    return run


def _step_call(path, split):
    def run():
        pm = W.random_bodies(9000, 9800)
        v = W.random_velocities(9000, 9800)
        return gpu_leapfrog(pm, v, 1e-3, 1e-3, 3, path, split)
    return run


def _neighbors_call():
    import torch
    import all_pairs_body_gb300 as nb
    p = W.points_2d(5000)
    nn, nl = nb.neighbors_2d(torch.from_numpy(p.x).cuda(), torch.from_numpy(p.y).cuda(),
                             p.cutoff, 8)
    nb.sync()


@pytest.mark.parametrize("slot,call", [
    ("rows", _accel_call(1, 0)),
    ("partial", _accel_call(2, 3)),
    ("partial", _accel_call(3, 5)),
    ("react", _accel_call(4, 0)),
    ("rows", _step_call(0, 0)),
    ("rows", _step_call(4, 0)),
    ("neighbors", _neighbors_call),
])
def test_shrunk_capacity_reports_ebounds(slot, call, monkeypatch):
    """With one capacity at zero the checks stop the accesses, nbody_sync
    returns NBODY_EBOUNDS once, and the next call runs clean."""
    import all_pairs_body_gb300 as nb
    monkeypatch.setenv("NBODY_BOUNDS_SHRINK", slot)
    with pytest.raises(nb.NBodyError) as e:
        call()
    assert e.value.status == nb.EBOUNDS
    monkeypatch.delenv("NBODY_BOUNDS_SHRINK")
    nb.sync()
    pm = W.random_bodies(20000, 9700)
    a = gpu_accel(pm, 1e-2, 4)
    assert rel_err(a, oracle.accel(pm, 1e-2)) <= ACC_TOL
