#!/usr/bin/env python3
"""Throughput of the all-pairs softened-gravity step on GB300, one JSON line.

Workload (default): 2^20 bodies uniform in the unit ball with log-normal
masses (total 1), seed 3, eps2 = 1e-3.  One step = one leapfrog kick/drift
step through the C ABI: the all-pairs acceleration over every (i, j) pair
plus the fused half-kick and drift ("CUDA N-Body Simulation" §1.2-1.3), i.e.
N^2 body-body interactions per step.

    value    = interactions of all ranks / max-over-ranks device time,
               in billions of interactions per second (CUDA events on the
               launching stream; L2 flushed by a 512 MiB write between steps,
               which also keeps the host ahead of the device at small N)
    e2e      = the same metric with host (pinned) buffers: each step copies
               positions and velocities in, runs the step and copies
               positions, velocities and accelerations back
    roofline = the force kernel alone against the FP32 issue roofline
               SMs x f_SM x 128 lanes / FP32 lane-ops per interaction: 12 for
               the one-sided kernels, 8 for the pair-symmetric kernel (16 per
               pair, which serves two interactions)
    cpu_baseline = the FP64 CPU oracle on a bounded sample of the same bodies

``--impl reference`` times the FP64 CPU oracle on the host cores instead.
Multi-GPU (torchrun) runs independent replicas, one per rank.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "body-body interactions/s (billions) at N=2^20 FP32; % of FFMA/MUFU roofline"
UNIT = "Ginteractions/s"
DEFAULT_WORKLOAD = "ball-lognormal-1048576"
FLOP_PER_INTERACTION = 20  # bodybodyinteraction FLOP comments, "Cuda Nbody Notes"
FP32_OPS_PER_INTERACTION = 12  # 3 FADD + 3 FFMA (|r|^2+eps2) + 3 FMUL (m q^3) + 3 FFMA (a += s r)
# pair-symmetric kernel, per pair (two interactions): 3 FADD + 3 FFMA + 2 FMUL (q^3)
# + 2 FMUL (both mass factors) + 6 FFMA (action and reaction) = 16
FP32_OPS_PER_INTERACTION_PAIRS = 8
FP32_LANES_PER_SM = 128  # per clock: 4 SM sub-partitions x 32 FP32 lanes
# > 129 MB L2; 512 MiB takes ~80 us of device time, longer than the host needs
# to issue the next flush, event and call, so a small step's time is its own
FLUSH_BYTES = 512 << 20
PROFILE_SUMMARIES = {  # force kernel -> committed ncu summary of one launch
    "force_tiled": os.path.join(ROOT, "profiles", "force_tiled_ball-lognormal-1048576.md"),
    "force_pairs": os.path.join(ROOT, "profiles", "force_pairs_ball-lognormal-1048576.md"),
}
KERNEL_SOURCE = os.path.join(ROOT, "all_pairs_body_gb300", "csrc", "nbody_kernels.cuh")
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--mode", choices=("step", "accel", "kdk", "render", "neighbors"),
                    default="step",
                    help="step: one leapfrog kick/drift step (default); accel: acceleration "
                         "only; kdk: one kick-drift-kick step (two force passes); render: the "
                         "point-shader kernel (memory-bound, reported in GB/s); neighbors: the "
                         "2-D cutoff neighbour list (pair tests/s; default points2d-1048576)")
    ap.add_argument("--path", choices=("auto", "tiled", "split", "warp", "pairs"), default="auto",
                    help="force-pass path for --mode step|accel|kdk (the library's choice by "
                         "default); NBODY_TILED_CONFIG selects a row of the tiled-kernel table")
    ap.add_argument("--split", type=int, default=0,
                    help="j slices per target block for --path split|warp (0: library's choice)")
    ap.add_argument("--layout", choices=("rows4", "rows3", "blocks3"), default="rows4",
                    help="velocity/acceleration layout for --mode step|accel (float4 rows, "
                         "float3 rows, or x/y/z blocks)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other benchmark configurations measured after the "
                         "default workload (the line's \"configs\")")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--phases", action="store_true",
                    help="load the profiling build (clock64 stamps around the phases of the "
                         "pair kernel's tiles) and add the cycle split to the line; its timings "
                         "are not the release library's")
    ap.add_argument("--tuning", action="store_true",
                    help="load the tuning build (every measured kernel shape, selected with "
                         "NBODY_TILED_CONFIG / NBODY_PAIRS_CONFIG / NBODY_WARP_CONFIG) instead of "
                         "the release library")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return rank, local, world


def init_dist(world: int, use_cuda: bool):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return dist


def reduce_max(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (the value itself without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def aggregate_value(per_rank_interactions: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput (billions/s): every rank does the same work."""
    return world * per_rank_interactions / max_seconds / 1e9


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------


def gpu_selector(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis.strip():
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


class ClockSampler:
    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", self.gpu],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_lines(out.splitlines())


def parse_clock_lines(lines) -> dict | None:
    sm, smax, power, reasons = [], [], [], set()
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            smax.append(float(f[2]))
            power.append(float(f[3]))
        except ValueError:
            continue
        for name, val in zip(REASON_NAMES, f[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
            "reasons": sorted(reasons), "samples": len(sm),
            "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# roofline
# ---------------------------------------------------------------------------


def measured_sm_max_mhz(clocks: dict | None) -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["sm_max_mhz"])
            return v, "MEASURED_PEAKS.json sm_max_mhz"
    except (OSError, KeyError, ValueError, TypeError):
        pass
    if clocks and clocks.get("sm_max_mhz"):
        return float(clocks["sm_max_mhz"]), "nvidia-smi clocks.max.sm"
    return 2070.0, "fallback maximum SM clock"


def alu_peak_ginter(sms: int, mhz: float, ops: int = FP32_OPS_PER_INTERACTION) -> float:
    """FP32 issue roofline in billions of interactions/s at `ops` FP32
    lane-ops per interaction."""
    return sms * mhz * 1e6 * FP32_LANES_PER_SM / ops / 1e9


def kernel_source_digest() -> str:
    """First 16 hex digits of the SHA-256 of the kernel source's code: the
    file with its // comments and blank lines left out, so that an edit to
    the comments alone keeps the committed ncu figures."""
    with open(KERNEL_SOURCE, encoding="utf-8") as f:
        lines = [ln.split("//", 1)[0].rstrip() for ln in f.read().splitlines()]
    code = "\n".join(ln for ln in lines if ln.strip())
    return hashlib.sha256(code.encode("utf-8")).hexdigest()[:16]


def profiled_traffic(n: int, kernel: str = "force_tiled") -> float | None:
    """DRAM bytes per force-kernel launch from the committed ncu summary,
    scaled to n bodies (by n, or n^2 where the summary says the traffic grows
    so), or None if there is no summary or the kernel changed since."""
    try:
        text = open(PROFILE_SUMMARIES[kernel]).read()
    except (OSError, KeyError):
        return None
    fields = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    try:
        if fields.get("kernel_source_sha256_16") != kernel_source_digest():
            return None
        bytes_captured = float(fields["dram_bytes_per_launch"])
        n_captured = float(fields["n_captured"])
    except (KeyError, ValueError):
        return None
    power = 2 if fields.get("traffic_scales_as") == "n^2" else 1
    return bytes_captured * (n / n_captured) ** power


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------


# accelerations: max_i |a_gpu,i - a_ref,i| / RMS_i |a_ref,i| (3-vectors) must not pass this
ACC_TOL = 1e-4


def parity_errors(got, ref) -> tuple[float, float]:
    """(max, RMS) over the bodies of |a_got,i - a_ref,i| / RMS_i |a_ref,i|,
    |.| the Euclidean norm of the 3-vector."""
    import numpy as np
    got = np.asarray(got, dtype=np.float64)[:, :3]
    ref = np.asarray(ref, dtype=np.float64)[:, :3]
    diff = np.linalg.norm(got - ref, axis=1)
    scale = float(np.sqrt(np.mean(np.sum(ref * ref, axis=1)))) if len(ref) else 0.0
    scale = scale if scale > 0.0 else 1.0
    return (float(diff.max(initial=0.0)) / scale,
            float(np.sqrt(np.mean(diff * diff))) / scale if len(diff) else 0.0)


def oracle_sample_rate(pos_mass, eps2: float, seconds: float, seed: int):
    """FP64 oracle on seeded target samples x all sources; returns
    (Ginteractions/s, targets, threads, wall seconds, target indices, their
    accelerations)."""
    import numpy as np

    import oracle
    n = pos_mass.shape[0]
    rng = np.random.default_rng(seed)
    # enough targets to keep every OpenMP thread busy while calibrating
    probe = np.sort(rng.choice(n, size=min(16 * oracle.threads(), n), replace=False))
    t0 = time.perf_counter()
    oracle.accel(pos_mass, eps2, idx=probe)
    per_target = (time.perf_counter() - t0) / len(probe)
    k = int(max(64, min(n, seconds / max(per_target, 1e-9))))
    idx = np.sort(rng.choice(n, size=k, replace=False))
    t0 = time.perf_counter()
    ref = oracle.accel(pos_mass, eps2, idx=idx)
    wall = time.perf_counter() - t0
    return k * n / wall / 1e9, k, oracle.threads(), wall, idx, ref


MODE_TEXT = {
    "step": "one leapfrog kick/drift step (all-pairs acceleration + fused half-kick and drift, "
            "dt={dt:g}); N^2 interactions per step",
    "accel": "one all-pairs acceleration evaluation; N^2 interactions per step",
    "kdk": "one kick-drift-kick step (two all-pairs passes: half kick + drift, then the closing "
           "half kick, dt={dt:g}); 2 N^2 interactions per step",
    "render": "one pass of the point-shader kernel (NDC + mass colour); 48 bytes per body",
    "neighbors": "one all-pairs 2-D cutoff neighbour list",
}


def workload_config(w, mode: str, world: int) -> dict:
    what = MODE_TEXT[mode].format(dt=w.dt)
    return {
        "workload": f"{w.name}: N={w.n} bodies, eps2={w.eps2:g}, seed {w.seed}; each step is {what}",
        "n_bodies": w.n,
        "l2": "flushed between timed steps (512 MiB write); sources 16N bytes",
        "parallelism": "replicas" if world > 1 else "single GPU",
    }


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


# The benchmark's other configurations, measured after the default workload in
# the same process (rank 0 of a one-GPU run): (workload, mode, path, calls,
# warm-up calls, steps per call).  C1 (an acceleration and a step), C2 and C3
# (trajectories: 10 steps per call), C5 (accelerations), and at 2^20 the
# one-sided kernel's step and the kick-drift-kick step.
OTHER_CONFIGS = (
    ("uniform-cube-1024", "accel", "auto", 200, 10, 1),
    ("uniform-cube-1024", "step", "auto", 200, 10, 1),
    ("plummer-16384", "step", "auto", 10, 2, 10),
    ("two-plummer-131072", "step", "auto", 3, 1, 10),
    ("cube-sweep-1000", "accel", "auto", 200, 10, 1),
    ("cube-sweep-4097", "accel", "auto", 200, 10, 1),
    ("cube-sweep-65537", "accel", "auto", 10, 3, 1),
    ("cube-sweep-500000", "accel", "auto", 5, 2, 1),
    ("cube-sweep-4194304", "accel", "auto", 1, 1, 1),
    ("ball-lognormal-1048576", "step", "split", 3, 1, 1),
    ("ball-lognormal-1048576", "kdk", "auto", 1, 1, 1),
)
RENDER_CONFIG = ("ball-lognormal-16777216", 20, 3)  # point-shader kernel: workload, calls, warm-up
NEIGHBOR_CONFIG = ("points2d-1048576", 3, 1)  # 2-D neighbour list


def measure_configs(nb, torch, stream, flush, sms: int, f_max: float) -> list[dict]:
    """Per-call device time of each OTHER_CONFIGS entry, timed like the main
    line (CUDA events around each call, the L2 flushed before it), and its
    force kernel alone from a second, profiled run of the same calls."""
    import workloads
    paths = {"auto": nb.PATH_AUTO, "split": nb.PATH_SPLIT}
    out = []
    for name, mode, path_name, calls, warm, steps in OTHER_CONFIGS:
        w = workloads.by_name(name)
        n, path = w.n, paths[path_name]
        pm = torch.from_numpy(w.pos_mass).cuda()
        vel = torch.from_numpy(w.vel).cuda()
        acc = torch.empty_like(pm)

        def call():
            if mode == "step":
                nb.leapfrog_step(pm, vel, acc, w.eps2, w.dt, steps, path=path)
            elif mode == "kdk":
                nb.leapfrog_kdk(pm, vel, acc, w.eps2, w.dt, steps, path=path)
            else:
                nb.accel(pm, w.eps2, out=acc, path=path)

        for _ in range(warm):
            call()
        nb.sync()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(calls)]
        nb.profile_read()
        torch.cuda.synchronize()
        for s, e in ev:
            flush.zero_()
            s.record(stream)
            call()
            e.record(stream)
        torch.cuda.synchronize()
        nb.sync()
        _, _, launches = nb.profile_read()
        call_s = sum(s.elapsed_time(e) for s, e in ev) / 1e3 / calls
        plan = nb.last_plan()
        nb.profile_enable(True)
        nb.profile_read()
        for _ in range(calls):
            flush.zero_()
            call()
        torch.cuda.synchronize()
        nb.sync()
        force_ms, force_launches, _ = nb.profile_read()
        nb.profile_enable(False)
        passes = force_launches / max(plan["chunks"], 1) if force_launches else 0
        force_s = force_ms / 1e3 / passes if passes else None
        inter = float(n) * float(n)  # per force pass; a kick-drift-kick step takes two
        per_call = float(steps) * (2.0 if mode == "kdk" else 1.0)  # force passes per call
        kernel = {nb.PATH_WARP: "force_warp", nb.PATH_PAIRS: "force_pairs"}.get(plan["path"],
                                                                             "force_tiled")
        ops = FP32_OPS_PER_INTERACTION_PAIRS if kernel == "force_pairs" else FP32_OPS_PER_INTERACTION
        r_one_sided = alu_peak_ginter(sms, f_max)
        force_rate = inter / force_s / 1e9 if force_s else None
        out.append({
            "workload": name, "mode": mode, "path": path_name, "n": n, "calls": calls,
            "steps_per_call": steps, "us_per_call": 1e6 * call_s,
            "us_per_step": 1e6 * call_s / steps if mode != "accel" else None,
            "value": per_call * inter / call_s / 1e9, "unit": UNIT,
            "kernel": kernel, "force_us_per_pass": 1e6 * force_s if force_s else None,
            "call_over_force": call_s / (per_call * force_s) if force_s else None,
            "force_frac_of_R": force_rate / r_one_sided if force_rate else None,
            "force_frac_of_own_roofline": (force_rate / alu_peak_ginter(sms, f_max, ops)
                                           if force_rate else None),
            "kernels_per_call": launches / calls,
        })
        del pm, vel, acc
    out.append(measure_render(nb, torch, stream, flush))
    out.append(measure_neighbors(nb, torch, stream, flush, sms, f_max))
    return out


def timed_calls(torch, stream, flush, call, calls: int, warm: int) -> float:
    """Mean device seconds per call, CUDA events around each, L2 flushed before it."""
    for _ in range(warm):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(calls)]
    torch.cuda.synchronize()
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        call()
        e.record(stream)
    torch.cuda.synchronize()
    return sum(s.elapsed_time(e) for s, e in ev) / 1e3 / calls


def measure_render(nb, torch, stream, flush) -> dict:
    """The point-shader kernel: 16 bytes read and 32 written per body."""
    import workloads
    name, calls, warm = RENDER_CONFIG
    w = workloads.by_name(name)
    pm = torch.from_numpy(w.pos_mass).cuda()
    ndc = torch.empty_like(pm)
    rgba = torch.empty_like(pm)
    m_lo = float(w.pos_mass[:, 3].min())
    m_hi = max(float(w.pos_mass[:, 3].max()), m_lo * (1 + 1e-6) + 1e-30)
    s = timed_calls(torch, stream, flush,
                    lambda: nb.render_points(pm, (1.0, 1.0, 1.0), m_lo, m_hi, ndc=ndc, rgba=rgba),
                    calls, warm)
    nb.sync()
    gbs = 48.0 * w.n / s / 1e9
    peak, src = measured_hbm_gbs()
    return {"workload": name, "mode": "render", "n": w.n, "calls": calls,
            "us_per_call": 1e6 * s, "value": gbs, "unit": "GB/s", "kernel": "render_points",
            "frac_of_hbm": gbs / peak, "peak_basis": src}


def measure_neighbors(nb, torch, stream, flush, sms: int, f_max: float) -> dict:
    """The 2-D cutoff neighbour list: N^2 ordered pair tests per call."""
    import workloads
    name, calls, warm = NEIGHBOR_CONFIG
    p = workloads.by_name(name)
    x = torch.from_numpy(p.x).cuda()
    y = torch.from_numpy(p.y).cuda()
    nn = torch.empty(p.n, dtype=torch.int32, device="cuda")
    nl = torch.empty((p.max_neighbors, p.n), dtype=torch.int32, device="cuda")
    s = timed_calls(torch, stream, flush,
                    lambda: nb.neighbors_2d(x, y, p.cutoff, p.max_neighbors, nn=nn, nl=nl),
                    calls, warm)
    nb.sync()
    value = float(p.n) * float(p.n) / s / 1e9
    peak = sms * f_max * 1e6 * FP32_LANES_PER_SM / NEIGHBOR_FP32_OPS / 1e9
    return {"workload": name, "mode": "neighbors", "n": p.n, "calls": calls,
            "us_per_call": 1e6 * s, "value": value, "unit": "Gpairs/s", "kernel": "neighbors_2d",
            "frac_of_own_roofline": value / peak}


def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__
    import workloads

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, True)
    __graft_entry__.build()
    import all_pairs_body_gb300 as nb
    if args.tuning or args.phases:
        from all_pairs_body_gb300 import build as nbuild
        nb._lib = nb.load(nbuild.build(tuning=args.tuning, phases=args.phases))

    w = workloads.by_name(args.workload)
    n = w.n
    dt = w.dt
    layout = {"rows4": 0, "rows3": 1, "blocks3": 2}[args.layout]
    if layout and args.mode not in ("step", "accel"):
        raise SystemExit("--layout applies to --mode step and accel")
    pm = torch.from_numpy(w.pos_mass).cuda()
    vel = torch.from_numpy(w.vel).cuda()
    acc = torch.empty_like(pm)
    if layout:
        vel = vel[:, :3].contiguous() if layout == 1 else vel[:, :3].t().contiguous()
        acc = torch.empty_like(vel)
    stream = torch.cuda.current_stream()

    ndc = torch.empty_like(pm) if args.mode == "render" else None
    rgba = torch.empty_like(pm) if args.mode == "render" else None
    m_lo = float(w.pos_mass[:, 3].min())
    m_hi = max(float(w.pos_mass[:, 3].max()), m_lo * (1 + 1e-6) + 1e-30)

    path = {"auto": nb.PATH_AUTO, "tiled": nb.PATH_TILED, "split": nb.PATH_SPLIT,
            "warp": nb.PATH_WARP, "pairs": nb.PATH_PAIRS}[args.path]
    if (path or args.split) and (layout or args.mode == "render"):
        raise SystemExit("--path/--split apply to --mode step|accel|kdk with rows4")

    def run_once(p_, v_, a_):
        """One timed unit of work on the given device tensors."""
        if args.mode == "render":
            nb.render_points(p_, (1.0, 1.0, 1.0), m_lo, m_hi, ndc=ndc, rgba=rgba)
        elif layout and args.mode == "step":
            nb.leapfrog_step_layout(p_, v_, a_, w.eps2, dt, 1, layout)
        elif layout:
            nb.accel_layout(p_, a_, w.eps2, layout)
        elif args.mode == "step":
            nb.leapfrog_step(p_, v_, a_, w.eps2, dt, 1, path=path, split=args.split)
        elif args.mode == "kdk":
            nb.leapfrog_kdk(p_, v_, a_, w.eps2, dt, 1, path=path, split=args.split)
        else:
            nb.accel(p_, w.eps2, out=a_, path=path, split=args.split)

    def step():
        run_once(pm, vel, acc)

    for _ in range(max(args.warmup, 0)):
        step()
    nb.sync()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    plan = nb.plan(n, path, args.split)

    sampler = ClockSampler(gpu_selector(local)).start()
    nb.profile_read()  # starts a new count of kernel launches
    if args.phases:
        nb.phase_read()  # starts a new count of phase cycles
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    clocks = sampler.stop()
    nb.sync()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    _, _, launches = nb.profile_read()
    total_s = reduce_max(sum(step_ms) / 1e3, dist, device="cuda")
    # the force kernels alone, in a second run of the same steps with the
    # library's events around each force launch (kept out of the timed run:
    # recording them costs host time per launch)
    nb.profile_enable(True)
    nb.profile_read()
    for k in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    nb.sync()
    force_ms, force_launches, _ = nb.profile_read()
    nb.profile_enable(False)
    phases = None
    if args.phases:
        cyc = nb.phase_read()
        total_cyc = sum(cyc.values())
        phases = {"cycles": cyc,
                  "share": {k: (v / total_cyc if total_cyc else None) for k, v in cyc.items()},
                  "what": "SM cycles of the pair kernel's warps per phase of a tile, summed over "
                          "the timed and the profiled steps (clock64 stamps, profiling build)"}
    if args.mode == "render":
        if rank == 0:
            print(json.dumps(render_line(args, w, world, total_s, launches, clocks)), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    interactions = float(n) * float(n) * (2.0 if args.mode == "kdk" else 1.0)
    value = aggregate_value(interactions * args.steps, world, total_s)
    if args.mode == "kdk":
        force_launches = max(force_launches, 1)
        interactions_per_pass = float(n) * float(n)
    else:
        interactions_per_pass = interactions

    # end to end through the same API with pinned host buffers
    e2e = None
    if not args.no_e2e and not layout:
        h_pm = torch.from_numpy(w.pos_mass).pin_memory()
        h_v = torch.from_numpy(w.vel).pin_memory()
        o_pm = torch.empty_like(h_pm).pin_memory()
        o_v = torch.empty_like(h_v).pin_memory()
        o_a = torch.empty_like(h_pm).pin_memory()
        d_pm = torch.empty_like(pm)
        d_v = torch.empty_like(vel)
        d_a = torch.empty_like(acc)
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        e_start.record(stream)
        for _ in range(args.steps):
            d_pm.copy_(h_pm, non_blocking=True)
            d_v.copy_(h_v, non_blocking=True)
            run_once(d_pm, d_v, d_a)
            o_pm.copy_(d_pm, non_blocking=True)
            o_v.copy_(d_v, non_blocking=True)
            o_a.copy_(d_a, non_blocking=True)
        e_end.record(stream)
        torch.cuda.synchronize()
        nb.sync()
        e2e_s = reduce_max(e_start.elapsed_time(e_end) / 1e3, dist, device="cuda")
        assert np.all(np.isfinite(o_a.numpy()))
        e2e = {"value": aggregate_value(interactions * args.steps, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": 2 * 16 * n, "d2h_bytes_per_step": 3 * 16 * n,
               "ms_per_step": 1e3 * e2e_s / args.steps}

    # roofline of the force kernel
    sms = plan["sms"]
    f_max, f_src = measured_sm_max_mhz(clocks)
    # a pair pass in chunks launches the force kernel once per chunk
    chunks = plan["chunks"]
    passes = force_launches / chunks if force_launches else 0
    achieved = (interactions_per_pass / (force_ms / 1e3 / passes) / 1e9
                if force_launches else None)
    kernel = {nb.PATH_WARP: "force_warp", nb.PATH_PAIRS: "force_pairs"}.get(plan["path"],
                                                                         "force_tiled")
    ops = FP32_OPS_PER_INTERACTION_PAIRS if kernel == "force_pairs" else FP32_OPS_PER_INTERACTION
    peak = alu_peak_ginter(sms, f_max, ops)
    roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": UNIT,
            "frac": (achieved / peak) if achieved else None,
            "traffic": profiled_traffic(n, kernel),
            "peak_basis": f"{sms} SMs x {f_max:g} MHz ({f_src}) x {FP32_LANES_PER_SM} FP32 lanes"
                          f" / {ops} FP32 ops per interaction",
            "kernel": kernel,
            "force_ms_per_launch": force_ms / force_launches if force_launches else None,
            "force_ms_per_pass": force_ms / passes if force_launches else None,
            "force_launches_per_pass": chunks}
    if kernel == "force_pairs" and achieved:
        # the same launch against the one-sided form's 12 ops per interaction
        roof["frac_of_one_sided_roofline"] = achieved / alu_peak_ginter(sms, f_max)
    if clocks and achieved:
        pc = alu_peak_ginter(sms, clocks["sm_mhz"], ops)
        roof["peak_at_measured_clock"] = pc
        roof["frac_at_measured_clock"] = achieved / pc

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, k, cores, wall, idx, ref = oracle_sample_rate(w.pos_mass, w.eps2, args.cpu_seconds,
                                                            12345)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{k} seeded target bodies x all {n} sources, FP64, one acceleration "
                         f"evaluation ({wall:.1f} s)"}
    if cpu is not None and not layout:
        # the same bodies once more through the timed path (untimed here), at the
        # oracle's sample; a failure is reported in the line, never raised
        try:
            a_gpu = nb.accel(torch.from_numpy(w.pos_mass).cuda(), w.eps2, path=path,
                             split=args.split)
            nb.sync()
            worst, rms = parity_errors(a_gpu.cpu().numpy()[idx], ref)
            parity = {"max_rel_err": worst, "rms_rel_err": rms, "tolerance": ACC_TOL,
                      "pass": worst <= ACC_TOL, "against": "FP64 oracle",
                      "sample": f"the cpu_baseline's {k} target bodies, accelerations at the "
                                f"initial positions"}
        except Exception as exc:  # noqa: BLE001
            parity = {"error": f"{type(exc).__name__}: {exc}"}

    configs = None
    if (rank == 0 and world == 1 and not args.no_configs and args.workload == DEFAULT_WORKLOAD
            and args.mode == "step" and path == nb.PATH_AUTO and not layout and not args.split
            and not (args.tuning or args.phases)):
        configs = {"what": "the other benchmark configurations, the one-sided kernel and the "
                           "kick-drift-kick step at 2^20, the point-shader kernel at 2^24 and "
                           "the 2-D neighbour list at 2^20, measured after the timed steps in "
                           "this process: device time per call between CUDA events (L2 flushed "
                           "before each call), the force kernel alone from a second, profiled "
                           "run; R = the one-sided 12-op FP32 roofline at sm_max_mhz"}
        try:
            configs["results"] = measure_configs(nb, torch, stream, flush, sms, f_max)
        except Exception as exc:  # noqa: BLE001 - reported in the line, never fatal
            configs["error"] = f"{type(exc).__name__}: {exc}"

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(w, args.mode, world),
        "gflops_20": value * FLOP_PER_INTERACTION, "roofline": roof, "cpu_baseline": cpu,
        "e2e": e2e, "gpu_launches": launches, "clocks": clocks, "parity": parity,
        "plan": plan, "layout": args.layout, "path": args.path, "impl": "ours",
        "library": "tuning" if args.tuning else ("phase clocks" if args.phases else "release"),
    }
    if configs is not None:
        line["configs"] = configs
    if phases is not None:
        line["phases"] = phases
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def measured_hbm_gbs() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "MEASURED_PEAKS.json hbm_gbs"
    except (OSError, KeyError, ValueError, TypeError):
        return 6800.0, "fallback HBM copy bandwidth"


def render_line(args, w, world, total_s, launches, clocks) -> dict:
    """JSON line of the memory-bound point-shader kernel: 16 bytes read and
    32 bytes written per body (the algorithmic traffic)."""
    nbytes = 48.0 * w.n * args.steps
    gbs = world * nbytes / total_s / 1e9
    peak, src = measured_hbm_gbs()
    return {
        "metric": "point-shader kernel throughput (NDC + mass colour)", "value": gbs,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, "render", world),
        "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peak, "unit": "GB/s",
                     "frac": gbs / world / peak, "traffic": None, "peak_basis": src},
        "gpu_launches": launches, "clocks": clocks, "impl": "ours",
    }


# ---------------------------------------------------------------------------
# reference arm: the FP64 CPU oracle on the host cores
# ---------------------------------------------------------------------------


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    import workloads

    w = workloads.by_name(args.workload)
    n = w.n
    # size one step so warm-up + timed steps end within a few minutes
    per_step_s = min(8.0, 150.0 / max(1, args.steps + args.warmup))
    rng = np.random.default_rng(777)
    probe = np.sort(rng.choice(n, size=min(16 * oracle.threads(), n), replace=False))
    t0 = time.perf_counter()
    oracle.accel(w.pos_mass, w.eps2, idx=probe)
    per_target = (time.perf_counter() - t0) / len(probe)
    k = int(max(16, min(n, per_step_s / max(per_target, 1e-9))))
    samples = [np.sort(rng.choice(n, size=k, replace=False)) for _ in range(args.steps + args.warmup)]
    for s in samples[:args.warmup]:
        oracle.accel(w.pos_mass, w.eps2, idx=s)
    t0 = time.perf_counter()
    for s in samples[args.warmup:]:
        oracle.accel(w.pos_mass, w.eps2, idx=s)
    wall = time.perf_counter() - t0
    value = k * n * args.steps / wall / 1e9
    sample = (f"each step: {k} seeded target bodies x all {n} sources, FP64 oracle, one "
              f"acceleration evaluation")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wall / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.mode, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


NEIGHBOR_FP32_OPS = 5  # per pair test: 2 subtracts, 2 squares, 1 add


def run_neighbors(args):
    """Pair tests per second of the 2-D cutoff neighbour list on one GPU."""
    import torch

    import __graft_entry__
    import workloads

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, True)
    __graft_entry__.build()
    import all_pairs_body_gb300 as nb

    name = args.workload if args.workload.startswith("points2d-") else "points2d-1048576"
    p = workloads.by_name(name)
    x = torch.from_numpy(p.x).cuda()
    y = torch.from_numpy(p.y).cuda()
    nn = torch.empty(p.n, dtype=torch.int32, device="cuda")
    nl = torch.empty((p.max_neighbors, p.n), dtype=torch.int32, device="cuda")
    for _ in range(max(args.warmup, 0)):
        nb.neighbors_2d(x, y, p.cutoff, p.max_neighbors, nn=nn, nl=nl)
    nb.sync()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(gpu_selector(local)).start()
    nb.profile_read()  # starts a new count of kernel launches
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()
        starts[k].record(stream)
        nb.neighbors_2d(x, y, p.cutoff, p.max_neighbors, nn=nn, nl=nl)
        ends[k].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    clocks = sampler.stop()
    nb.sync()
    _, _, launches = nb.profile_read()
    total_s = reduce_max(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3, dist,
                         device="cuda")
    tests = float(p.n) * float(p.n)
    value = aggregate_value(tests * args.steps, world, total_s)
    sms = nb.plan(p.n)["sms"]
    f_max, f_src = measured_sm_max_mhz(clocks)
    peak = sms * f_max * 1e6 * FP32_LANES_PER_SM / NEIGHBOR_FP32_OPS / 1e9
    line = {
        "metric": "2-D cutoff neighbour list: pair tests/s (billions)", "value": value,
        "unit": "Gpairs/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{p.name}: N={p.n} uniform 2-D points, 0.4 per unit area, "
                               f"cutoff {p.cutoff}, {p.max_neighbors} list slots; each step "
                               "tests all N^2 ordered pairs",
                   "n_points": p.n, "l2": "flushed between timed steps (512 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "alu", "achieved": value / world, "peak": peak, "unit": "Gpairs/s",
                     "frac": value / world / peak, "traffic": None,
                     "peak_basis": f"{sms} SMs x {f_max:g} MHz ({f_src}) x {FP32_LANES_PER_SM} "
                                   f"FP32 lanes / {NEIGHBOR_FP32_OPS} FP32 ops per pair test"},
        "mean_neighbors": float(nn.double().mean().item()), "gpu_launches": launches,
        "clocks": clocks, "impl": "ours",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "ours" and args.mode == "neighbors":
        run_neighbors(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
