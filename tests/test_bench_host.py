"""Host-side logic of bench.py: conventions, clocks parsing, roofline arithmetic,
the rank reduction (world size 2 over gloo on CPU) and the reference arm."""
import io
import json
import os
import socket
import subprocess
import sys
import contextlib

import pytest

import bench

HERE = os.path.dirname(os.path.abspath(__file__))


def test_flop_convention_matches_the_page():
    rows = [l.split() for l in open(os.path.join(HERE, "golden", "flop_convention.txt"))
            if l.strip() and not l.startswith("#")]
    total = int(rows[-1][-1])
    assert sum(int(r[-1]) for r in rows[:-1]) == total
    assert bench.FLOP_PER_INTERACTION == total == 20


def test_alu_peak_arithmetic():
    # 152 SMs x 2070 MHz x 128 lanes / 12 ops
    assert bench.alu_peak_ginter(152, 2070.0) == pytest.approx(152 * 2.07 * 128 / 12)
    assert bench.alu_peak_ginter(160, 1000.0) == pytest.approx(160 * 128 / 12)


def test_aggregate_value():
    assert bench.aggregate_value(2.0e12, 1, 1.0) == pytest.approx(2000.0)
    assert bench.aggregate_value(2.0e12, 4, 2.0) == pytest.approx(4000.0)


def test_parse_clock_lines():
    lines = [
        "0, 1965, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1800, 2070, 1380.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1700, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage",
    ]
    c = bench.parse_clock_lines(lines)
    assert c["sm_mhz"] == 1800 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert bench.parse_clock_lines(["x"]) is None


def test_gpu_selector(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.gpu_selector(1) == "5"
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.gpu_selector(2) == "2"


def test_traffic_needs_matching_kernel(tmp_path, monkeypatch):
    summary = tmp_path / "s.md"
    summary.write_text("- kernel_source_sha256_16: `deadbeef`\n- dram_bytes_per_launch: 1000\n"
                       "- n_captured: 10\n")
    monkeypatch.setitem(bench.PROFILE_SUMMARIES, "force_tiled", str(summary))
    assert bench.profiled_traffic(20) is None
    summary.write_text(f"- kernel_source_sha256_16: `{bench.kernel_source_digest()}`\n"
                       "- dram_bytes_per_launch: 1000\n- n_captured: 10\n")
    assert bench.profiled_traffic(20) == pytest.approx(2000.0)
    # reaction sums of the pair kernel grow with n^2
    summary.write_text(f"- kernel_source_sha256_16: `{bench.kernel_source_digest()}`\n"
                       "- dram_bytes_per_launch: 1000\n- n_captured: 10\n"
                       "- traffic_scales_as: n^2\n")
    monkeypatch.setitem(bench.PROFILE_SUMMARIES, "force_pairs", str(summary))
    assert bench.profiled_traffic(20, "force_pairs") == pytest.approx(4000.0)
    assert bench.profiled_traffic(20, "force_warp") is None


def test_other_configs_name_known_workloads():
    """Every row of the default run's configs block names a workload the
    generators know, in a mode the binding has, so the default run cannot
    stop on a name after its timed steps."""
    import workloads
    for name, mode, path, calls, warm, steps in bench.OTHER_CONFIGS:
        assert mode in ("accel", "step", "kdk") and path in ("auto", "split")
        assert calls >= 1 and warm >= 1 and steps >= 1
        assert workloads.by_name(name).n == int(name.rsplit("-", 1)[1])
    for name in (bench.RENDER_CONFIG[0], bench.NEIGHBOR_CONFIG[0]):
        assert name.rsplit("-", 1)[0] in ("ball-lognormal", "points2d")
    assert workloads.by_name(bench.NEIGHBOR_CONFIG[0]).n == 1048576


def test_pair_roofline_counts_eight_ops():
    one_sided = bench.alu_peak_ginter(152, 2070.0)
    assert one_sided == pytest.approx(152 * 2070e6 * 128 / 12 / 1e9)
    assert bench.alu_peak_ginter(152, 2070.0, bench.FP32_OPS_PER_INTERACTION_PAIRS) == \
        pytest.approx(1.5 * one_sided)


def test_reference_arm_prints_contract_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "cube-sweep-1000", "--steps", "2",
                    "--warmup", "1"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
rank, local, world = bench.dist_env()
dist = bench.init_dist(world, False)
t = bench.reduce_max(1.0 + rank, dist)
bench.barrier(dist)
v = bench.aggregate_value(1e9, world, t)
print(json.dumps({{"rank": rank, "t": t, "v": v}}))
dist.destroy_process_group()
"""


def test_two_rank_reduction_over_gloo(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(WORKER.format(root=os.path.dirname(HERE)))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    assert all(r["t"] == 2.0 for r in res)  # max over ranks
    assert all(r["v"] == pytest.approx(2 * 1e9 / 2.0 / 1e9) for r in res)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "cube-sweep-1000"])
    assert buf.getvalue() == ""


def test_parity_errors_definition():
    """max and RMS of |a_got,i - a_ref,i| over RMS_i |a_ref,i|, 3-vectors only."""
    import numpy as np
    ref = np.array([[3.0, 4.0, 0.0], [0.0, 0.0, 5.0]])  # |a| = 5 each: RMS 5
    got = np.array([[3.0, 4.0, 0.5, 9.0], [0.0, 0.0, 5.0, -9.0]])  # w ignored
    worst, rms = bench.parity_errors(got, ref)
    assert worst == pytest.approx(0.5 / 5.0)
    assert rms == pytest.approx(np.sqrt((0.25 + 0.0) / 2) / 5.0)
    assert bench.parity_errors(ref, ref) == (0.0, 0.0)
    assert bench.ACC_TOL == 1e-4
