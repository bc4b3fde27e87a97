"""Plausible mistakes planted in copies of the oracle are each caught by a pin.

Every mutant is a text edit of ``oracle/nbody_oracle.c`` compiled on the CPU
into a temporary library; the pins of ``oracle_pins.py`` run against it and
at least one must fail.  This shows the pins constrain every part of the
oracle (sign, mass index, power, softening, loop bounds, component indices,
kick factor, step order, start-of-step accelerations, mass column, sampling).
"""
import os

import pytest

import oracle
from oracle import build as obuild
from oracle_pins import failing_pins

SRC = os.path.join(os.path.dirname(obuild.__file__), "nbody_oracle.c")

STEP_LOOPS = (
    "#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)\n"
    "        for (int64_t i = 0; i < n; ++i)\n"
    "            accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);\n"
    "#pragma omp parallel for schedule(static) num_threads(nt)\n"
    "        for (int64_t i = 0; i < n; ++i) {\n"
)
FUSED_IN_PLACE = (
    "        for (int64_t i = 0; i < n; ++i) {\n"
    "            accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);\n"
)
KICK_DRIFT = (
    "                vel[3 * i + c] = vel[3 * i + c] + 0.5 * dt * acc[3 * i + c];\n"
    "                pos_mass[4 * i + c] = pos_mass[4 * i + c] + dt * vel[3 * i + c];\n"
)
DRIFT_KICK = (
    "                pos_mass[4 * i + c] = pos_mass[4 * i + c] + dt * vel[3 * i + c];\n"
    "                vel[3 * i + c] = vel[3 * i + c] + 0.5 * dt * acc[3 * i + c];\n"
)

KDK_CLOSING = (
    "#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)\n"
    "        for (int64_t i = 0; i < n; ++i)\n"
    "            accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);\n"
    "#pragma omp parallel for schedule(static) num_threads(nt)\n"
    "        for (int64_t i = 0; i < n; ++i)\n"
    "            for (int c = 0; c < 3; ++c)\n"
    "                vel[3 * i + c] = vel[3 * i + c] + 0.5 * dt * acc[3 * i + c];\n"
    "    }\n"
)
KDK_CLOSING_STALE = (
    "#pragma omp parallel for schedule(static) num_threads(nt)\n"
    "        for (int64_t i = 0; i < n; ++i)\n"
    "            for (int c = 0; c < 3; ++c)\n"
    "                vel[3 * i + c] = vel[3 * i + c] + 0.5 * dt * acc[3 * i + c];\n"
    "#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)\n"
    "        for (int64_t i = 0; i < n; ++i)\n"
    "            accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);\n"
    "    }\n"
)
KDK_CLOSING_DROPPED = (
    "#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)\n"
    "        for (int64_t i = 0; i < n; ++i)\n"
    "            accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);\n"
    "    }\n"
)
KDK_FIRST_ACCEL = (
    "    if (steps == 0)\n"
    "        return nt;\n"
    "#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)\n"
    "    for (int64_t i = 0; i < n; ++i)\n"
    "        accel_of_body(pos_mass, n, eps2, i, acc + 3 * i);\n"
)

MUTANTS = {
    "neighbors_not_strict": [("if (distance_square < cutoff_square && n2 != n1)",
                              "if (distance_square <= cutoff_square && n2 != n1)")],
    "neighbors_self_included": [("if (distance_square < cutoff_square && n2 != n1)",
                                 "if (distance_square < cutoff_square)")],
    "neighbors_cutoff_not_squared": [("const float cutoff_square = cutoff * cutoff;",
                                      "const float cutoff_square = cutoff;")],
    "neighbors_row_major_list": [("nl[(int64_t)count * n_idx + k] = (int32_t)n2;",
                                  "nl[k * mn + count] = (int32_t)n2;")],
    "neighbors_empty_slots_not_cleared": [("            nl[(int64_t)q * n_idx + k] = -1;",
                                           "            (void)q;")],
    "neighbors_sample_index_ignored": [("const int64_t n1 = idx ? idx[k] : k;",
                                        "const int64_t n1 = k;")],
    "render_colours_swapped": [("const double green[3] = {0.0, 1.0, 0.0};",
                                "const double green[3] = {1.0, 0.0, 0.0};"),
                               ("const double red[3] = {1.0, 0.0, 0.0};",
                                "const double red[3] = {0.0, 1.0, 0.0};")],
    "render_weight_not_normalised": [("/ (max_w - min_w);", "/ max_w;")],
    "render_offset_dropped": [("/ (lim[c] - (-lim[c])) - 1.0;", "/ (lim[c] - (-lim[c]));")],
    "render_half_range": [("/ (lim[c] - (-lim[c])) - 1.0;", "/ lim[c] - 1.0;")],
    "kdk_closing_kick_dropped": [(KDK_CLOSING, KDK_CLOSING_DROPPED)],
    "kdk_closing_kick_with_old_accel": [(KDK_CLOSING, KDK_CLOSING_STALE)],
    "kdk_first_accel_skipped": [(KDK_FIRST_ACCEL, "    if (steps == 0)\n        return nt;\n")],
    "reversed_separation": [("pm[4 * j + 0] - xi", "xi - pm[4 * j + 0]"),
                            ("pm[4 * j + 1] - yi", "yi - pm[4 * j + 1]"),
                            ("pm[4 * j + 2] - zi", "zi - pm[4 * j + 2]")],
    "target_mass_not_source": [("pm[4 * j + 3] / (", "pm[4 * i + 3] / (")],
    "inverse_square_power": [("(d * sqrt(d))", "(d * d)")],
    "inverse_first_power": [("(d * sqrt(d))", "(sqrt(d))")],
    "softening_dropped": [("rz * rz + eps2;", "rz * rz;")],
    "softening_squared": [("rz * rz + eps2;", "rz * rz + eps2 * eps2;")],
    "softening_outside_power": [("const double w = pm[4 * j + 3] / (d * sqrt(d));",
                                 "const double w = pm[4 * j + 3] / ((d - eps2) * sqrt(d - eps2) + eps2);")],
    "last_source_dropped": [("for (int64_t j = 0; j < n; ++j)", "for (int64_t j = 0; j < n - 1; ++j)")],
    "first_source_dropped": [("for (int64_t j = 0; j < n; ++j)", "for (int64_t j = 1; j < n; ++j)")],
    "component_mixed_up": [("ay += w * ry;", "ay += w * rx;")],
    "accumulator_not_zeroed": [("double ax = 0.0, ay = 0.0, az = 0.0;",
                                "double ax = xi, ay = 0.0, az = 0.0;")],
    "full_kick": [("+ 0.5 * dt * acc[3 * i + c]", "+ dt * acc[3 * i + c]")],
    "half_drift": [("+ dt * vel[3 * i + c]", "+ 0.5 * dt * vel[3 * i + c]")],
    "drift_before_kick": [(KICK_DRIFT, DRIFT_KICK)],
    "in_place_update_race": [(STEP_LOOPS, FUSED_IN_PLACE)],
    # (stays in bounds: widening the drift loop to 4 columns would write past vel)
    "mass_drifted": [("for (int c = 0; c < 3; ++c) {\n                vel[3 * i + c]",
                      "pos_mass[4 * i + 3] = pos_mass[4 * i + 3] + dt * vel[3 * i];\n"
                      "            for (int c = 0; c < 3; ++c) {\n                vel[3 * i + c]")],
    "sample_index_ignored": [("const int64_t i = idx ? idx[k] : k;", "const int64_t i = k;")],
    "sampled_step_full_kick": [("vel[3 * i + c] + 0.5 * dt * acc_out[3 * k + c];",
                                "vel[3 * i + c] + dt * acc_out[3 * k + c];")],
    "sampled_step_drift_with_old_velocity": [
        ("pos_mass[4 * i + c] + dt * vel_out[3 * k + c];",
         "pos_mass[4 * i + c] + dt * vel[3 * i + c];")],
    "sampled_step_mass_not_copied": [("pos_out[4 * k + 3] = pos_mass[4 * i + 3];",
                                      "pos_out[4 * k + 3] = 0.0;")],
    "sampled_step_row_not_indexed": [("        const int64_t i = idx[k];\n        for (int c = 0; c < 3; ++c) {\n            vel_out",
                                      "        const int64_t i = k;\n        for (int c = 0; c < 3; ++c) {\n            vel_out")],
}


def _mutant_lib(name, edits, tmp_path):
    with open(SRC) as f:
        text = f.read()
    for old, new in edits:
        assert old in text, f"mutant {name}: pattern not found: {old!r}"
        text = text.replace(old, new)
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    return obuild.compile_c([str(src)], str(tmp_path / f"lib{name}.so"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    lib = _mutant_lib(name, MUTANTS[name], tmp_path)
    failed = failing_pins(oracle.Oracle(lib))
    assert failed, f"mutant {name} passes every pin"


def test_unmutated_copy_passes(tmp_path):
    lib = _mutant_lib("identity", [], tmp_path)
    assert failing_pins(oracle.Oracle(lib)) == []
