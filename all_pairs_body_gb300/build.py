"""Build the CUDA library in-tree: all_pairs_body_gb300/libnbody_gb300.so.

One translation unit, one -gencode (sm_103a), compiled with nvcc directly
(no cmake, no torch extension machinery), so it builds in well under a
minute on x86-64 and on the aarch64 GPU hosts alike.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libnbody_gb300.so")
# The index-checked build (NBODY_BOUNDS_CHECK): every computed index into a
# scratch or output array is tested on the device; for tests, not for use.
LIB_CHECKED = os.path.join(HERE, "libnbody_gb300_checked.so")
# The tuning build (NBODY_TUNING_TABLE): the release library plus every other
# kernel shape and scheme measured while choosing the release rows, reachable
# through NBODY_TILED_CONFIG / NBODY_PAIRS_CONFIG; for tests and sweeps.
LIB_TUNING = os.path.join(HERE, "libnbody_gb300_tuning.so")
# The profiling build (NBODY_PHASE_CLOCKS): the release library with clock64
# stamps around the phases of the pair kernel's tiles (nbody_phase_read).
LIB_PHASES = os.path.join(HERE, "libnbody_gb300_phases.so")
# The FP32-pipe calibration program (a standalone binary, not part of the
# library): python -m all_pairs_body_gb300.build --probe builds and runs it.
PROBE = os.path.join(HERE, "fp32_pipe_probe")
SOURCES = ["nbody_api.cu"]
DEPS = SOURCES + ["nbody_kernels.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-ftz=true", "-Xcompiler", "-fPIC",
              "-shared", "-Xcompiler", "-Wall"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          checked: bool = False, tuning: bool = False, phases: bool = False) -> str:
    if checked + tuning + phases > 1:
        raise ValueError("the checked, tuning and phase-clock builds are separate libraries")
    out = LIB_CHECKED if checked else (LIB_TUNING if tuning else (LIB_PHASES if phases else LIB))
    deps = [os.path.join(CSRC, s) for s in DEPS] + [os.path.join(INCLUDE, "nbody.h")]
    if not force and os.path.exists(out):
        t = os.path.getmtime(out)
        if all(os.path.getmtime(d) <= t for d in deps):
            return out
    tmp = out + f".tmp{os.getpid()}"
    flags = (["-DNBODY_BOUNDS_CHECK"] if checked else
             ["-DNBODY_TUNING_TABLE"] if tuning else ["-DNBODY_PHASE_CLOCKS"] if phases else [])
    cmd = ([nvcc()] + ARCH + NVCC_FLAGS + flags + ["-I", INCLUDE, "-I", CSRC] + list(extra or [])
           + ["-o", tmp] + [os.path.join(CSRC, s) for s in SOURCES] + ["-lcudart"])
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build_probe(force: bool = False) -> str:
    """Compile the FP32-pipe calibration program (fp32_pipe_probe.cu)."""
    src = os.path.join(CSRC, "fp32_pipe_probe.cu")
    deps = [src, os.path.join(CSRC, "nbody_kernels.cuh"), os.path.join(INCLUDE, "nbody.h")]
    if not force and os.path.exists(PROBE):
        t = os.path.getmtime(PROBE)
        if all(os.path.getmtime(d) <= t for d in deps):
            return PROBE
    tmp = PROBE + f".tmp{os.getpid()}"
    cmd = ([nvcc()] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-ftz=true", "-I", INCLUDE,
                              "-I", CSRC, "-o", tmp, src])
    subprocess.run(cmd, check=True)
    os.replace(tmp, PROBE)
    return PROBE


if __name__ == "__main__":
    if "--probe" in sys.argv:
        sys.exit(subprocess.run([build_probe()]).returncode)
    extra = ["-Xptxas", "-v"] if "-v" in sys.argv else None
    print(build(force=True, verbose=True, extra=extra))
