"""Compile the FP64 CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc with OpenMP; -ffp-contract=off keeps every multiply and add
separately rounded so the oracle gives the same bits on x86-64 and aarch64.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ["nbody_oracle.c"]
LIB = os.path.join(HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
          "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra"]


def compile_c(sources: list[str], out: str, verbose: bool = False) -> str:
    """gcc ``sources`` into the shared library ``out`` (atomic replace)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc"] + CFLAGS + ["-o", tmp] + list(sources) + ["-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False, verbose: bool = False) -> str:
    srcs = [os.path.join(HERE, s) for s in SOURCES]
    if not force and os.path.exists(LIB):
        lib_t = os.path.getmtime(LIB)
        if all(os.path.getmtime(s) <= lib_t for s in srcs):
            return LIB
    return compile_c(srcs, LIB, verbose)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
