"""A C program as the library's client: `tests/c_client/two_bodies.c`.

It includes only `include/nbody.h` and the CUDA runtime, passes plain device
pointers, and checks two bodies against the closed form of the softened law
and one leapfrog step from rest against the half-kick-then-drift update.  On
the CPU the program must compile and link against the built library; on the
GPU it must run and exit 0.
"""
import os
import shutil
import subprocess

import pytest

from all_pairs_body_gb300 import build as nbuild

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c_client", "two_bodies.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_client(out_dir):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("CUDA headers not found")
    lib = nbuild.build()
    lib_dir = os.path.dirname(lib)
    exe = os.path.join(str(out_dir), "two_bodies")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", nbuild.INCLUDE,
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe, "-L", lib_dir, "-lnbody_gb300",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm", f"-Wl,-rpath,{lib_dir}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_client_compiles_and_links(tmp_path):
    exe = compile_client(tmp_path)
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_c_client_runs(tmp_path):
    exe = compile_client(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "two_bodies: ok" in r.stdout
