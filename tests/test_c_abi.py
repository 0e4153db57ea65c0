"""The boundary from plain C: `include/transpose.h` compiles as strict C99 and a
C program links against libtranspose and gets host-side answers (no GPU)."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from shared_memory_tiled_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")


def test_c_program_uses_the_abi(tmp_path):
    build_mod.build()
    lib_dir = os.path.dirname(build_mod.LIB_PATH)
    exe = str(tmp_path / "abi_host")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_host.c"),
           "-L", lib_dir, "-ltranspose", f"-Wl,-rpath,{lib_dir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


@pytest.mark.gpu
def test_c_program_on_the_gpu(tmp_path):
    """A C program allocates device memory with the CUDA runtime, transposes
    through the C entry points and compares every byte with the oracle's C
    routines (liboracle), output padding included."""
    import oracle
    build_mod.build()
    oracle_lib = oracle.build()
    lib_dir = os.path.dirname(build_mod.LIB_PATH)
    oracle_dir = os.path.dirname(oracle_lib)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cuda_lib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                     if os.path.exists(os.path.join(d, "libcudart.so"))), None)
    if cuda_lib is None:
        pytest.skip("libcudart.so not found")
    exe = str(tmp_path / "abi_gpu")
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c", "abi_gpu.c"),
           "-L", lib_dir, "-ltranspose", "-L", oracle_dir, "-loracle", "-L", cuda_lib, "-lcudart",
           f"-Wl,-rpath,{lib_dir}:{oracle_dir}:{cuda_lib}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
