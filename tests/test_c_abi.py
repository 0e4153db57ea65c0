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
