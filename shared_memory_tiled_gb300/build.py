"""Builds ``libtranspose.so`` in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` compiles in parallel to an object file
under ``_build/``, then nvcc links the shared library (CUDA runtime linked
statically, no link against the driver library: the tensor-map encoder is
fetched through the runtime's driver entry-point query).

Run as ``python -m shared_memory_tiled_gb300.build`` or call ``build()``.
``build(debug=True)`` (``--debug``) makes the bounds-checked library instead,
compiled with ``TR_DEBUG`` into ``_build_debug/``: every global load and store
of every kernel is first checked against its side's logical elements and
refused (skipped and counted) when it falls outside them; the release library
is not touched.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libtranspose.so")
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_BUILD_DIR, "libtranspose.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-Xcompiler", "-fvisibility=hidden",  # only the header's tr_* entry points are exported
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
SOURCES = ["api.cu", "copy.cu", "tile_lsu.cu", "tile_vec.cu", "tile_vec_u32.cu",
           "tile_vec_u32_prefetch.cu", "tile_vec_u16.cu", "tile_vec_u16_prefetch.cu",
           "tile_tma.cu", "inplace.cu", "bank_probe.cu", "operand_tiles.cu", "bounds.cu"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtranspose")
    return path


def _inputs_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, extra: list[str], build_dir: str = BUILD_DIR) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Compile the library if any source is newer than it; return its path.
    With ``debug`` the bounds-checked library is built (``_build_debug/``)."""
    build_dir, lib_path = (DEBUG_BUILD_DIR, DEBUG_LIB_PATH) if debug else (BUILD_DIR, LIB_PATH)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _inputs_mtime():
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if debug:
        extra += ["-DTR_DEBUG=1"]
    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), max(2, os.cpu_count() or 2))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--ptxas-v" in sys.argv,
                debug="--debug" in sys.argv))
