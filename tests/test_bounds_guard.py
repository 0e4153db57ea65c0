"""The bounds-checked build's guard predicates (csrc/bounds.cuh) on the CPU.

The guards decide, before a kernel of the checked build touches global
memory, whether an access belongs to its side: every element a logical one
(`all_logical`), or every byte between the side's first and last logical
element (`in_extent`).  Here they are compiled for the host and compared with
a plain enumeration of the logical elements of small random sides -- batch
planes of rows x cols elements at row pitch ld and plane pitch stride -- on
accesses of every width at addresses in and around each side."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "shared_memory_tiled_gb300", "csrc")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not available")


@pytest.fixture(scope="module")
def guard(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("guard") / "libguard.so")
    subprocess.run(["nvcc", "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-o", out,
                    os.path.join(ROOT, "tests", "c", "bounds_guard.cu")], check=True)
    lib = ctypes.CDLL(out)
    argt = [ctypes.c_ulonglong] + [ctypes.c_longlong] * 5 + [ctypes.c_int, ctypes.c_ulonglong,
                                                            ctypes.c_int]
    for name in ("guard_all_logical", "guard_in_extent"):
        getattr(lib, name).argtypes = argt
        getattr(lib, name).restype = ctypes.c_int
    return lib


def _logical_bytes(base, batch, rows, cols, ld, stride, esize):
    """Set of byte addresses covered by the side's logical elements."""
    out = set()
    for b in range(batch):
        for i in range(rows):
            for j in range(cols):
                e = (b * stride if batch > 1 else 0) + i * ld + j
                out.update(range(base + e * esize, base + (e + 1) * esize))
    return out


def test_guards_against_enumeration(guard):
    rng = np.random.default_rng(7)
    base = 1 << 20
    for _ in range(400):
        esize = int(rng.choice([1, 2, 4]))
        batch = int(rng.integers(1, 4))
        rows, cols = int(rng.integers(1, 6)), int(rng.integers(1, 7))
        ld = cols + int(rng.integers(0, 4))
        stride = (rows - 1) * ld + cols + int(rng.integers(0, 5))
        side = (base, batch, rows, cols, ld, stride, esize)
        logical = _logical_bytes(*side)
        first, last = min(logical), max(logical)
        span = (batch - 1) * stride + rows * ld + 8
        for _ in range(60):
            bytes_ = int(rng.choice([esize, 2 * esize, 4, 8, 16]))
            addr = base + int(rng.integers(-3 * esize, span * esize + 8))
            want_logical = (addr - base) % esize == 0 and bytes_ % esize == 0 and \
                all(a in logical for a in range(addr, addr + bytes_))
            want_extent = first <= addr and addr + bytes_ - 1 <= last
            assert guard.guard_all_logical(*side, addr, bytes_) == want_logical, (side, addr, bytes_)
            assert guard.guard_in_extent(*side, addr, bytes_) == want_extent, (side, addr, bytes_)


def test_guards_on_hand_picked_accesses(guard):
    # 2 planes of 3 x 5 four-byte elements, row pitch 8, plane pitch 32 (the
    # device self-test's side): logical elements sit at plane*32 + row*8 + col
    side = (4096, 2, 3, 5, 8, 32, 4)
    at = lambda e: 4096 + 4 * e  # noqa: E731
    assert guard.guard_all_logical(*side, at(32 + 2 * 8 + 4), 4) == 1   # last element
    assert guard.guard_all_logical(*side, at(32 + 2 * 8 + 5), 4) == 0   # one past a row
    assert guard.guard_all_logical(*side, at(8), 16) == 1               # row 1, columns 0..3
    assert guard.guard_all_logical(*side, at(3), 16) == 0               # columns 3..6
    assert guard.guard_all_logical(*side, at(24), 4) == 0               # the gap between planes
    assert guard.guard_all_logical(*side, at(0) + 2, 4) == 0            # off an element boundary
    assert guard.guard_in_extent(*side, at(53) - 16, 16) == 1           # the extent's last bytes
    assert guard.guard_in_extent(*side, at(53) - 15, 16) == 0           # one byte past it
    assert guard.guard_in_extent(*side, at(0) - 1, 4) == 0              # before the first element
