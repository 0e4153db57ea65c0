"""CPU oracle for the out-of-place transpose -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and nothing
here imports the product package: the two share no code.

The arithmetic lives in ``oracle.c`` (a plain double loop over raw bit
patterns, see the header of that file for the passages it follows).  This
module only compiles it with gcc and marshals numpy arrays into it.

Definition (all sizes in elements), for b < batch, i < rows, j < cols::

    out[b*stride_out + j*ld_out + i] = in[b*stride_in + i*ld_in + j]

Parity status: pinned by ``tests/test_oracle.py`` (hand-written golden
fixtures, closed forms for index-valued inputs, numpy's transpose on dense
cases, involution, permutation and sentinel invariants, brute force on tiny
shapes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

_I64 = ctypes.c_int64
_ARGS_T = [ctypes.c_void_p, ctypes.c_void_p, _I64, _I64, _I64, _I64, _I64, _I64, _I64]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` with gcc and return its path."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-Wextra",
                    "-o", tmp, _SRC], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name in ("oracle_transpose_u32", "oracle_transpose_u16",
                         "oracle_transpose_scatter_u32", "oracle_transpose_scatter_u16"):
                fn = getattr(lib, name)
                fn.argtypes = _ARGS_T
                fn.restype = None
            lib.oracle_copy_bytes.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _I64]
            lib.oracle_copy_bytes.restype = None
            lib.oracle_operand_tiles_u32.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _I64, _I64,
                                                     _I64, _I64, _I64]
            lib.oracle_operand_tiles_u32.restype = None
            for name in ("oracle_transpose_inplace_u32", "oracle_transpose_inplace_u16"):
                fn = getattr(lib, name)
                fn.argtypes = [ctypes.c_void_p, _I64, _I64, _I64, _I64]
                fn.restype = None
            _lib = lib
    return _lib


def _extent(batch, rows, cols, ld, stride):
    """Number of elements from the first to one past the last logical element."""
    if batch == 0 or rows == 0 or cols == 0:
        return 0
    return (batch - 1) * stride + (rows - 1) * ld + cols


def transpose(x: np.ndarray, out: np.ndarray, *, batch: int = 1, rows: int, cols: int,
              ld_in: int | None = None, ld_out: int | None = None,
              stride_in: int | None = None, stride_out: int | None = None,
              form: str = "gather") -> np.ndarray:
    """Write the transpose of the logical region of ``x`` into ``out`` in place.

    ``x`` and ``out`` are flat, C-contiguous numpy arrays of ``uint32`` (fp32
    bit patterns) or ``uint16`` (bf16 bit patterns).  ``rows``/``cols``
    describe the input; the output is ``cols`` x ``rows`` per batch plane.
    Only the logical output elements are written; everything else in ``out``
    keeps its previous contents.  ``form`` picks the gather (output-order) or
    scatter (input-order) loop.
    """
    ld_in = cols if ld_in is None else ld_in
    ld_out = rows if ld_out is None else ld_out
    stride_in = rows * ld_in if stride_in is None else stride_in
    stride_out = cols * ld_out if stride_out is None else stride_out
    if x.dtype != out.dtype or x.dtype not in (np.uint32, np.uint16):
        raise TypeError("oracle works on uint32 or uint16 bit patterns")
    if not (x.flags.c_contiguous and out.flags.c_contiguous and x.ndim == 1 and out.ndim == 1):
        raise ValueError("oracle wants flat C-contiguous arrays")
    if min(batch, rows, cols) < 0 or ld_in < cols or ld_out < rows:
        raise ValueError("bad sizes")
    if x.size < _extent(batch, rows, cols, ld_in, stride_in) or \
            out.size < _extent(batch, cols, rows, ld_out, stride_out):
        raise ValueError("buffer smaller than its logical extent")
    lib = _load()
    suffix = "u32" if x.dtype == np.uint32 else "u16"
    name = {"gather": "oracle_transpose_", "scatter": "oracle_transpose_scatter_"}[form] + suffix
    getattr(lib, name)(x.ctypes.data, out.ctypes.data, batch, rows, cols,
                       ld_in, ld_out, stride_in, stride_out)
    return out


def copy_bytes(x: np.ndarray, out: np.ndarray) -> np.ndarray:
    """Byte-for-byte copy of ``x`` into ``out`` (same byte length)."""
    if x.nbytes != out.nbytes:
        raise ValueError("size mismatch")
    _load().oracle_copy_bytes(x.ctypes.data, out.ctypes.data, x.nbytes)
    return out


def transpose_inplace(data: np.ndarray, *, batch: int = 1, n: int, ld: int | None = None,
                      stride: int | None = None) -> np.ndarray:
    """Transpose each n x n plane of ``data`` in place (element (i, j) swaps with
    (j, i)); padding between ``n`` and ``ld`` and between planes is untouched."""
    ld = n if ld is None else ld
    stride = n * ld if stride is None else stride
    if data.dtype not in (np.uint32, np.uint16) or data.ndim != 1 or not data.flags.c_contiguous:
        raise TypeError("oracle works on flat uint32 or uint16 bit patterns")
    if min(batch, n) < 0 or ld < n or (batch > 1 and stride < (n - 1) * ld + n):
        raise ValueError("bad sizes")
    if data.size < _extent(batch, n, n, ld, stride):
        raise ValueError("buffer smaller than its logical extent")
    lib = _load()
    name = "oracle_transpose_inplace_" + ("u32" if data.dtype == np.uint32 else "u16")
    getattr(lib, name)(data.ctypes.data, batch, n, ld, stride)
    return data


def operand_tiles(a: np.ndarray, out: np.ndarray, *, m: int, k: int, lda: int, bm: int,
                  bk: int) -> np.ndarray:
    """Blocked transposed operand tiles of a row-major M x K matrix (fp32 bits):
    tile (mt, kt) of ``out`` holds As[k][m] = A[mt*bm + m][kt*bk + k], unpadded,
    tiles in (mt, kt) row-major order.  M and K must be multiples of bm, bk."""
    if a.dtype != np.uint32 or out.dtype != np.uint32:
        raise TypeError("operand tiles are fp32 bit patterns (uint32)")
    if m % bm or k % bk or lda < k or min(m, k, bm, bk) <= 0:
        raise ValueError("bad sizes")
    if a.size < (m - 1) * lda + k or out.size < m * k:
        raise ValueError("buffer smaller than its extent")
    _load().oracle_operand_tiles_u32(a.ctypes.data, out.ctypes.data, m, k, lda, bm, bk)
    return out
