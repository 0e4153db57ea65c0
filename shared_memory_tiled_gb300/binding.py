"""ctypes binding of libtranspose's C ABI (``include/transpose.h``).

Argument marshalling only: every function below forwards to the entry point
of the same name in ``_build/libtranspose.so`` and every step of the
transpose runs in the library's CUDA kernels.  Pointers are integers (device
addresses); ``stream`` is a ``cudaStream_t`` as an integer (0 = legacy
default stream), e.g. ``torch.cuda.current_stream().cuda_stream``.

The library is opened on first use.  If it has not been built, or cannot be
loaded, every call raises ``LibraryMissing``: there is no fallback path.

``transpose`` / ``copy`` are conveniences for torch tensors: they read sizes
and pitches off the tensors' strides and call the same entry points.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

from . import build as _build

LIB_PATH = _build.LIB_PATH

_lock = threading.Lock()
_lib = None

I64 = ctypes.c_int64
VP = ctypes.c_void_p


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL = 1
    ERR_BAD_DIM = 2
    ERR_BAD_LD = 3
    ERR_OVERLAP = 4
    ERR_UNSUPPORTED = 5
    ERR_CUDA = 6
    ERR_TIMEOUT = 7


class DType(enum.IntEnum):
    F32 = 0
    BF16 = 1


class Variant(enum.IntEnum):
    AUTO = 0
    NAIVE_ROW = 1
    NAIVE_COL = 2
    TILE_PAD = 3
    TILE_VEC = 4
    TMA = 5


class Options(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("tile_order", ctypes.c_int32), ("out_stages", ctypes.c_int32),
                ("tile_rows", ctypes.c_int32), ("tile_cols", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("threads", ctypes.c_int32)]


class Args(ctypes.Structure):
    _fields_ = [("in_", VP), ("out", VP), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("batch", I64), ("rows", I64), ("cols", I64), ("ld_in", I64), ("ld_out", I64),
                ("stride_in", I64), ("stride_out", I64), ("stream", VP)]


class Plan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("tile_rows", ctypes.c_int32),
                ("tile_cols", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("vec_in", ctypes.c_int32),
                ("vec_out", ctypes.c_int32)]


class BoundsReport(ctypes.Structure):
    _fields_ = [("refused", I64), ("first_address", ctypes.c_uint64),
                ("first_bytes", ctypes.c_int32), ("first_store", ctypes.c_int32)]


class LibraryMissing(RuntimeError):
    pass


class TransposeError(RuntimeError):
    def __init__(self, status: int, message: str = ""):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{self.status!r}: {message}".rstrip(": "))


# Every symbol the header declares, with its ctypes signature.
SIGNATURES = {
    "tr_transpose_f32": ([VP, VP, I64, I64, I64, I64, VP], ctypes.c_int),
    "tr_transpose_bf16": ([VP, VP, I64, I64, I64, I64, VP], ctypes.c_int),
    "tr_transpose_batched_f32": ([VP, VP, I64, I64, I64, I64, I64, I64, I64, VP], ctypes.c_int),
    "tr_transpose_batched_bf16": ([VP, VP, I64, I64, I64, I64, I64, I64, I64, VP], ctypes.c_int),
    "tr_transpose_ex": ([ctypes.POINTER(Args), ctypes.POINTER(Options)], ctypes.c_int),
    "tr_copy": ([VP, VP, ctypes.c_size_t, VP], ctypes.c_int),
    "tr_transpose_inplace_f32": ([VP, I64, I64, I64, I64, VP], ctypes.c_int),
    "tr_transpose_inplace_bf16": ([VP, I64, I64, I64, I64, VP], ctypes.c_int),
    "tr_plan_variant": ([ctypes.POINTER(Args), ctypes.POINTER(Options)], ctypes.c_int32),
    "tr_plan_ex": ([ctypes.POINTER(Args), ctypes.POINTER(Options), ctypes.POINTER(Plan)],
                   ctypes.c_int),
    "tr_bank_probe": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, VP, VP], ctypes.c_int),
    "tr_operand_tiles_f32": ([VP, VP, I64, I64, I64, ctypes.c_int32, ctypes.c_int32,
                              ctypes.c_int32, VP], ctypes.c_int),
    "tr_device_status": ([], ctypes.c_int),
    "tr_selftest_bounded_wait": ([ctypes.c_int32, I64, VP], ctypes.c_int),
    "tr_debug_bounds": ([ctypes.POINTER(BoundsReport)], ctypes.c_int),
    "tr_debug_bounds_selftest": ([ctypes.c_uint64, VP], ctypes.c_int),
    "tr_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "tr_last_error": ([], ctypes.c_char_p),
    "tr_version": ([], ctypes.c_int32),
}


def open_library(path: str):
    """Open a build of the library at ``path`` (e.g. the bounds-checked one)
    as its own ctypes handle with every entry point's signature set."""
    if not os.path.exists(path):
        raise LibraryMissing(
            f"libtranspose is not built ({path} missing); run "
            "`python -m shared_memory_tiled_gb300.build`")
    try:
        lib = ctypes.CDLL(path)
    except OSError as e:  # pragma: no cover - depends on the machine
        raise LibraryMissing(f"cannot load {path}: {e}") from e
    for name, (argtypes, restype) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = restype
    return lib


def load(path: str | None = None):
    """Open the library (once) and return the ctypes handle."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(path or LIB_PATH)
    return _lib


def _call(name, *args):
    return getattr(load(), name)(*args)


# --- the C entry points, same names ------------------------------------------------

def tr_transpose_f32(in_ptr, out_ptr, rows, cols, ld_in, ld_out, stream=0) -> int:
    return _call("tr_transpose_f32", in_ptr, out_ptr, rows, cols, ld_in, ld_out, stream)


def tr_transpose_bf16(in_ptr, out_ptr, rows, cols, ld_in, ld_out, stream=0) -> int:
    return _call("tr_transpose_bf16", in_ptr, out_ptr, rows, cols, ld_in, ld_out, stream)


def tr_transpose_batched_f32(in_ptr, out_ptr, batch, rows, cols, ld_in, ld_out, stride_in,
                             stride_out, stream=0) -> int:
    return _call("tr_transpose_batched_f32", in_ptr, out_ptr, batch, rows, cols, ld_in, ld_out,
                 stride_in, stride_out, stream)


def tr_transpose_batched_bf16(in_ptr, out_ptr, batch, rows, cols, ld_in, ld_out, stride_in,
                              stride_out, stream=0) -> int:
    return _call("tr_transpose_batched_bf16", in_ptr, out_ptr, batch, rows, cols, ld_in, ld_out,
                 stride_in, stride_out, stream)


def make_args(in_ptr, out_ptr, dtype, batch, rows, cols, ld_in, ld_out, stride_in=0,
              stride_out=0, stream=0) -> Args:
    return Args(in_ptr, out_ptr, int(dtype), 0, batch, rows, cols, ld_in, ld_out, stride_in,
                stride_out, stream)


def make_options(variant=Variant.AUTO, pad=0, ctas_per_sm=0, stages=0, tile_order=0,
                 out_stages=0, tile_rows=0, tile_cols=0, schedule=0, threads=0) -> Options:
    return Options(int(variant), pad, ctas_per_sm, stages, tile_order, out_stages, tile_rows,
                   tile_cols, schedule, threads)


def tr_transpose_ex(args: Args, opts: Options | None = None) -> int:
    return _call("tr_transpose_ex", ctypes.byref(args), ctypes.byref(opts) if opts else None)


def tr_transpose_inplace_f32(ptr, batch, n, ld, stride, stream=0) -> int:
    return _call("tr_transpose_inplace_f32", ptr, batch, n, ld, stride, stream)


def tr_transpose_inplace_bf16(ptr, batch, n, ld, stride, stream=0) -> int:
    return _call("tr_transpose_inplace_bf16", ptr, batch, n, ld, stride, stream)


def tr_copy(in_ptr, out_ptr, nbytes, stream=0) -> int:
    return _call("tr_copy", in_ptr, out_ptr, nbytes, stream)


def tr_plan_variant(args: Args, opts: Options | None = None) -> int:
    return _call("tr_plan_variant", ctypes.byref(args), ctypes.byref(opts) if opts else None)


def tr_plan_ex(args: Args, opts: Options | None, plan: Plan) -> int:
    return _call("tr_plan_ex", ctypes.byref(args), ctypes.byref(opts) if opts else None,
                 ctypes.byref(plan) if plan is not None else None)


def tr_operand_tiles_f32(a_ptr, out_ptr, m, k, lda, bm, bk, pad=-1, stream=0) -> int:
    return _call("tr_operand_tiles_f32", a_ptr, out_ptr, m, k, lda, bm, bk, pad, stream)


def tr_bank_probe(layout, reps, blocks, result_ptr, stream=0) -> int:
    return _call("tr_bank_probe", layout, reps, blocks, result_ptr, stream)


def tr_selftest_bounded_wait(arrive, limit_ns, stream=0) -> int:
    return _call("tr_selftest_bounded_wait", arrive, limit_ns, stream)


def tr_debug_bounds(report: BoundsReport) -> int:
    return _call("tr_debug_bounds", ctypes.byref(report) if report is not None else None)


def tr_debug_bounds_selftest(base, stream=0) -> int:
    return _call("tr_debug_bounds_selftest", base, stream)


def tr_device_status() -> int:
    return _call("tr_device_status")


def tr_status_string(status: int) -> str:
    return _call("tr_status_string", int(status)).decode()


def tr_last_error() -> str:
    return _call("tr_last_error").decode()


def tr_version() -> int:
    return _call("tr_version")


def check(status: int) -> None:
    """Raise TransposeError for a non-OK status."""
    if status != Status.OK:
        raise TransposeError(status, f"{tr_status_string(status)}; {tr_last_error()}")


# --- torch conveniences -------------------------------------------------------------

def _dtype_of(t) -> DType:
    import torch
    if t.element_size() == 4 and t.dtype in (torch.float32, torch.int32, torch.uint32):
        return DType.F32
    if t.element_size() == 2 and t.dtype in (torch.bfloat16, torch.float16, torch.int16,
                                             torch.uint16):
        return DType.BF16
    raise TypeError(f"unsupported dtype {t.dtype}: 4-byte (fp32) or 2-byte (bf16) elements")


def _geometry(t):
    """(batch, rows, cols, ld, stride) of a 2-D or 3-D tensor with unit inner stride."""
    if t.dim() == 2:
        t = t.unsqueeze(0)
    if t.dim() != 3:
        raise ValueError("expected a 2-D or 3-D tensor")
    b, r, c = t.shape
    sb, sr, sc = t.stride()
    if c > 1 and sc != 1:
        raise ValueError("the innermost dimension must be contiguous")
    if r <= 1:
        sr = max(sr, c)
    if b <= 1:
        sb = max(sb, r * sr)
    return b, r, c, sr, sb


def transpose(x, out=None, *, variant=Variant.AUTO, pad=0, ctas_per_sm=0, stages=0,
              tile_order=0, out_stages=0, tile_rows=0, tile_cols=0, schedule=0, threads=0,
              stream=None):
    """Transpose the last two dims of a CUDA tensor ``x`` ([R, C] or [B, R, C]).

    ``out`` (optional) receives the result and may be a strided view (its row
    pitch becomes ``ld_out``); otherwise a dense output is allocated with torch.
    Launches asynchronously on ``stream`` (default: torch's current stream).
    """
    import torch
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor: the library has no CPU path")
    dt = _dtype_of(x)
    b, r, c, ld_in, s_in = _geometry(x)
    if out is None:
        shape = (c, r) if x.dim() == 2 else (b, c, r)
        out = torch.empty(shape, dtype=x.dtype, device=x.device)
    if out.dtype != x.dtype or out.device != x.device:
        raise ValueError("out must match x in dtype and device")
    ob, orr, oc, ld_out, s_out = _geometry(out)
    if (ob, orr, oc) != (b, c, r):
        raise ValueError(f"out has shape {tuple(out.shape)}, expected {(b, c, r)}")
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    args = make_args(x.data_ptr(), out.data_ptr(), dt, b, r, c, ld_in, ld_out, s_in, s_out,
                     stream)
    opts = make_options(variant, pad, ctas_per_sm, stages, tile_order, out_stages, tile_rows,
                        tile_cols, schedule, threads)
    with torch.cuda.device(x.device):  # the library sets kernels up per current device
        check(tr_transpose_ex(args, opts))
    return out


def copy(src, dst, stream=None):
    """Byte copy of a contiguous CUDA tensor into another of the same byte size
    (on the same device)."""
    import torch
    if not (src.is_cuda and dst.is_cuda and src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("copy wants contiguous CUDA tensors")
    n = src.numel() * src.element_size()
    if n != dst.numel() * dst.element_size():
        raise ValueError("size mismatch")
    if src.device != dst.device:
        raise ValueError("copy wants both tensors on one device")
    if stream is None:
        stream = torch.cuda.current_stream(src.device).cuda_stream
    with torch.cuda.device(src.device):
        check(tr_copy(src.data_ptr(), dst.data_ptr(), n, stream))
    return dst


def transpose_(x, stream=None):
    """Transpose the last two (equal) dims of a CUDA tensor in place."""
    import torch
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor: the library has no CPU path")
    dt = _dtype_of(x)
    b, r, c, ld, s = _geometry(x)
    if r != c:
        raise ValueError("in-place transpose needs square planes")
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    f = tr_transpose_inplace_f32 if dt == DType.F32 else tr_transpose_inplace_bf16
    with torch.cuda.device(x.device):
        check(f(x.data_ptr(), b, r, ld, s, stream))
    return x
