"""Helpers for the GPU parity tests: run one transpose through the C ABI on
device copies of host buffers, and the oracle on the same host buffers."""
from __future__ import annotations

import numpy as np

import oracle
from shared_memory_tiled_gb300 import binding as B

TORCH_VIEW = {np.uint32: np.int32, np.uint16: np.int16}


def to_device(host: np.ndarray, offset_elems: int = 0, slack: int = 16):
    """Copy a flat uint32/uint16 host array into a fresh device buffer, starting
    ``offset_elems`` elements into it; returns (buffer, pointer to the copy)."""
    import torch
    view = host.view(TORCH_VIEW[host.dtype.type])
    buf = torch.empty(host.size + offset_elems + slack, dtype=torch.from_numpy(view[:0]).dtype,
                      device="cuda")
    buf[offset_elems: offset_elems + host.size].copy_(torch.from_numpy(view))
    return buf, buf.data_ptr() + offset_elems * host.itemsize


def from_device(buf, n: int, offset_elems: int, dtype) -> np.ndarray:
    return buf[offset_elems: offset_elems + n].cpu().numpy().view(dtype)


def oracle_out(x: np.ndarray, prefill: np.ndarray, batch, rows, cols, ld_in, ld_out, si, so):
    out = prefill.copy()
    oracle.transpose(x, out, batch=batch, rows=rows, cols=cols, ld_in=ld_in, ld_out=ld_out,
                     stride_in=si, stride_out=so)
    return out


def gpu_out(x: np.ndarray, prefill: np.ndarray, batch, rows, cols, ld_in, ld_out, si, so,
            variant=B.Variant.AUTO, in_off=0, out_off=0, entry="ex", stream=0, lib=None, **opt):
    """Transpose on the GPU through the C ABI; returns the whole output buffer.
    ``lib`` is a library handle from ``binding.open_library`` (another build of
    the library, e.g. the bounds-checked one), used with entry="ex"; default:
    the binding's own library."""
    import ctypes

    import torch
    dt = B.DType.F32 if x.dtype == np.uint32 else B.DType.BF16
    dev_in, p_in = to_device(x, in_off)
    dev_out, p_out = to_device(prefill, out_off)
    torch.cuda.synchronize()
    if entry == "ex":
        args = B.make_args(p_in, p_out, dt, batch, rows, cols, ld_in, ld_out, si, so, stream)
        opts = B.make_options(variant, **opt)
        st = (lib.tr_transpose_ex(ctypes.byref(args), ctypes.byref(opts)) if lib is not None
              else B.tr_transpose_ex(args, opts))
    elif entry == "plain":
        assert batch == 1
        f = B.tr_transpose_f32 if dt == B.DType.F32 else B.tr_transpose_bf16
        st = f(p_in, p_out, rows, cols, ld_in, ld_out, stream)
    elif entry == "batched":
        f = B.tr_transpose_batched_f32 if dt == B.DType.F32 else B.tr_transpose_batched_bf16
        st = f(p_in, p_out, batch, rows, cols, ld_in, ld_out, si, so, stream)
    else:
        raise ValueError(entry)
    if st != B.Status.OK and lib is not None:
        raise B.TransposeError(st, lib.tr_last_error().decode())
    B.check(st)
    torch.cuda.synchronize()
    return from_device(dev_out, prefill.size, out_off, x.dtype.type)


def first_mismatch(got: np.ndarray, want: np.ndarray) -> str:
    bad = np.flatnonzero(got != want)
    if bad.size == 0:
        return "identical"
    k = bad[0]
    return (f"{bad.size} mismatches, first at flat index {k}: got 0x{int(got[k]):x} "
            f"want 0x{int(want[k]):x}")


def oracle_out_banded(x: np.ndarray, out: np.ndarray, batch, rows, cols, ld_in, ld_out, si, so,
                      threads: int | None = None) -> np.ndarray:
    """The oracle's transpose of ``x`` into ``out`` (in place), run as one call
    per batch plane and band of input rows on every host core.  Each call is
    the oracle's own loop restricted to those rows (input rows r0..r0+n-1 fill
    output columns r0..r0+n-1 of every output row), so the union of the calls
    writes exactly what one whole call writes; the loop releases the
    interpreter lock, so bands run in parallel."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    n = threads or len(os.sched_getaffinity(0))
    step = max(1, -(-rows // n))
    jobs = [(b, r0, min(step, rows - r0)) for b in range(batch) for r0 in range(0, rows, step)]

    def one(job):
        b, r0, nr = job
        oracle.transpose(x[b * si + r0 * ld_in:], out[b * so + r0:], rows=nr, cols=cols,
                         ld_in=ld_in, ld_out=ld_out)

    with ThreadPoolExecutor(max_workers=n) as pool:
        list(pool.map(one, jobs))
    return out


def mismatch_report(got: np.ndarray, want: np.ndarray, chunk: int = 1 << 26) -> str:
    """Bitwise comparison of two equal-length flat arrays, chunk by chunk (so no
    full-size temporary is made): "identical" or the count and first mismatch."""
    assert got.dtype == want.dtype and got.size == want.size
    count, first = 0, None
    for s in range(0, got.size, chunk):
        bad = np.flatnonzero(got[s:s + chunk] != want[s:s + chunk])
        if bad.size:
            count += bad.size
            if first is None:
                first = s + int(bad[0])
    if first is None:
        return "identical"
    return (f"{count} mismatches, first at flat index {first}: got 0x{int(got[first]):x} "
            f"want 0x{int(want[first]):x}")
