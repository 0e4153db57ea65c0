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
            variant=B.Variant.AUTO, in_off=0, out_off=0, entry="ex", stream=0, **opt):
    """Transpose on the GPU through the C ABI; returns the whole output buffer."""
    import torch
    dt = B.DType.F32 if x.dtype == np.uint32 else B.DType.BF16
    dev_in, p_in = to_device(x, in_off)
    dev_out, p_out = to_device(prefill, out_off)
    torch.cuda.synchronize()
    if entry == "ex":
        args = B.make_args(p_in, p_out, dt, batch, rows, cols, ld_in, ld_out, si, so, stream)
        st = B.tr_transpose_ex(args, B.make_options(variant, **opt))
    elif entry == "plain":
        assert batch == 1
        f = B.tr_transpose_f32 if dt == B.DType.F32 else B.tr_transpose_bf16
        st = f(p_in, p_out, rows, cols, ld_in, ld_out, stream)
    elif entry == "batched":
        f = B.tr_transpose_batched_f32 if dt == B.DType.F32 else B.tr_transpose_batched_bf16
        st = f(p_in, p_out, batch, rows, cols, ld_in, ld_out, si, so, stream)
    else:
        raise ValueError(entry)
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
