"""Sizes past 2**31 elements and 2**32 bytes: the 64-bit index arithmetic of
every kernel.  Each case transposes random bit patterns on the GPU into an
output buffer prefilled with a sentinel, copies the whole output buffer back
and compares it bit for bit with the oracle's result on the same input and the
same prefill (pitch padding included), with the oracle run band by band on
every host core ("Shared memory and the bank conflict", "The barrier": every
element checked at its own index)."""
import numpy as np
import pytest

from shared_memory_tiled_gb300 import binding as B
from gpu_util import mismatch_report, oracle_out_banded

pytestmark = pytest.mark.gpu

PREFILL = {np.uint32: 0xFFC0BEEF, np.uint16: 0xFFBE}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()


def tdt_np(dtype):
    return np.int32 if dtype is np.uint32 else np.int16


def _run(dtype, batch, rows, cols, ld_in, ld_out, si, so, seed, call):
    """Random input of the whole input extent, sentinel-prefilled output; run
    ``call(in_ptr, out_ptr)`` on the GPU; return (got, want) as flat host arrays."""
    import torch
    tdt = torch.int32 if dtype is np.uint32 else torch.int16
    n_in = (batch - 1) * si + (rows - 1) * ld_in + cols
    n_out = (batch - 1) * so + (cols - 1) * ld_out + rows + 16   # 16 elements past the extent
    g = torch.Generator(device="cuda").manual_seed(seed)
    bits = 32 if dtype is np.uint32 else 16
    x = torch.randint(-2 ** (bits - 1), 2 ** (bits - 1) - 1, (n_in,), dtype=tdt, device="cuda",
                      generator=g)
    fill = int(np.array(PREFILL[dtype], dtype=dtype).view(tdt_np(dtype)))
    out = torch.full((n_out,), fill, dtype=tdt, device="cuda")
    B.check(call(x.data_ptr(), out.data_ptr()))
    torch.cuda.synchronize()
    x_host = x.cpu().numpy().view(dtype)
    got = out.cpu().numpy().view(dtype)
    del x, out
    torch.cuda.empty_cache()
    want = np.full(n_out, PREFILL[dtype], dtype=dtype)
    oracle_out_banded(x_host, want, batch, rows, cols, ld_in, ld_out, si, so)
    return got, want


def _ex(dt, batch, rows, cols, ld_in, ld_out, si, so, variant=B.Variant.AUTO, schedule=0):
    def call(pi, po):
        args = B.make_args(pi, po, dt, batch, rows, cols, ld_in, ld_out, si, so)
        return B.tr_transpose_ex(args, B.make_options(variant, schedule=schedule))
    return call


@pytest.mark.parametrize("variant,schedule", [(B.Variant.AUTO, 0), (B.Variant.TMA, 0),
                                              (B.Variant.TMA, 3), (B.Variant.TMA, 4)])
def test_fp32_beyond_2_31_elements(variant, schedule):
    rows, cols = 65537, 32801          # 2,149,679,137 elements, 8.6 GB each way
    ld_in, ld_out = 32804, 65540       # 16-byte aligned pitches (TMA-eligible)
    got, want = _run(np.uint32, 1, rows, cols, ld_in, ld_out, 0, 0, 11,
                     _ex(B.DType.F32, 1, rows, cols, ld_in, ld_out, 0, 0, variant, schedule))
    assert mismatch_report(got, want) == "identical"


def test_bf16_batched_beyond_2_32_bytes():
    batch, rows, cols = 3, 40000, 24000   # 2.88e9 elements, 5.76 GB each way
    si = so = rows * cols

    def call(pi, po):
        return B.tr_transpose_batched_bf16(pi, po, batch, rows, cols, cols, rows, si, so)

    got, want = _run(np.uint16, batch, rows, cols, cols, rows, si, so, 12, call)
    assert mismatch_report(got, want) == "identical"


def test_fp32_batched_beyond_2_32_bytes_tma():
    """The TMA path's 3-D tensor maps with planes starting past 2**32 bytes."""
    batch, rows, cols = 3, 32000, 24000   # 2.3e9 elements, 9.2 GB each way; plane 2 at 6.1 GB
    si = so = rows * cols
    got, want = _run(np.uint32, batch, rows, cols, cols, rows, si, so, 13,
                     _ex(B.DType.F32, batch, rows, cols, cols, rows, si, so, B.Variant.TMA))
    assert mismatch_report(got, want) == "identical"


def test_inplace_beyond_2_31_elements():
    import torch
    n = 46349                              # 2,148,229,801 elements
    g = torch.Generator(device="cuda").manual_seed(14)
    x = torch.randint(-2**31, 2**31 - 1, (n * n,), dtype=torch.int32, device="cuda", generator=g)
    x_host = x.cpu().numpy().view(np.uint32)
    B.check(B.tr_transpose_inplace_f32(x.data_ptr(), 1, n, n, n * n))
    torch.cuda.synchronize()
    got = x.cpu().numpy().view(np.uint32)
    del x
    torch.cuda.empty_cache()
    # the in-place result is the out-of-place transpose of the original planes
    want = np.empty_like(x_host)
    oracle_out_banded(x_host, want, 1, n, n, n, n, n * n, n * n)
    assert mismatch_report(got, want) == "identical"


@pytest.mark.parametrize("ld_in,ld_out", [(32804, 65539), (32803, 65540)],
                         ids=["odd-output-pitch", "odd-input-pitch"])
def test_fp32_misaligned_pitches_beyond_2_31_elements(ld_in, ld_out):
    """Past 2**31 elements with rows that start off 16-byte boundaries: the
    shifted stores (with their halo rows) on the output side, per-chunk 4-byte
    loads on the input side."""
    rows, cols = 65537, 32801          # 2,149,679,137 elements
    got, want = _run(np.uint32, 1, rows, cols, ld_in, ld_out, 0, 0, 15,
                     _ex(B.DType.F32, 1, rows, cols, ld_in, ld_out, 0, 0))
    assert mismatch_report(got, want) == "identical"


@pytest.mark.parametrize("ld_in,ld_out", [(32803, 65544), (32803, 65539)],
                         ids=["odd-input-pitch", "both-pitches-odd"])
def test_bf16_misaligned_pitches_beyond_2_31_elements(ld_in, ld_out):
    """bf16 past 2**31 elements with input rows at every 2-byte offset from a
    16-byte boundary: aligned chunks realigned on chip (row offsets taken from
    the low 32 bits of the addresses), alone and with shifted stores."""
    rows, cols = 65537, 32801          # 2,149,679,137 elements, 4.3 GB each way
    got, want = _run(np.uint16, 1, rows, cols, ld_in, ld_out, 0, 0, 16,
                     _ex(B.DType.BF16, 1, rows, cols, ld_in, ld_out, 0, 0))
    assert mismatch_report(got, want) == "identical"
