"""The bounds-checked build (``TR_DEBUG``): every global load and store of
every kernel is checked against its side before it is made; a refused access
is skipped and counted, never performed ("Shared memory and the bank
conflict", "The barrier": an indexing mistake can leave the output right most
of the time, so the addresses themselves are checked).

The library is built a second time into ``_build_debug/`` and opened as its
own handle.  The cases are the ones whose addresses come from run-time shifts
and halos -- odd output pitches (shifted stores fed by halo rows), odd input
pitches (bf16 rows realigned on chip, fp32 widest per-chunk loads), both at
once -- every variant, the in-place transpose, the copy, the operand-tile stage,
the bank probe, a replay of the release fuzz sweep's random configurations,
every configured workload at full size and one case past 2**31 elements.  Each output is compared with the oracle bit for
bit, and the record of refused accesses must stay empty."""
from __future__ import annotations

import ctypes
import zlib

import numpy as np
import pytest

import pins
from fuzz_cases import U16, U32, draw
from gpu_util import first_mismatch, from_device, gpu_out, mismatch_report, oracle_out, \
    oracle_out_banded, to_device
from shared_memory_tiled_gb300 import binding as B
from shared_memory_tiled_gb300 import workloads as W

pytestmark = pytest.mark.gpu

V = B.Variant


@pytest.fixture(scope="module")
def dlib():
    from shared_memory_tiled_gb300 import build
    lib = B.open_library(build.build(debug=True))
    assert _report(lib).refused == 0
    return lib


def _report(lib) -> B.BoundsReport:
    rep = B.BoundsReport()
    st = lib.tr_debug_bounds(ctypes.byref(rep))
    assert st == B.Status.OK, st
    return rep


def _clean(lib, what):
    rep = _report(lib)
    assert rep.refused == 0, (
        f"{what}: {rep.refused} accesses refused, e.g. a {rep.first_bytes}-byte "
        f"{'store' if rep.first_store else 'load'} at 0x{rep.first_address:x}")


def test_guards_refuse_what_they_should(dlib):
    """The guards' own self-test: of five accesses to a made-up side that is
    never dereferenced, exactly the two that leave it are refused."""
    import torch
    base = 0x10000
    assert dlib.tr_debug_bounds_selftest(base, 0) == B.Status.OK
    torch.cuda.synchronize()
    rep = _report(dlib)
    assert rep.refused == 2
    assert rep.first_address == base + 212 and rep.first_bytes == 4 and rep.first_store == 0
    assert _report(dlib).refused == 0  # reading clears the record


def _check(dlib, dtype, geo, what, in_off=0, out_off=0, **opt):
    x, prefill, _ = pins.alloc_case(dtype, *geo, seed=zlib.crc32(what.encode()) & 0xFFFF)
    want = oracle_out(x, prefill, *geo)
    got = gpu_out(x, prefill, *geo, in_off=in_off, out_off=out_off, lib=dlib, **opt)
    assert np.array_equal(got, want), f"{what}: {first_mismatch(got, want)}"
    _clean(dlib, what)


def _geo(rows, cols, ld_in, ld_out, batch=1, gap=0):
    return (batch, rows, cols, ld_in, ld_out, rows * ld_in + gap, cols * ld_out + gap)


ODD = [
    # (rows, cols, ld_in, ld_out, batch, gap): odd output pitch, odd input
    # pitch, both, with tiles that end inside the matrix and batches with gaps
    (1229, 791, 800, 1229, 1, 0),
    (791, 1229, 1229, 800, 1, 0),
    (1229, 791, 793, 1231, 1, 0),
    (300, 517, 521, 303, 3, 5),
    (129, 65, 67, 131, 2, 7),
    (1000, 77, 77, 1001, 1, 0),
    (33, 1031, 1033, 35, 1, 0),
]


@pytest.mark.parametrize("dtype", [U32, U16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", ODD, ids=[f"{r}x{c}_ld{a}_{b}_b{n}" for r, c, a, b, n, _ in ODD])
def test_misaligned_pitches(dlib, dtype, case):
    rows, cols, ld_in, ld_out, batch, gap = case
    geo = _geo(rows, cols, ld_in, ld_out, batch, gap)
    _check(dlib, dtype, geo, f"AUTO {case}")
    for nt, tr, tc in ((256, 128, 64), (256, 64, 128), (128, 128, 64)) if dtype is U32 else \
            ((256, 128, 128), (128, 64, 128), (128, 128, 128)):
        _check(dlib, dtype, geo, f"TILE_VEC {tr}x{tc}/{nt} {case}", variant=V.TILE_VEC,
               threads=nt, tile_rows=tr, tile_cols=tc)


@pytest.mark.parametrize("dtype", [U32, U16], ids=["fp32", "bf16"])
def test_every_variant(dlib, dtype):
    vec = 4 if dtype is U32 else 8
    shapes = [(1, 1, 1, 1), (257, 129, 129, 257), (200, 333, 333 + (-333) % vec, 200 + (-200) % vec),
              (128, 128, 128, 128)]
    for rows, cols, ld_in, ld_out in shapes:
        geo = _geo(rows, cols, ld_in, ld_out)
        aligned = (ld_in * (16 // vec)) % 16 == 0 and (ld_out * (16 // vec)) % 16 == 0
        opts = [dict(variant=V.AUTO), dict(variant=V.TILE_VEC, schedule=2),
                dict(variant=V.TILE_VEC, tile_order=1), dict(variant=V.NAIVE_ROW),
                dict(variant=V.NAIVE_COL)] + [dict(variant=V.TILE_PAD, pad=p) for p in (0, 1, 2)]
        if aligned:
            opts += [dict(variant=V.TMA, schedule=s) for s in range(5)]
        for opt in opts:
            _check(dlib, dtype, geo, f"{opt} {rows}x{cols} ld {ld_in}/{ld_out}", **opt)


@pytest.mark.parametrize("seed", range(2))
def test_random_configurations(dlib, seed):
    """The release fuzz sweep's first cases, replayed through the checked build."""
    rng = np.random.default_rng(1000 + seed)
    for k in range(120):
        dtype, geo, in_off, out_off, opt = draw(rng)
        x, prefill, _ = pins.alloc_case(dtype, *geo, seed=int(rng.integers(1 << 30)))
        want = oracle_out(x, prefill, *geo)
        got = gpu_out(x, prefill, *geo, in_off=in_off, out_off=out_off, lib=dlib, **opt)
        what = f"case {k}: {np.dtype(dtype).name} {geo} offsets {in_off}/{out_off} {opt}"
        assert np.array_equal(got, want), f"{what}: {first_mismatch(got, want)}"
        _clean(dlib, what)


def test_inplace_copy_operand_tiles_probe(dlib):
    import oracle
    import torch
    rng = np.random.default_rng(7)
    for k in range(40):
        dt = U32 if k % 2 == 0 else U16
        vec = 4 if dt is U32 else 8
        batch = int(rng.choice([1, 2]))
        n = int(rng.integers(1, 400))
        ld = n + int(rng.choice([0, 1, 3, (-n) % vec]))
        stride = n * ld + (int(rng.integers(0, 9)) if batch > 1 else 0)
        off = int(rng.choice([0, 1]))
        x = rng.integers(0, np.iinfo(dt).max, batch * stride, dtype=dt, endpoint=True)
        want = oracle.transpose_inplace(x.copy(), batch=batch, n=n, ld=ld, stride=stride)
        buf, ptr = to_device(x, off)
        fn = dlib.tr_transpose_inplace_f32 if dt is U32 else dlib.tr_transpose_inplace_bf16
        assert fn(ptr, batch, n, ld, stride, None) == B.Status.OK
        torch.cuda.synchronize()
        got = from_device(buf, x.size, off, dt)
        what = f"in place {np.dtype(dt).name} batch {batch} n {n} ld {ld} offset {off}"
        assert np.array_equal(got, want), f"{what}: {first_mismatch(got, want)}"
        _clean(dlib, what)

    for n in (1, 15, 16, 17, 4095, 1 << 20, (1 << 20) + 13):
        for a, b in ((0, 0), (3, 3), (1, 5), (2, 6)):
            src = torch.randint(0, 255, (n + 32,), dtype=torch.uint8, device="cuda")
            dst = torch.zeros(n + 32, dtype=torch.uint8, device="cuda")
            assert dlib.tr_copy(src.data_ptr() + a, dst.data_ptr() + b, n, None) == 0
            torch.cuda.synchronize()
            assert torch.equal(dst[b:b + n], src[a:a + n])
            assert int(dst[:b].count_nonzero()) == 0 and int(dst[b + n:].count_nonzero()) == 0
            _clean(dlib, f"copy of {n} bytes, offsets {a}/{b}")

    m, kk = 256, 96
    a = torch.randint(-2**31, 2**31 - 1, (m * (kk + 4),), dtype=torch.int32, device="cuda")
    for bm, bk in ((128, 32), (64, 16)):
        out = torch.zeros(m * kk, dtype=torch.int32, device="cuda")
        assert dlib.tr_operand_tiles_f32(a.data_ptr(), out.data_ptr(), m, kk, kk + 4, bm, bk, -1,
                                         None) == 0
        torch.cuda.synchronize()
        want = np.zeros(m * kk, dtype=np.uint32)
        oracle.operand_tiles(a.cpu().numpy().view(np.uint32), want, m=m, k=kk, lda=kk + 4, bm=bm,
                             bk=bk)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want)
        _clean(dlib, f"operand tiles {bm}x{bk}")

    res = torch.zeros(4 * 256, dtype=torch.int32, device="cuda")
    for layout in range(4):
        assert dlib.tr_bank_probe(layout, 64, 4, res.data_ptr(), None) == 0
        torch.cuda.synchronize()
        _clean(dlib, f"bank probe layout {layout}")


def test_beyond_2_31_elements_both_pitches_odd(dlib):
    """bf16 past 2**31 elements with both pitches odd: realigned loads and
    shifted stores with 64-bit addresses, every access checked."""
    import torch
    rows, cols, ld_in, ld_out = 65537, 32801, 32803, 65539
    n_in, n_out = (rows - 1) * ld_in + cols, (cols - 1) * ld_out + rows + 16
    g = torch.Generator(device="cuda").manual_seed(21)
    x = torch.randint(-2**15, 2**15 - 1, (n_in,), dtype=torch.int16, device="cuda", generator=g)
    out = torch.full((n_out,), -66, dtype=torch.int16, device="cuda")   # 0xFFBE
    args = B.make_args(x.data_ptr(), out.data_ptr(), B.DType.BF16, 1, rows, cols, ld_in, ld_out)
    opts = B.make_options(V.AUTO)
    assert dlib.tr_transpose_ex(ctypes.byref(args), ctypes.byref(opts)) == B.Status.OK
    torch.cuda.synchronize()
    _clean(dlib, "bf16 65537x32801, pitches 32803/65539")
    x_host = x.cpu().numpy().view(np.uint16)
    got = out.cpu().numpy().view(np.uint16)
    del x, out
    torch.cuda.empty_cache()
    want = np.full(n_out, 0xFFBE, dtype=np.uint16)
    oracle_out_banded(x_host, want, 1, rows, cols, ld_in, ld_out, 0, 0)
    assert mismatch_report(got, want) == "identical"


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_configured_workloads_full_size(dlib, name):
    """Every configured workload at full size through AUTO (and the default TMA
    pipeline where both sides allow it): oracle-exact, nothing refused."""
    w = W.WORKLOADS[name]
    x = W.make_input(w)
    prefill = W.make_output(w)
    geo = (w.batch, w.rows, w.cols, w.ld_in, w.ld_out, w.sin, w.sout)
    want = oracle_out(x, prefill, *geo)
    aligned = (w.ld_in * w.esize) % 16 == 0 and (w.ld_out * w.esize) % 16 == 0
    for opt in [dict(variant=V.AUTO)] + ([dict(variant=V.TMA)] if aligned else []):
        got = gpu_out(x, prefill, *geo, lib=dlib, **opt)
        assert np.array_equal(got, want), f"{name} {opt}: {first_mismatch(got, want)}"
        _clean(dlib, f"{name} {opt}")


@pytest.mark.parametrize("name", ["c2", "c5"])
def test_inplace_full_size(dlib, name):
    import oracle
    import torch
    w = W.WORKLOADS[name]
    x = W.make_input(w)
    want = oracle.transpose_inplace(x.copy(), n=w.rows)
    buf, ptr = to_device(x)
    fn = dlib.tr_transpose_inplace_f32 if w.esize == 4 else dlib.tr_transpose_inplace_bf16
    assert fn(ptr, 1, w.rows, w.ld_in, w.sin, None) == B.Status.OK
    torch.cuda.synchronize()
    got = from_device(buf, x.size, 0, x.dtype.type)
    assert np.array_equal(got, want), f"{name} in place: {first_mismatch(got, want)}"
    _clean(dlib, f"{name} in place")
