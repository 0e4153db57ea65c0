"""GPU parity: every kernel variant against the CPU oracle, bit for bit, through
the C ABI.  The whole output buffer is compared, pitch padding included (it
must keep its prefill)."""
from __future__ import annotations


import numpy as np
import pytest

import pins
from gpu_util import first_mismatch, gpu_out, oracle_out
from shared_memory_tiled_gb300 import binding as B
from shared_memory_tiled_gb300 import workloads as W

pytestmark = pytest.mark.gpu

V = B.Variant
U32, U16 = np.uint32, np.uint16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()
    yield
    assert B.tr_device_status() == B.Status.OK, "a bounded in-kernel wait ran out"


def case(dtype, batch, rows, cols, ld_pad_in=0, ld_pad_out=0, plane_pad=0, seed=0, values=None):
    ld_in, ld_out = cols + ld_pad_in, rows + ld_pad_out
    si, so = rows * ld_in + plane_pad, cols * ld_out + plane_pad
    x, prefill, p = pins.alloc_case(dtype, batch, rows, cols, ld_in, ld_out, si, so,
                                    values=values, seed=seed)
    return x, prefill, (batch, rows, cols, ld_in, ld_out, si, so)


def check(x, prefill, geo, **kw):
    want = oracle_out(x, prefill, *geo)
    got = gpu_out(x, prefill, *geo, **kw)
    assert np.array_equal(got, want), f"{geo} {kw}: {first_mismatch(got, want)}"


SHAPES = [(1, 1), (1, 300), (300, 1), (64, 64), (128, 128), (200, 333), (257, 129),
          (1000, 77), (33, 1031)]


VEC_SHAPES = {U32: [(128, 64), (64, 128), (128, 128), (128, 32)],
              U16: [(256, 128), (128, 256), (256, 64)]}
VEC_128 = {U32: [(64, 64), (32, 64), (128, 64)], U16: [(128, 128), (64, 128)]}
VEC_SMALL = {U32: [(64, 32, 64), (64, 64, 32), (32, 32, 32)],
             U16: [(64, 64, 128), (64, 128, 64), (32, 64, 64)]}  # threads, rows, cols


def _variants(dtype, aligned):
    vs = [dict(variant=V.NAIVE_ROW), dict(variant=V.NAIVE_COL),
          dict(variant=V.TILE_PAD, pad=0), dict(variant=V.TILE_PAD, pad=1),
          dict(variant=V.TILE_PAD, pad=2), dict(variant=V.TILE_VEC), dict(variant=V.AUTO)]
    vs += [dict(variant=V.TILE_VEC, tile_rows=r, tile_cols=c) for r, c in VEC_SHAPES[dtype]]
    vs += [dict(variant=V.TILE_VEC, threads=128, tile_rows=r, tile_cols=c) for r, c in VEC_128[dtype]]
    vs += [dict(variant=V.TILE_VEC, threads=n, tile_rows=r, tile_cols=c)
           for n, r, c in VEC_SMALL[dtype]]
    vs += [dict(variant=V.TILE_VEC, schedule=2),
           dict(variant=V.TILE_VEC, schedule=2, tile_rows=VEC_SHAPES[dtype][0][0],
                tile_cols=VEC_SHAPES[dtype][0][1])]
    if aligned:
        deep = 6 if dtype is U32 else 4   # 8 x 32 KiB bf16 stages would not fit
        vs += [dict(variant=V.TMA), dict(variant=V.TMA, stages=3, out_stages=3),
               dict(variant=V.TMA, stages=2, out_stages=4, ctas_per_sm=1),
               dict(variant=V.TMA, stages=8, tile_order=1),
               dict(variant=V.TMA, schedule=1), dict(variant=V.TMA, schedule=1, stages=3,
                                                     out_stages=3),
               dict(variant=V.TMA, schedule=1, stages=deep, tile_order=1),
               dict(variant=V.TMA, schedule=3), dict(variant=V.TMA, schedule=3, stages=2),
               dict(variant=V.TMA, schedule=3, stages=8, tile_order=1),
               dict(variant=V.TMA, schedule=4), dict(variant=V.TMA, schedule=4, stages=2),
               dict(variant=V.TMA, schedule=4, stages=3, ctas_per_sm=1),
               dict(variant=V.TMA, schedule=4, stages=deep + 2, tile_order=1)]
    return vs


@pytest.mark.parametrize("dtype", [U32, U16], ids=["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_small_shapes_all_variants(dtype, rows, cols):
    """Dense pitches: several tiles plus ragged tails on both axes."""
    x, prefill, geo = case(dtype, 1, rows, cols, seed=rows * 7 + cols)
    aligned = (cols * x.itemsize) % 16 == 0 and (rows * x.itemsize) % 16 == 0
    for kw in _variants(dtype, aligned):
        check(x, prefill, geo, **kw)


@pytest.mark.parametrize("dtype", [U32, U16], ids=["f32", "bf16"])
def test_pitched_and_batched(dtype):
    """Row pitches that keep or break 16-byte alignment, gaps between planes."""
    al = 16 // np.dtype(dtype).itemsize
    for (b, r, c, pi, po, pp) in [(1, 130, 70, al, 2 * al, 0), (3, 65, 129, 3, 5, 7),
                                  (4, 96, 160, al, al, 4 * al), (2, 129, 257, 1, 0, 1),
                                  (5, 8, 8, 0, 0, 0), (1, 70, 130, 6 * al, 3, 0),
                                  # 16-byte aligned pitches but output rows that end
                                  # mid-chunk (the TMA path's element-store edge)
                                  (1, 190, 250, 6, 10, 0), (2, 190, 250, 6, 10, 8),
                                  (1, 61, 64, 0, 3, 0), (3, 129, 8, 0, 7, 0)]:
        x, prefill, geo = case(dtype, b, r, c, pi, po, pp, seed=b + r + c)
        es = np.dtype(dtype).itemsize
        aligned = all(v * es % 16 == 0 for v in (geo[3], geo[4])) and \
            (b == 1 or all(v * es % 16 == 0 for v in (geo[5], geo[6])))
        for kw in _variants(dtype, aligned):
            check(x, prefill, geo, **kw)


@pytest.mark.parametrize("dtype", [U32, U16], ids=["f32", "bf16"])
def test_misaligned_base_pointers(dtype):
    """Base pointers off a 16-byte boundary: the vector tile falls back to
    single-element accesses on that side; TMA refuses."""
    x, prefill, geo = case(dtype, 2, 100, 136, 8, 8, seed=3)
    for in_off, out_off in [(1, 0), (0, 1), (3, 5), (2, 7)]:
        for kw in [dict(variant=V.AUTO), dict(variant=V.TILE_VEC), dict(variant=V.TILE_PAD, pad=1)] + \
                [dict(variant=V.TILE_VEC, tile_rows=r, tile_cols=c) for r, c in VEC_SHAPES[dtype]]:
            check(x, prefill, geo, in_off=in_off, out_off=out_off, **kw)
        with pytest.raises(B.TransposeError) as e:
            gpu_out(x, prefill, *geo, variant=V.TMA, in_off=in_off, out_off=out_off)
        assert e.value.status == B.Status.ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", [U32, U16], ids=["f32", "bf16"])
def test_input_pitch_not_a_multiple_of_16_bytes(dtype):
    """Odd input pitches and base offsets.  bf16 tiles inside the matrix read
    aligned 16-byte chunks and realign them on chip, except the first tile and
    a tile holding the last row whose segments end within one chunk of its end
    (per-chunk loads there); the shapes put full tiles against both of those
    edges, with one or more planes and aligned or odd output pitches."""
    vec = 16 // np.dtype(dtype).itemsize
    kws = [dict(variant=V.AUTO), dict(variant=V.TILE_VEC, schedule=2)] + \
        [dict(variant=V.TILE_VEC, tile_rows=r, tile_cols=c) for r, c in VEC_SHAPES[dtype]] + \
        [dict(variant=V.TILE_VEC, threads=128, tile_rows=r, tile_cols=c) for r, c in VEC_128[dtype]]
    for (b, r, c, pi, po, pp) in [(1, 256, 256, 1, 0, 0), (1, 256, 257, 3, 0, 0),
                                  (2, 256, 256 + vec - 1, 5, 0, 3), (1, 256, 256 + vec, 1, 0, 0),
                                  (1, 384, 264, 1, 1, 0), (3, 129, 385, 7, 3, 2),
                                  (2, 512, 128, 2, 5, 0)]:
        x, prefill, geo = case(dtype, b, r, c, pi, po, pp, seed=r + c + pi)
        for in_off in (0, 1, vec - 1):
            for kw in kws:
                check(x, prefill, geo, in_off=in_off, **kw)


@pytest.mark.parametrize("dtype", [U32, U16], ids=["f32", "bf16"])
def test_output_pitch_not_a_multiple_of_16_bytes(dtype):
    """Odd output pitches: every output row starts at a different offset from a
    16-byte boundary (the shifted-store path), full tiles and ragged edges."""
    for (b, r, c, pi, po, pp) in [(1, 515, 300, 4, 1, 0), (2, 256, 256, 0, 3, 5),
                                  (1, 1025, 263, 9, 0, 0), (3, 130, 129, 7, 2, 1),
                                  (1, 515, 300, 4, 2, 0), (2, 256, 200, 0, 1, 3),
                                  (1, 384, 70, 0, 5, 0)]:
        x, prefill, geo = case(dtype, b, r, c, pi, po, pp, seed=r + c)
        for kw in [dict(variant=V.AUTO), dict(variant=V.TILE_VEC),
                   dict(variant=V.TILE_VEC, schedule=2)] + \
                [dict(variant=V.TILE_VEC, threads=128, tile_rows=rr, tile_cols=cc)
                 for rr, cc in VEC_128[dtype]] + \
                [dict(variant=V.TILE_VEC, tile_rows=rr, tile_cols=cc) for rr, cc in VEC_SHAPES[dtype]]:
            check(x, prefill, geo, **kw)


def test_bf16_shifted_stores_every_32_byte_offset():
    """bf16 tiles of 128 rows own output runs that start on 32-byte boundaries:
    with an odd output pitch the rows' offsets cover every residue modulo 16
    elements (heads of up to 15 elements in the first tile row), and shifting
    the output base moves them all; exact and ragged last tile rows (the
    bounds-checked path past the last full tile row), a ragged tile column and
    batched planes with a plane pitch that shifts them again."""
    for (b, r, c, po, pp) in [(1, 384, 150, 1, 0), (1, 421, 150, 3, 0), (2, 256, 136, 5, 3),
                              (1, 143, 300, 15, 0), (3, 128, 70, 9, 7)]:
        x, prefill, geo = case(U16, b, r, c, 0, po, pp, seed=r + c + po)
        for out_off in (0, 1, 5, 8, 13):
            for kw in [dict(variant=V.AUTO), dict(variant=V.TILE_VEC, tile_rows=128, tile_cols=128),
                       dict(variant=V.TILE_VEC, threads=128, tile_rows=64, tile_cols=128)]:
                check(x, prefill, geo, out_off=out_off, **kw)
            # and with the input rows misaligned too (realigned loads + shifted stores)
            check(x, prefill, geo, in_off=3, out_off=out_off, variant=V.AUTO)


def test_unsupported_vector_tile_shape_is_refused():
    x, prefill, geo = case(U32, 1, 64, 64)
    with pytest.raises(B.TransposeError) as e:
        gpu_out(x, prefill, *geo, variant=V.TILE_VEC, tile_rows=96, tile_cols=64)
    assert e.value.status == B.Status.ERR_UNSUPPORTED


def test_tma_stage_count_that_does_not_fit_is_refused():
    x, prefill, geo = case(U16, 1, 128, 128)
    with pytest.raises(B.TransposeError) as e:
        gpu_out(x, prefill, *geo, variant=V.TMA, schedule=1, stages=8)  # 10 x 32 KiB
    assert e.value.status == B.Status.ERR_UNSUPPORTED
    with pytest.raises(B.TransposeError) as e:
        gpu_out(x, prefill, *geo, variant=V.TMA, schedule=4, stages=8)  # 8 x 32 KiB
    assert e.value.status == B.Status.ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", [U32, U16], ids=["f32", "bf16"])
def test_plain_entry_points(dtype):
    x, prefill, geo = case(dtype, 1, 190, 250, 6, 10, seed=9)
    check(x, prefill, geo, entry="plain")
    x, prefill, geo = case(dtype, 3, 64, 96, 0, 0, 8, seed=10)
    check(x, prefill, geo, entry="batched")


def test_nan_payloads_survive_every_variant():
    for dtype in (U32, U16):
        sp = np.array([0x7F800001, 0x7FA00000, 0xFF800123, 0x7FC00000, 0xFFFFFFFF, 0x80000000,
                       0x00000001, 0x807FFFFF], dtype=np.uint64)
        if dtype is U16:
            sp = np.array([0x7F81, 0x7FA0, 0xFF81, 0x7FC0, 0xFFFF, 0x8000, 0x0001, 0x807F],
                          dtype=np.uint64)
        vals = np.resize(sp, 128 * 128).astype(dtype)
        x, prefill, geo = case(dtype, 1, 128, 128, values=vals)
        for kw in _variants(dtype, True):
            check(x, prefill, geo, **kw)


@pytest.mark.parametrize("variant", [dict(variant=V.TILE_PAD, pad=1), dict(variant=V.TILE_VEC),
                                     dict(variant=V.TMA), dict(variant=V.TMA, schedule=3),
                                     dict(variant=V.TMA, schedule=4)],
                         ids=["pad1", "vec", "tma", "tma_ldst", "tma_ws"])
def test_index_check_repeated(variant):
    """The exact index check run many times: a tile read before it was fully
    written fails it ("Shared memory and the bank conflict", "The barrier")."""
    import torch
    w = W.WORKLOADS["c1_index"]
    x = W.make_input(w)
    want = oracle_out(x, W.make_output(w), 1, w.rows, w.cols, w.ld_in, w.ld_out, w.sin, w.sout)
    from gpu_util import to_device
    dev_in, p_in = to_device(x)
    outs = [torch.empty(w.out_elems, dtype=torch.int32, device="cuda") for _ in range(50)]
    for o in outs:
        args = B.make_args(p_in, o.data_ptr(), B.DType.F32, 1, w.rows, w.cols, w.ld_in, w.ld_out)
        B.check(B.tr_transpose_ex(args, B.make_options(**variant)))
    torch.cuda.synchronize()
    for o in outs:
        got = o.cpu().numpy().view(np.uint32)
        assert np.array_equal(got, want), first_mismatch(got, want)


# --- the configured workloads at full size -----------------------------------------

@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_workload_full_size(name):
    w = W.WORKLOADS[name]
    x = W.make_input(w)
    prefill = W.make_output(w)
    geo = (w.batch, w.rows, w.cols, w.ld_in, w.ld_out, w.sin, w.sout)
    want = oracle_out(x, prefill, *geo)
    es = w.esize
    aligned = (w.ld_in * es % 16 == 0 and w.ld_out * es % 16 == 0)
    kws = [dict(variant=V.AUTO), dict(variant=V.TILE_VEC), dict(variant=V.TILE_VEC, schedule=2)]
    kws += [dict(variant=V.TILE_VEC, tile_rows=r, tile_cols=c)
            for r, c in VEC_SHAPES[U32 if es == 4 else U16]]
    kws += [dict(variant=V.TILE_VEC, threads=128, tile_rows=r, tile_cols=c)
            for r, c in VEC_128[U32 if es == 4 else U16]]
    kws += [dict(variant=V.TILE_VEC, threads=n, tile_rows=r, tile_cols=c)
            for n, r, c in VEC_SMALL[U32 if es == 4 else U16]]
    if aligned:
        kws += [dict(variant=V.TMA), dict(variant=V.TMA, schedule=1), dict(variant=V.TMA, schedule=3),
                dict(variant=V.TMA, schedule=4)]
    if name.startswith("c1"):
        kws += [dict(variant=V.TILE_PAD, pad=0), dict(variant=V.TILE_PAD, pad=1),
                dict(variant=V.TILE_PAD, pad=2), dict(variant=V.NAIVE_ROW),
                dict(variant=V.NAIVE_COL)]
    for kw in kws:
        got = gpu_out(x, prefill, *geo, **kw)
        assert np.array_equal(got, want), f"{name} {kw}: {first_mismatch(got, want)}"
    if name == "c1_index":
        o = want.reshape(w.cols, w.rows).view(np.float32)
        assert o[5, 7] == 7 * w.cols + 5


# --- the copy kernel -------------------------------------------------------------

def test_copy_all_alignments():
    import torch
    rng = np.random.default_rng(0)
    src_host = rng.integers(0, 256, 1 << 20, dtype=np.uint8)
    src = torch.from_numpy(src_host).cuda()
    for n in [0, 1, 15, 16, 17, 1000, 4096, 65537, (1 << 20) - 64]:
        for a_off, b_off in [(0, 0), (4, 4), (3, 3), (4, 8), (1, 2), (0, 7), (13, 13)]:
            if n + max(a_off, b_off) > src_host.size:
                continue
            dst = torch.zeros(src_host.size + 64, dtype=torch.uint8, device="cuda")
            B.check(B.tr_copy(src.data_ptr() + a_off, dst.data_ptr() + b_off, n))
            got = dst.cpu().numpy()
            assert np.array_equal(got[b_off:b_off + n], src_host[a_off:a_off + n]), (n, a_off, b_off)
            assert not got[:b_off].any() and not got[b_off + n:].any(), (n, a_off, b_off)


def test_copy_large():
    import torch
    n = 3 * (1 << 28) + 12
    src = torch.randint(0, 255, (n,), dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    B.check(B.tr_copy(src.data_ptr(), dst.data_ptr(), n))
    torch.cuda.synchronize()
    assert torch.equal(src, dst)


def test_non_default_stream():
    import torch
    x, prefill, geo = case(U32, 2, 300, 200, 4, 4, seed=4)
    s = torch.cuda.Stream()
    for v in (V.TILE_VEC, V.TMA):
        check(x, prefill, geo, variant=v, stream=s.cuda_stream)


def test_torch_convenience_wrapper():
    import torch
    x = torch.randn(3, 300, 500, device="cuda")
    y = B.transpose(x)
    assert torch.equal(y, x.transpose(1, 2))
    xb = torch.randn(777, 333, device="cuda").to(torch.bfloat16)
    assert torch.equal(B.transpose(xb), xb.t())
    big = torch.zeros(500, 310, device="cuda")
    view = big[:, :300]
    B.transpose(x[0], out=view)
    assert torch.equal(view, x[0].t()) and not big[:, 300:].any()
