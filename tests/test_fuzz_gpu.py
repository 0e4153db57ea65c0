"""Seeded random sweep of transpose configurations against the oracle.

Each case draws an element type, a batch count, a shape, row pitches (dense,
padded by a few elements -- usually breaking 16-byte alignment -- or padded up
to a 16-byte multiple), plane gaps, base-pointer offsets and a variant with its
options, and compares the whole output buffer with the oracle bit for bit
(pitch padding and plane gaps included: they must keep their prefill)."""
from __future__ import annotations

import numpy as np
import pytest

import pins
from gpu_util import first_mismatch, gpu_out, oracle_out
from shared_memory_tiled_gb300 import binding as B

pytestmark = pytest.mark.gpu

V = B.Variant
U32, U16 = np.uint32, np.uint16

# (threads, tile rows, tile cols) the vector tile accepts, per element type
VEC = {U32: [(256, 64, 64), (256, 128, 32), (256, 128, 64), (256, 64, 128), (256, 128, 128),
             (128, 64, 64), (128, 32, 64), (128, 128, 64), (64, 32, 64), (64, 64, 32),
             (32, 32, 32)],
       U16: [(256, 128, 128), (256, 256, 64), (256, 256, 128), (256, 128, 256),
             (128, 128, 128), (128, 64, 128), (64, 64, 128), (64, 128, 64), (32, 64, 64)]}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()
    yield
    assert B.tr_device_status() == B.Status.OK, "a bounded in-kernel wait ran out"


def _aligned(esize, off, ld, stride, batch):
    return (off * esize) % 16 == 0 and (ld * esize) % 16 == 0 and \
        (batch == 1 or (stride * esize) % 16 == 0)


def _draw(rng):
    dtype = U32 if rng.random() < 0.5 else U16
    esize, vec = (4, 4) if dtype is U32 else (2, 8)
    batch = int(rng.choice([1, 1, 1, 2, 3]))
    rows, cols = int(rng.integers(1, 700)), int(rng.integers(1, 700))

    def pitch(n):
        c = rng.random()
        if c < 0.4:
            return n
        if c < 0.75:
            return n + int(rng.integers(1, 9))
        return n + (-n) % vec + vec * int(rng.integers(0, 3))

    ld_in, ld_out = pitch(cols), pitch(rows)
    gap = int(rng.integers(0, 17)) if batch > 1 else 0
    si, so = rows * ld_in + gap, cols * ld_out + gap
    in_off = int(rng.choice([0, 0, 0, 1, 3]))
    out_off = int(rng.choice([0, 0, 0, 1, 2]))
    tma_ok = _aligned(esize, in_off, ld_in, si, batch) and _aligned(esize, out_off, ld_out, so, batch)
    kinds = ["auto", "vec", "vec", "pad", "naive"] + (["tma"] * 3 if tma_ok else [])
    kind = str(rng.choice(kinds))
    if kind == "auto":
        opt = dict(variant=V.AUTO)
    elif kind == "vec":
        nt, tr, tc = VEC[dtype][int(rng.integers(len(VEC[dtype])))]
        opt = dict(variant=V.TILE_VEC, threads=nt, tile_rows=tr, tile_cols=tc,
                   tile_order=int(rng.integers(0, 2)))
        if nt == 256 and rng.random() < 0.25:
            opt["schedule"] = 2
    elif kind == "pad":
        opt = dict(variant=V.TILE_PAD, pad=int(rng.choice([0, 1, 2, 3, 4, 8])))
    elif kind == "naive":
        opt = dict(variant=V.NAIVE_ROW if rng.random() < 0.5 else V.NAIVE_COL)
    else:
        sched = int(rng.integers(0, 5))
        opt = dict(variant=V.TMA, schedule=sched, tile_order=int(rng.integers(0, 2)))
        if sched in (0, 2):
            opt["stages"] = int(rng.integers(2, 7 if dtype is U32 else 5))
        elif sched == 1:
            opt["stages"] = int(rng.integers(2, 5))
        elif sched == 3:
            opt["stages"] = int(rng.integers(2, 9 if dtype is U32 else 7))
        else:
            opt["stages"] = int(rng.integers(2, 9 if dtype is U32 else 7))
    return dtype, (batch, rows, cols, ld_in, ld_out, si, so), in_off, out_off, opt


@pytest.mark.parametrize("seed", range(6))
def test_random_configurations(seed):
    rng = np.random.default_rng(1000 + seed)
    for k in range(150):
        dtype, geo, in_off, out_off, opt = _draw(rng)
        batch, rows, cols, ld_in, ld_out, si, so = geo
        x, prefill, _ = pins.alloc_case(dtype, batch, rows, cols, ld_in, ld_out, si, so,
                                        seed=int(rng.integers(1 << 30)))
        want = oracle_out(x, prefill, *geo)
        got = gpu_out(x, prefill, *geo, in_off=in_off, out_off=out_off, **opt)
        assert np.array_equal(got, want), \
            f"case {k}: {np.dtype(dtype).name} {geo} offsets {in_off}/{out_off} {opt}: " \
            f"{first_mismatch(got, want)}"


@pytest.mark.parametrize("seed", range(3))
def test_random_inplace_configurations(seed):
    """The in-place square transpose over random sizes, pitches, plane gaps and
    base offsets, against the oracle's pairwise swaps."""
    import oracle
    import torch
    from gpu_util import from_device, to_device
    rng = np.random.default_rng(2000 + seed)
    for k in range(60):
        dt = U32 if rng.random() < 0.5 else U16
        vec = 4 if dt is U32 else 8
        batch = int(rng.choice([1, 1, 2, 3]))
        n = int(rng.integers(1, 600))
        c = rng.random()
        ld = n if c < 0.4 else n + int(rng.integers(1, 9)) if c < 0.75 else n + (-n) % vec
        stride = n * ld + (int(rng.integers(0, 17)) if batch > 1 else 0)
        off = int(rng.choice([0, 0, 1, 3]))
        x = rng.integers(0, np.iinfo(dt).max, batch * stride, dtype=dt, endpoint=True)
        want = oracle.transpose_inplace(x.copy(), batch=batch, n=n, ld=ld, stride=stride)
        buf, ptr = to_device(x, off)
        f = B.tr_transpose_inplace_f32 if dt is U32 else B.tr_transpose_inplace_bf16
        B.check(f(ptr, batch, n, ld, stride))
        torch.cuda.synchronize()
        got = from_device(buf, x.size, off, dt)
        assert np.array_equal(got, want), \
            f"case {k}: {np.dtype(dt).name} batch {batch} n {n} ld {ld} stride {stride} " \
            f"offset {off}: {first_mismatch(got, want)}"
