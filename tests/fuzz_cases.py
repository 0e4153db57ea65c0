"""Random transpose configurations shared by the GPU sweeps (the release
library's fuzz test and the bounds-checked build's test): element type, batch,
shape, row pitches (dense, padded by a few elements -- usually breaking 16-byte
alignment -- or padded up to a 16-byte multiple), plane gaps, base-pointer
offsets and a variant with its options, each drawn from a seeded generator."""
from __future__ import annotations

import numpy as np

from shared_memory_tiled_gb300 import binding as B

V = B.Variant
U32, U16 = np.uint32, np.uint16

# (threads, tile rows, tile cols) the vector tile accepts, per element type
VEC = {U32: [(256, 64, 64), (256, 128, 32), (256, 128, 64), (256, 64, 128), (256, 128, 128),
             (128, 64, 64), (128, 32, 64), (128, 128, 64), (64, 32, 64), (64, 64, 32),
             (32, 32, 32)],
       U16: [(256, 128, 128), (256, 256, 64), (256, 256, 128), (256, 128, 256),
             (128, 128, 128), (128, 64, 128), (64, 64, 128), (64, 128, 64), (32, 64, 64)]}


def aligned(esize, off, ld, stride, batch):
    return (off * esize) % 16 == 0 and (ld * esize) % 16 == 0 and \
        (batch == 1 or (stride * esize) % 16 == 0)


def draw(rng):
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
    tma_ok = aligned(esize, in_off, ld_in, si, batch) and aligned(esize, out_off, ld_out, so, batch)
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
