"""Host-side model of the aligned-chunk loads for misaligned input rows
(tile_vec_kernel.cuh).

When input rows do not start on 16-byte boundaries, a tile that lies wholly
inside the matrix (with shifted stores, its halo rows below included) reads
each of its row segments as the aligned 16-byte chunks that cover it: thread lcc the chunk holding its first element, and a helper
thread the chunk past the segment's end when the row is not aligned.  Every
thread then takes elements s .. s+V-1 of (its chunk, the next chunk: the next
lane's own by a warp shuffle, or for a row's last lane the helper's chunk staged
in shared memory), s being the row's element offset from its 16-byte boundary,
which the kernel derives
from the low 32 bits of one row address and a per-row step.  Two tiles take the
per-chunk path instead: the first tile of the first plane, and a tile in the
last plane reading the last input row whose row segments end fewer than V
elements before that row's end.

The model restates those rules and checks, over a sweep of shapes, pitches,
plane gaps and base offsets, that (1) every byte the aligned loads touch lies
inside the input's extent [in, in + extent), (2) the cut-out chunks hold the
elements they must, and (3) the 32-bit shift arithmetic gives each row's true
offset.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest

M32 = (1 << 32) - 1


def _raw_tile(g, TR, TC, V, full, b, tr, tc, halo=0):
    end = (tr + 1) * TR + halo  # one past the last row the tile reads
    first = b == 0 and tr == 0 and tc == 0
    last = b == g["batch"] - 1 and end >= g["rows"] and (tc + 1) * TC + V > g["cols"]
    return full and end <= g["rows"] and not first and not last


def _check(esize, TR, TC, RPP, batch, rows, cols, ld_in, gap, base_elems, halo):
    V = 16 // esize
    MC = TC // V
    stride = (rows - 1) * ld_in + cols + gap if batch > 1 else rows * ld_in
    extent = (batch - 1) * stride + (rows - 1) * ld_in + cols  # elements
    # memory: a 16-byte aligned arena with the input placed base_elems in;
    # every element holds its own index within the input (-1 outside)
    lead = base_elems
    arena = np.full(lead + extent + 64, -1, dtype=np.int64)
    arena[lead:lead + extent] = np.arange(extent)
    in_lo, in_hi = lead * esize, (lead + extent) * esize  # byte bounds, arena at 0
    g = dict(batch=batch, rows=rows, cols=cols)
    tiles_r, tiles_c = -(-rows // TR), -(-cols // TC)
    raw_tiles = 0
    for b, tr, tc in itertools.product(range(batch), range(tiles_r), range(tiles_c)):
        r0, c0 = tr * TR, tc * TC
        full = r0 + TR <= rows and c0 + TC <= cols
        if not _raw_tile(g, TR, TC, V, full, b, tr, tc, halo):
            continue
        raw_tiles += 1
        for lr in range(RPP):  # the tile rows one thread visits: lr, lr + RPP, ...
            a0 = ((lead + b * stride + (r0 + lr) * ld_in + c0) * esize) & M32
            step = (ld_in * RPP * esize) & M32
            for k in range(TR // RPP):
                a_row = (lead + b * stride + (r0 + lr + RPP * k) * ld_in + c0) * esize
                assert (((a0 + k * step) & M32) & 15) == a_row & 15                 # (3)
        for r in range(TR + halo):  # tile rows, then halo rows
            a_row = (lead + b * stride + (r0 + r) * ld_in + c0) * esize
            sh = (a_row & 15) // esize
            chunks = [((a_row + 16 * c) & ~15) for c in range(MC)]
            if a_row & 15:
                chunks.append((a_row + 16 * MC) & ~15)                          # helper's
            for a in chunks:
                assert in_lo <= a and a + 16 <= in_hi, (b, tr, tc, r, a - in_lo)  # (1)
            for c in range(MC):
                own = arena[chunks[c] // esize: chunks[c] // esize + V]
                nxt = (arena[chunks[c + 1] // esize: chunks[c + 1] // esize + V]
                       if c + 1 < len(chunks) else np.zeros(V, np.int64))
                got = np.concatenate([own, nxt])[sh: sh + V]
                first = b * stride + (r0 + r) * ld_in + c0 + c * V
                assert np.array_equal(got, np.arange(first, first + V)), (b, tr, tc, r, c)  # (2)
    return raw_tiles


@pytest.mark.parametrize("halo", [False, True], ids=["aligned-output", "shifted-stores"])
@pytest.mark.parametrize("esize", [4, 2])
def test_aligned_chunk_loads_stay_inside_the_input(esize, halo):
    V = 16 // esize
    total_raw = 0
    for TR, TC, RPP in [(8 * V, 8 * V, 4), (16 * V, 8 * V, 8), (8 * V, 16 * V, 16)]:
        for rows in (TR, 2 * TR + 3):
            for cols in (TC, TC + 1, TC + V - 1, TC + V, 2 * TC):
                for ld_in in (cols, cols + 1, cols + V + 3):
                    for batch, gap in ((1, 0), (2, 0), (3, 5)):
                        for base in range(V):
                            total_raw += _check(esize, TR, TC, RPP, batch, rows, cols, ld_in, gap,
                                                base, V if halo else 0)
    assert total_raw > 0


def test_the_exclusions_are_needed():
    """Without the two exclusions the rule would read outside the input: the
    first tile's first chunk starts before it, and the last row's helper chunk
    runs past its end when the segment ends within V elements of it."""
    esize, V, TR, TC = 4, 4, 32, 32
    # base one element past a boundary; the last row starts one element past one too
    lead, rows, cols, ld_in = 1, 2 * TR, TC + 1, TC + 4
    in_lo = lead * esize
    assert ((lead * esize) & ~15) < in_lo                       # first chunk, first tile
    extent = (rows - 1) * ld_in + cols
    in_hi = (lead + extent) * esize
    a_row = (lead + (rows - 1) * ld_in) * esize                 # last row, tile column 0
    helper = (a_row + 16 * (TC // V)) & ~15
    assert a_row & 15 and helper + 16 > in_hi                   # reaches past the input
    g = dict(batch=1, rows=rows, cols=cols)
    assert not _raw_tile(g, TR, TC, V, True, 0, 0, 0)           # excluded: first tile
    assert not _raw_tile(g, TR, TC, V, True, 0, 1, 0)           # excluded: holds the last row
    assert _raw_tile(dict(g, cols=TC + V), TR, TC, V, True, 0, 1, 0)  # V columns to spare
