"""Host-side model of the shifted stores' column ownership (tile_vec_kernel.cuh).

When output rows do not start on aligned boundaries, the tile at tile row tr
(input rows r0 = tr*TR ..) owns, in an output row whose first boundary of the
shift granule G lies d elements past r0, the output columns
[r0 + d, r0 + TR + d), plus [0, d) in the first tile row; tiles of the last,
short tile row take bounds-checked element stores and skip the first d
columns.  G is one 16-byte chunk for fp32 (V = 4) and for bf16 tiles shorter
than 128 rows, and two chunks for bf16 tiles of 128 rows or more (V = 8, so
that 8 consecutive chunks cover whole 32-byte sectors).  fp32: lane A of a
micro-block row writes the aligned chunk made of its own last V-d elements and
the first d of micro-block A+1 (the halo rows below the tile for the last
lane).  bf16: each lane gathers the chunk at r0 + d + V*A from the shared tile,
input rows r0 + d + V*A .. of the output row's column, the G halo rows below
the tile supplying the rows past it.

The model below restates that rule and checks, for every row count, tile
height, element width and row offset in range, that each output column is
written exactly once, from the input row it must come from, and that no tile
reads past its halo.
"""
from __future__ import annotations

import pytest


def _granule(TR, V):
    return 2 * V if V == 8 and TR >= 128 else V


def _writes(rows, TR, V, s):
    """Output column -> source input row, as the kernel's stores produce them."""
    G = _granule(TR, V)
    d = (G - s) % G
    MR = TR // V
    writes = {}

    def put(col, src, r0):
        assert col not in writes, f"column {col} written twice"
        assert src < r0 + TR + G, "read past the halo"
        writes[col] = src

    for tr in range((rows + TR - 1) // TR):
        r0 = tr * TR
        if r0 + TR <= rows:                         # shifted path
            for A in range(MR):
                wc = r0 + V * A + d                 # first column of the aligned chunk
                for q in range(V):
                    if wc + q < rows:
                        put(wc + q, r0 + d + V * A + q, r0)
                if tr == 0 and A == 0:
                    for q in range(d):
                        put(q, q, r0)
        else:                                       # bounds-checked path
            lo = r0 + d if tr > 0 else 0
            for A in range(MR):
                oc = r0 + V * A
                for q in range(V):
                    if lo <= oc + q < rows:
                        put(oc + q, oc + q, r0)
    return writes


@pytest.mark.parametrize("V", [4, 8])
def test_every_output_column_written_once_from_its_row(V):
    for TR in (8 * V, 16 * V, 32 * V):
        G = _granule(TR, V)
        for rows in list(range(1, 2 * TR + G + 2)) + [12289, 7919]:
            for s in range(G):
                w = _writes(rows, TR, V, s)
                assert sorted(w) == list(range(rows)), (rows, TR, V, s)
                assert all(src == col for col, src in w.items()), (rows, TR, V, s)
