"""Host-side model of the shifted stores' column ownership (tile_vec_kernel.cuh).

When output rows do not start on 16-byte boundaries, the tile at tile row tr
(input rows r0 = tr*TR ..) owns, in an output row whose first 16-byte boundary
lies d elements past r0, the output columns [r0 + d, r0 + TR + d), plus [0, d)
in the first tile row; tiles of the last, short tile row take bounds-checked
element stores and skip the first d columns.  Lane A of a micro-block row
writes the aligned chunk made of its own last V-d elements and the first d of
micro-block A+1 (the halo rows below the tile for the last lane).

The bf16 kernel gathers each aligned chunk from the shared tile instead (input
rows r0 + d + V*A .. of the output row's column), which is the same column
ownership and the same source rows.

The model below restates that rule and checks, for every row count, tile
height, element width and row offset in range, that each output column is
written exactly once and from the input row it must come from.
"""
from __future__ import annotations

import pytest


def _writes(rows, TR, V, s):
    """Output column -> source input row, as the kernel's stores produce them."""
    d = (V - s) % V
    MR = TR // V
    writes = {}

    def put(col, src):
        assert col not in writes, f"column {col} written twice"
        writes[col] = src

    for tr in range((rows + TR - 1) // TR):
        r0 = tr * TR
        if r0 + TR <= rows:                         # shifted path
            for A in range(MR):
                oc = r0 + V * A
                if d == 0:
                    for q in range(V):
                        put(oc + q, oc + q)
                    continue
                seq = [r0 + V * A + i for i in range(2 * V)]   # own rows, then lane A+1's / halo
                wc = oc + d
                for q in range(V):
                    if wc + q < rows:
                        put(wc + q, seq[d + q])
                if tr == 0 and A == 0:
                    for q in range(d):
                        put(q, seq[q])
        else:                                       # bounds-checked path
            lo = r0 + d if tr > 0 else 0
            for A in range(MR):
                oc = r0 + V * A
                for q in range(V):
                    if lo <= oc + q < rows:
                        put(oc + q, oc + q)
    return writes


@pytest.mark.parametrize("V", [4, 8])
def test_every_output_column_written_once_from_its_row(V):
    for TR in (8 * V, 16 * V, 32 * V):
        for rows in list(range(1, 2 * TR + V + 2)) + [12289, 7919]:
            for s in range(V):
                w = _writes(rows, TR, V, s)
                assert sorted(w) == list(range(rows)), (rows, TR, V, s)
                assert all(src == col for col, src in w.items()), (rows, TR, V, s)
