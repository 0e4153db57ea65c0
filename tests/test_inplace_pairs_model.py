"""Host-side model of the in-place kernel's walk over tile pairs (inplace.cu).

Blocks walk a batch x T x T grid of tile coordinates; linear index w splits
into plane b and tile (ti, tj) by integer division, with 32-bit division when
the whole grid fits in 32 bits, and a block skips ti > tj because the pair is
handled at (tj, ti).  The model restates both divisions and checks, over a
sweep of batch counts and tile counts, that they agree and that every
unordered pair of tiles of every plane, diagonal tiles included, is taken
exactly once.
"""
from __future__ import annotations

import pytest

M32 = (1 << 32) - 1


def _split64(w, tiles):
    per_plane = tiles * tiles
    b = w // per_plane
    rem = w - b * per_plane
    ti = rem // tiles
    return b, ti, rem - ti * tiles


def _split32(w, tiles):
    w32, pp, t32 = w & M32, (tiles * tiles) & M32, tiles & M32
    bb = w32 // pp
    rem = (w32 - bb * pp) & M32
    i = rem // t32
    return bb, i, (rem - i * t32) & M32


@pytest.mark.parametrize("batch", [1, 2, 5])
def test_each_tile_pair_is_taken_once(batch):
    for tiles in list(range(1, 40)) + [64, 129]:
        total = batch * tiles * tiles
        seen = set()
        for w in range(total):
            b, ti, tj = _split64(w, tiles)
            assert _split32(w, tiles) == (b, ti, tj)
            if ti > tj:
                continue
            key = (b, ti, tj)
            assert key not in seen
            seen.add(key)
        want = {(b, i, j) for b in range(batch) for i in range(tiles) for j in range(i, tiles)}
        assert seen == want


def test_32_bit_split_at_the_edge_of_its_range():
    """The largest grids the 32-bit path takes: indices near 2**32 - 1 split
    the same way in 32 and 64 bits."""
    for tiles in (65535, 46341, 1 << 15):
        batch = M32 // (tiles * tiles)
        total = batch * tiles * tiles
        assert 0 < total <= M32
        for w in (0, 1, tiles - 1, tiles, total // 2, total - tiles, total - 1):
            assert _split32(w, tiles) == _split64(w, tiles)
