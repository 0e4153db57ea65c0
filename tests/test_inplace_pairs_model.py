"""Host-side model of the in-place kernel's walk over tile pairs (inplace.cu).

Blocks walk the pairs (ti <= tj) of each plane's upper triangle of T x T tiles,
T (T + 1) / 2 per plane, pair index p = tj (tj + 1) / 2 + ti.  Block w splits
into plane b = w / pairs and p = w - b * pairs, and p into (ti, tj) through the
root of x (x + 1) / 2 = p taken in float (sqrtf, correctly rounded as the
library is built without fast math), then corrected: by one step up or down
in 32-bit arithmetic when the launch holds at most 2^32 - 1 pairs, by as many
steps as it takes in 64-bit arithmetic otherwise.  The model restates those
formulas with numpy float32 rounding at every step and checks, over a sweep of
tile counts (exhaustively) and near the top of the 32-bit range (sampled),
that every pair of every plane is taken exactly once, that the 32-bit
triangular numbers never wrap, and that the float root is within the 0.02
the single correction step relies on.
"""
from __future__ import annotations

import numpy as np
import pytest

M32 = (1 << 32) - 1
F = np.float32


def float_root(p):
    """The kernel's (sqrtf(8.0f * float(p) + 1.0f) - 1.0f) * 0.5f, elementwise."""
    p = np.asarray(p)
    x = p.astype(np.float32)                       # float(p): round to nearest
    return ((np.sqrt(F(8.0) * x + F(1.0)) - F(1.0)) * F(0.5)).astype(np.float32)


def triangle32(n):
    """The kernel's triangle32 on uint32 values (wrapping like the hardware)."""
    n = np.asarray(n, dtype=np.uint64)
    odd = (n & 1) == 1
    r = np.where(odd, n * ((n + 1) >> 1), (n >> 1) * (n + 1))
    return (r & M32).astype(np.uint64)


def split_pair32(p):
    p = np.asarray(p, dtype=np.uint64)
    tj = float_root(p).astype(np.uint64)           # truncation toward zero
    tj = tj - (triangle32(tj) > p).astype(np.uint64)
    tj = tj + (triangle32(tj + 1) <= p).astype(np.uint64)
    return p - triangle32(tj), tj


def split_pair64(p):
    tj = int(float_root(p))
    while tj > 0 and tj * (tj + 1) // 2 > p:
        tj -= 1
    while (tj + 1) * (tj + 2) // 2 <= p:
        tj += 1
    return p - tj * (tj + 1) // 2, tj


@pytest.mark.parametrize("batch", [1, 2, 5])
def test_each_tile_pair_is_taken_once(batch):
    for tiles in list(range(1, 40)) + [64, 129, 256, 725]:
        pairs = tiles * (tiles + 1) // 2
        w = np.arange(batch * pairs, dtype=np.uint64)
        b = w // pairs                             # 32-bit division in the kernel
        ti, tj = split_pair32(w - b * pairs)
        assert np.all(ti <= tj) and np.all(tj < tiles)
        keys = set(zip(b.tolist(), ti.tolist(), tj.tolist()))
        assert len(keys) == batch * pairs
        want = {(bb, i, j) for bb in range(batch) for i in range(tiles) for j in range(i, tiles)}
        assert keys == want


def test_32_bit_path_exhaustive_to_two_thousand_tiles():
    tiles = 2048
    p = np.arange(tiles * (tiles + 1) // 2, dtype=np.uint64)
    ti, tj = split_pair32(p)
    assert np.array_equal(tj * (tj + 1) // 2 + ti, p)
    assert np.all(ti <= tj)


def test_32_bit_path_at_the_top_of_its_range():
    """92681 tiles per side is the largest plane whose pairs fit 32 bits: the
    triangular numbers compared with p stay below 2^32, the float root stays
    within 0.02 of the true one, and the split is exact."""
    tiles = 92681
    pairs = tiles * (tiles + 1) // 2
    assert pairs <= M32 < (tiles + 1) * (tiles + 2) // 2
    assert tiles * (tiles + 1) // 2 <= M32       # triangle32(tj + 1) with tj + 1 <= tiles
    rng = np.random.default_rng(5)
    edges = []
    for j in (0, 1, 2, 1000, 46340, 65535, 92679, 92680):
        t0 = j * (j + 1) // 2
        edges += [t0, t0 + j] + ([t0 - 1] if t0 else [])
    p = np.concatenate([np.array(edges, dtype=np.uint64),
                        rng.integers(0, pairs, 400000, dtype=np.uint64)])
    ti, tj = split_pair32(p)
    assert np.array_equal(tj * (tj + 1) // 2 + ti, p)
    assert np.all(ti <= tj) and np.all(tj < tiles)
    exact = (np.sqrt(8.0 * p.astype(np.float64) + 1.0) - 1.0) * 0.5
    assert np.max(np.abs(float_root(p).astype(np.float64) - exact)) < 0.02


def test_64_bit_path_agrees_and_reaches_past_32_bits():
    rng = np.random.default_rng(6)
    for tiles in (1, 2, 7, 129, 92682, 1 << 20):
        pairs = tiles * (tiles + 1) // 2
        for p in [0, pairs - 1] + [int(v) for v in rng.integers(0, pairs, 2000)]:
            ti, tj = split_pair64(p)
            assert 0 <= ti <= tj < tiles and tj * (tj + 1) // 2 + ti == p
            if pairs <= M32:
                ti32, tj32 = split_pair32(np.array([p], dtype=np.uint64))
                assert (int(ti32[0]), int(tj32[0])) == (ti, tj)
