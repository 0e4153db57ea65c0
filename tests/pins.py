"""Checks that pin a transpose implementation to facts fixed outside itself.

Each check takes ``fn(x, out, batch, rows, cols, ld_in, ld_out, stride_in,
stride_out)``, which must write the transpose of ``x`` into ``out`` (flat numpy
arrays of uint32 or uint16 bit patterns), and raises ``AssertionError`` when the
implementation disagrees with:

* hand-written worked examples (``tests/golden``);
* the closed form of the exact index check: with every input element holding
  its own linear index, output plane b, row j, column i holds
  ``b*rows*cols + i*cols + j`` ("Shared memory and the bank conflict",
  section "The barrier");
* numpy's own transpose of the dense special case (a library routine);
* involution: transposing twice gives the input back, bit for bit;
* permutation: the multiset of logical bit patterns is unchanged;
* sentinels: output pitch padding keeps its prefill and no input padding
  element reaches the output ("Shared-memory tiling and bank conflicts",
  "Worked example": padding never changes the logical contents);
* brute force: an element-by-element dictionary of where each input element
  must land, on tiny shapes;
* bit transparency: NaN payloads (signalling included), signed zeros and
  subnormals survive unchanged.

The same checks are run against deliberately wrong implementations in the
oracle tests, to show that each plausible mistake trips at least one of them.
"""
from __future__ import annotations

import itertools

import numpy as np

import golden_io

U32, U16 = np.uint32, np.uint16
PAD_IN = {U32: U32(0x7FC0DEAD), U16: U16(0x7FAD)}
PAD_OUT = {U32: U32(0xFFC0BEEF), U16: U16(0xFFBE)}


def _extent(batch, rows, cols, ld, stride):
    return 0 if 0 in (batch, rows, cols) else (batch - 1) * stride + (rows - 1) * ld + cols


def alloc_case(dtype, batch, rows, cols, ld_in=None, ld_out=None, stride_in=None,
               stride_out=None, values=None, seed=0):
    """Input filled with ``values`` (or random bits) in its logical region and the
    input sentinel elsewhere; output prefilled with the output sentinel."""
    ld_in = cols if ld_in is None else ld_in
    ld_out = rows if ld_out is None else ld_out
    stride_in = rows * ld_in if stride_in is None else stride_in
    stride_out = cols * ld_out if stride_out is None else stride_out
    n_in = max(batch * stride_in, _extent(batch, rows, cols, ld_in, stride_in))
    n_out = max(batch * stride_out, _extent(batch, cols, rows, ld_out, stride_out))
    x = np.full(n_in, PAD_IN[dtype], dtype=dtype)
    out = np.full(n_out, PAD_OUT[dtype], dtype=dtype)
    if values is None:
        rng = np.random.default_rng(seed)
        hi = 1 << (32 if dtype is U32 else 16)
        values = rng.integers(0, hi, batch * rows * cols, dtype=np.uint64).astype(dtype)
    logical_view(x, batch, rows, cols, ld_in, stride_in)[...] = \
        np.asarray(values, dtype=dtype).reshape(batch, rows, cols)
    return x, out, dict(batch=batch, rows=rows, cols=cols, ld_in=ld_in, ld_out=ld_out,
                        stride_in=stride_in, stride_out=stride_out)


def logical_view(buf, batch, rows, cols, ld, stride):
    """Strided (batch, rows, cols) view of the logical elements of a flat buffer."""
    if 0 in (batch, rows, cols):
        return np.zeros((batch, rows, cols), dtype=buf.dtype)
    it = buf.itemsize
    return np.lib.stride_tricks.as_strided(buf, shape=(batch, rows, cols),
                                           strides=(stride * it, ld * it, it))


def logical_mask(n, batch, rows, cols, ld, stride):
    mask = np.zeros(n, dtype=bool)
    logical_view(mask, batch, rows, cols, ld, stride)[...] = True
    return mask


def run(fn, x, out, p):
    fn(x, out, p["batch"], p["rows"], p["cols"], p["ld_in"], p["ld_out"],
       p["stride_in"], p["stride_out"])
    return out


def out_logical(out, p):
    return logical_view(out, p["batch"], p["cols"], p["rows"], p["ld_out"], p["stride_out"])


# ---------------------------------------------------------------------------

def check_golden(fn):
    for path in golden_io.transpose_fixtures():
        for dt in (U32, U16):
            p, x, want = golden_io.fixture_arrays(path, dt, PAD_IN[dt], PAD_OUT[dt])
            out = np.full(want.size, PAD_OUT[dt], dtype=dt)
            run(fn, x, out, p)
            assert np.array_equal(out, want), f"golden {path} ({dt.__name__})"


INDEX_SHAPES = [
    # batch, rows, cols, ld_in, ld_out, stride_in, stride_out
    (1, 1, 1, 1, 1, None, None),
    (1, 1, 37, 40, 1, None, None),
    (1, 37, 1, 1, 40, None, None),
    (1, 33, 65, 70, 40, None, None),
    (3, 17, 9, 11, 20, 17 * 11 + 5, 9 * 20 + 3),
    (2, 64, 48, 48, 64, None, None),
    (1, 1024, 1024, 1024, 1024, None, None),
]


def check_index_closed_form(fn):
    for (b, r, c, li, lo, si, so) in INDEX_SHAPES:
        n = b * r * c
        x, out, p = alloc_case(U32, b, r, c, li, lo, si, so, values=np.arange(n, dtype=U32))
        run(fn, x, out, p)
        bb, jj, ii = np.indices((b, c, r), dtype=np.int64)
        want = (bb * r * c + ii * c + jj).astype(U32)
        assert np.array_equal(out_logical(out, p), want), f"index closed form {p}"


def check_numpy_transpose(fn):
    for dt in (U32, U16):
        for (b, r, c, li, lo) in [(1, 31, 45, 45, 31), (1, 64, 96, 100, 70), (4, 10, 7, 9, 12),
                                  (2, 128, 3, 3, 128)]:
            x, out, p = alloc_case(dt, b, r, c, li, lo, seed=r * 1000 + c)
            run(fn, x, out, p)
            src = np.array(logical_view(x, b, r, c, li, p["stride_in"]))
            want = np.ascontiguousarray(src.transpose(0, 2, 1))
            assert np.array_equal(out_logical(out, p), want), f"numpy transpose {p} {dt.__name__}"


def check_involution(fn, cases=None):
    cases = cases or [(U32, 1, 45, 77, 80, 50), (U16, 3, 19, 64, 70, 21), (U32, 2, 128, 128, 128, 128)]
    for (dt, b, r, c, li, lo) in cases:
        x, out, p = alloc_case(dt, b, r, c, li, lo, seed=7 + r)
        run(fn, x, out, p)
        back = np.full(x.size, PAD_IN[dt], dtype=dt)
        q = dict(batch=b, rows=c, cols=r, ld_in=lo, ld_out=li, stride_in=p["stride_out"],
                 stride_out=p["stride_in"])
        run(fn, out, back, q)
        assert np.array_equal(back, x), f"involution {p}"


def check_permutation(fn):
    for dt in (U32, U16):
        x, out, p = alloc_case(dt, 2, 37, 53, 60, 40, seed=11)
        run(fn, x, out, p)
        a = np.sort(np.array(logical_view(x, 2, 37, 53, 60, p["stride_in"])).ravel())
        o = np.sort(np.array(out_logical(out, p)).ravel())
        assert np.array_equal(a, o), f"permutation {p}"


def check_sentinels(fn):
    for dt in (U32, U16):
        b, r, c, li, lo = 2, 23, 41, 48, 29
        # Values drawn below the sentinels' exponent field: never equal to them.
        rng = np.random.default_rng(5)
        hi = 0x7F000000 if dt is U32 else 0x7F00
        vals = rng.integers(0, hi, b * r * c, dtype=np.uint64).astype(dt)
        x, out, p = alloc_case(dt, b, r, c, li, lo, stride_in=r * li + 9, stride_out=c * lo + 4,
                               values=vals)
        run(fn, x, out, p)
        m = logical_mask(out.size, b, c, r, lo, p["stride_out"])
        assert np.all(out[~m] == PAD_OUT[dt]), "output padding was written"
        assert not np.any(out[m] == PAD_IN[dt]), "input padding reached the output"
        assert not np.any(out[m] == PAD_OUT[dt]), "a logical output element was not written"


def check_brute_force(fn, dims=range(1, 9), pads=(0, 1, 5), batches=(1, 3)):
    for dt in (U32, U16):
        for r, c, pad, b in itertools.product(dims, dims, pads, batches):
            li, lo = c + pad, r + pad
            si, so = r * li + pad, c * lo + pad
            x, out, p = alloc_case(dt, b, r, c, li, lo, si, so,
                                   values=np.arange(1, b * r * c + 1, dtype=dt))
            want = out.copy()
            for bb in range(b):
                for i in range(r):
                    for j in range(c):
                        want[bb * so + j * lo + i] = x[bb * si + i * li + j]
            run(fn, x, out, p)
            assert np.array_equal(out, want), f"brute force {p} {dt.__name__}"


def check_bit_transparency(fn):
    specials32 = np.array([0x7F800001, 0x7FA00000, 0xFF800123, 0x7FC00000, 0xFFFFFFFF,
                           0x80000000, 0x00000000, 0x00000001, 0x807FFFFF, 0x7F800000,
                           0xFF800000, 0x7FBFFFFF], dtype=U32)
    specials16 = np.array([0x7F81, 0x7FA0, 0xFF81, 0x7FC0, 0xFFFF, 0x8000, 0x0000, 0x0001,
                           0x807F, 0x7F80, 0xFF80, 0x7FBF], dtype=U16)
    for dt, sp in ((U32, specials32), (U16, specials16)):
        r, c = 6, 8
        vals = np.resize(sp, r * c)
        x, out, p = alloc_case(dt, 1, r, c, c + 3, r + 2, values=vals)
        run(fn, x, out, p)
        want = vals.reshape(r, c).T
        assert np.array_equal(out_logical(out, p)[0], want), f"bit patterns changed ({dt.__name__})"


ALL_CHECKS = [check_golden, check_index_closed_form, check_numpy_transpose, check_involution,
              check_permutation, check_sentinels, check_brute_force, check_bit_transparency]
