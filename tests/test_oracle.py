"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import pins
from shared_memory_tiled_gb300 import workloads as W


def oracle_fn(form):
    def fn(x, out, batch, rows, cols, ld_in, ld_out, stride_in, stride_out):
        oracle.transpose(x, out, batch=batch, rows=rows, cols=cols, ld_in=ld_in,
                         ld_out=ld_out, stride_in=stride_in, stride_out=stride_out, form=form)
    return fn


@pytest.mark.parametrize("form", ["gather", "scatter"])
@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pinned(form, check):
    check(oracle_fn(form))


def test_brute_force_ragged_shapes():
    """Wider brute force: every rows, cols in 1..70 in steps that cross 32 and 64."""
    dims = list(range(1, 12)) + [15, 16, 17, 31, 32, 33, 47, 63, 64, 65, 70]
    pins.check_brute_force(oracle_fn("gather"), dims=dims, pads=(0, 3), batches=(1,))


# --- each plausible mistake trips at least one pin --------------------------------

def _python_transpose(x, out, batch, rows, cols, ld_in, ld_out, stride_in, stride_out,
                      mistake=None):
    """Element loop with one planted mistake; the oracle itself is never edited."""
    for b in range(batch):
        for i in range(rows):
            for j in range(cols):
                if mistake == "drop_last_col" and j == cols - 1 and cols > 1:
                    continue
                src = b * stride_in + i * (cols if mistake == "dense_input_pitch" else ld_in) + j
                if mistake == "no_transpose":
                    dst = b * stride_out + i * ld_out + j
                elif mistake == "swapped_pitches":
                    src = b * stride_in + i * ld_out + j
                    dst = b * stride_out + j * ld_in + i
                elif mistake == "ignore_plane_stride_out":
                    dst = j * ld_out + i
                else:
                    dst = b * stride_out + j * ld_out + i
                if not (0 <= src < x.size and 0 <= dst < out.size):
                    continue
                v = x[src]
                if mistake == "quiet_nan":
                    # Routing the bits through a float register can quiet a
                    # signalling NaN: emulate exactly that side effect.
                    if x.dtype == np.uint32 and (v & 0x7F800000) == 0x7F800000 and (v & 0x7FFFFF):
                        v = v | np.uint32(0x400000)
                    if x.dtype == np.uint16 and (v & 0x7F80) == 0x7F80 and (v & 0x7F):
                        v = v | np.uint16(0x40)
                out[dst] = v
        if mistake == "write_whole_pitch":
            for j in range(cols):
                for i in range(rows, ld_out):
                    k = b * stride_out + j * ld_out + i
                    if k < out.size:
                        out[k] = 0


MISTAKES = ["no_transpose", "swapped_pitches", "dense_input_pitch", "drop_last_col",
            "ignore_plane_stride_out", "write_whole_pitch", "quiet_nan"]
# Checks cheap enough for a Python element loop.
FAST_CHECKS = [pins.check_golden, pins.check_numpy_transpose, pins.check_involution,
               pins.check_permutation, pins.check_sentinels, pins.check_bit_transparency,
               lambda fn: pins.check_brute_force(fn, dims=range(1, 5), pads=(0, 2), batches=(1, 2))]


def test_python_reference_loop_passes():
    """The unmutated Python loop passes the same checks the mutants must fail."""
    fn = lambda *a: _python_transpose(*a)
    for check in FAST_CHECKS:
        check(fn)


@pytest.mark.parametrize("mistake", MISTAKES)
def test_planted_mistake_is_caught(mistake):
    fn = lambda *a: _python_transpose(*a, mistake=mistake)
    caught = []
    for check in FAST_CHECKS:
        try:
            check(fn)
        except AssertionError:
            caught.append(check)
    assert caught, f"no pin caught the planted mistake {mistake!r}"


# --- the full-size workloads ---------------------------------------------------------

@pytest.mark.parametrize("name", ["c1_index", "c1_uniform", "c2", "c3", "c4", "c5"])
def test_workload_involution_and_invariants(name):
    """Transposing twice restores every configured input bit for bit; the first
    pass writes every logical output element and no padding."""
    w = W.WORKLOADS[name]
    x = W.make_input(w)
    out = W.make_output(w)
    kw = dict(batch=w.batch, rows=w.rows, cols=w.cols, ld_in=w.ld_in, ld_out=w.ld_out,
              stride_in=w.sin, stride_out=w.sout)
    oracle.transpose(x, out, **kw)
    if w.ld_out == w.rows:
        # dense output: every element written; the output sentinel cannot survive
        # unless the data hold it (only random 16-bit patterns can).
        if w.dist != "bits":
            assert not np.any(out == W.OUT_PAD_U32)
    back = np.full_like(x, W.IN_PAD_U32 if x.dtype == np.uint32 else W.IN_PAD_U16)
    oracle.transpose(out, back, batch=w.batch, rows=w.cols, cols=w.rows, ld_in=w.ld_out,
                     ld_out=w.ld_in, stride_in=w.sout, stride_out=w.sin)
    assert np.array_equal(back, x)
    if name == "c1_index":
        o = out.reshape(w.cols, w.rows)
        i = np.arange(w.rows)[None, :]
        j = np.arange(w.cols)[:, None]
        assert np.array_equal(o.view(np.float32), (i * w.cols + j).astype(np.float32))


def test_copy_oracle():
    x = np.random.default_rng(3).integers(0, 256, 1000, dtype=np.uint8)
    out = np.zeros_like(x)
    oracle.copy_bytes(x, out)
    assert np.array_equal(x, out)


def test_oracle_rejects_bad_sizes():
    x = np.zeros(10, dtype=np.uint32)
    with pytest.raises(ValueError):
        oracle.transpose(x, np.zeros(10, dtype=np.uint32), rows=3, cols=4)
    with pytest.raises(TypeError):
        oracle.transpose(x.view(np.float32), np.zeros(10, np.float32), rows=2, cols=5)


# --- in-place transpose ----------------------------------------------------------------

import golden_io  # noqa: E402


def test_inplace_golden():
    for path in golden_io.inplace_fixtures():
        for dt in (np.uint32, np.uint16):
            p, x, want = golden_io.fixture_arrays(path, dt, pins.PAD_IN[dt], pins.PAD_IN[dt])
            oracle.transpose_inplace(x, batch=p["batch"], n=p["rows"], ld=p["ld_in"],
                                     stride=p["stride_in"])
            assert np.array_equal(x, want), path


@pytest.mark.parametrize("dt", [np.uint32, np.uint16])
def test_inplace_matches_out_of_place_and_is_an_involution(dt):
    rng = np.random.default_rng(1)
    for batch, n, pad, ppad in [(1, 1, 0, 0), (1, 7, 0, 0), (2, 33, 3, 5), (3, 64, 0, 0),
                                (1, 130, 6, 0), (2, 257, 1, 3)]:
        ld, stride = n + pad, n * (n + pad) + ppad
        size = (batch - 1) * stride + (n - 1) * ld + n if n else 0
        x = rng.integers(0, np.iinfo(dt).max, size, dtype=dt, endpoint=True)
        want = x.copy()
        oracle.transpose(x, want, batch=batch, rows=n, cols=n, ld_in=ld, ld_out=ld,
                         stride_in=stride, stride_out=stride)
        got = x.copy()
        oracle.transpose_inplace(got, batch=batch, n=n, ld=ld, stride=stride)
        assert np.array_equal(got, want)
        oracle.transpose_inplace(got, batch=batch, n=n, ld=ld, stride=stride)
        assert np.array_equal(got, x)


def test_inplace_brute_force_tiny():
    for n in range(0, 7):
        for pad in (0, 2):
            ld = n + pad
            size = max(0, (n - 1) * ld + n)
            x = np.arange(size, dtype=np.uint32)
            got = x.copy()
            oracle.transpose_inplace(got, n=n, ld=ld)
            want = x.copy()
            for i in range(n):
                for j in range(n):
                    want[j * ld + i] = x[i * ld + j]
            assert np.array_equal(got, want)


# --- transposed operand tiles ("Padded Shared Memory", the As store) ---------------------

@pytest.mark.parametrize("bm,bk", [(128, 16), (128, 8), (64, 32), (2, 4)])
def test_operand_tiles_match_numpy_blocked_transpose(bm, bk):
    m, k, lda = 2 * bm, 3 * bk, 3 * bk + 5
    rng = np.random.default_rng(bm + bk)
    a = rng.integers(0, 1 << 32, (m - 1) * lda + k, dtype=np.uint64).astype(np.uint32)
    out = np.zeros(m * k, dtype=np.uint32)
    oracle.operand_tiles(a, out, m=m, k=k, lda=lda, bm=bm, bk=bk)
    dense = np.lib.stride_tricks.as_strided(a, shape=(m, k), strides=(lda * 4, 4))
    want = dense.reshape(m // bm, bm, k // bk, bk).transpose(0, 2, 3, 1)  # [mt][kt][k][m]
    assert np.array_equal(out.reshape(m // bm, k // bk, bk, bm), want)


def test_operand_tiles_index_closed_form_and_hand_example():
    # A is 2x4 (lda 4) holding its own linear index; BM = 2, BK = 2 gives two
    # tiles, each the transpose of a 2x2 block: [[0,4],[1,5]] and [[2,6],[3,7]].
    a = np.arange(8, dtype=np.uint32)
    out = np.zeros(8, dtype=np.uint32)
    oracle.operand_tiles(a, out, m=2, k=4, lda=4, bm=2, bk=2)
    assert out.tolist() == [0, 4, 1, 5, 2, 6, 3, 7]
    m, k, bm, bk = 8, 12, 4, 3
    a = np.arange(m * k, dtype=np.uint32)
    out = np.zeros(m * k, dtype=np.uint32)
    oracle.operand_tiles(a, out, m=m, k=k, lda=k, bm=bm, bk=bk)
    mt, kt, kk, mm = np.indices((m // bm, k // bk, bk, bm))
    assert np.array_equal(out.reshape(m // bm, k // bk, bk, bm),
                          ((mt * bm + mm) * k + kt * bk + kk).astype(np.uint32))
