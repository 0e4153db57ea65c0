"""The C-ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments before any CUDA call (no GPU needed)."""
from __future__ import annotations

import os
import re

import pytest

from shared_memory_tiled_gb300 import binding as B
from shared_memory_tiled_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "transpose.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tr_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["tr_transpose_f32", "tr_transpose_bf16", "tr_transpose_batched_f32",
                     "tr_transpose_batched_bf16", "tr_copy", "tr_transpose_ex",
                     "tr_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in transpose.h but not exported"
    assert set(declared_functions()) == set(B.SIGNATURES), "binding and header disagree"


def test_exports_are_c_linkage(lib):
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = set(re.findall(r"\bT (tr_[a-z0-9_]+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported


def test_only_the_declared_entry_points_are_exported(lib):
    """Everything else is hidden, so a second copy of the library (or any other
    library) in the same process shares none of its kernels or caches."""
    import shutil
    if shutil.which("nm") is None:
        pytest.skip("nm not available")
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    names = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert names == set(declared_functions()), sorted(names - set(declared_functions()))


def test_version_and_strings(lib):
    assert B.tr_version() == 10000
    for s in B.Status:
        msg = B.tr_status_string(s)
        assert msg and msg != "unknown status"
    assert B.tr_status_string(99) == "unknown status"
    assert isinstance(B.tr_last_error(), str)


FAKE_IN, FAKE_OUT = 0x7F0000000000, 0x7F1000000000  # never dereferenced


@pytest.mark.parametrize("fn", ["tr_transpose_f32", "tr_transpose_bf16"])
def test_single_matrix_argument_errors(lib, fn):
    f = getattr(B, fn)
    assert f(FAKE_IN, FAKE_OUT, -1, 4, 4, 4) == B.Status.ERR_BAD_DIM
    assert f(FAKE_IN, FAKE_OUT, 4, -1, 4, 4) == B.Status.ERR_BAD_DIM
    assert f(0, FAKE_OUT, 4, 4, 4, 4) == B.Status.ERR_NULL
    assert f(FAKE_IN, 0, 4, 4, 4, 4) == B.Status.ERR_NULL
    assert f(FAKE_IN, FAKE_OUT, 4, 5, 4, 4) == B.Status.ERR_BAD_LD     # ld_in < cols
    assert f(FAKE_IN, FAKE_OUT, 5, 4, 4, 4) == B.Status.ERR_BAD_LD     # ld_out < rows
    # overlapping ranges: output starts inside the input extent
    assert f(FAKE_IN, FAKE_IN + 8, 4, 4, 4, 4) == B.Status.ERR_OVERLAP
    assert f(FAKE_IN + 8, FAKE_IN, 4, 4, 4, 4) == B.Status.ERR_OVERLAP
    # overflowing extents
    assert f(FAKE_IN, FAKE_OUT, 1 << 40, 1 << 40, 1 << 40, 1 << 40) == B.Status.ERR_BAD_DIM
    # a pointer off its element boundary is refused before any launch
    es = 4 if fn.endswith("f32") else 2
    for off in range(1, es):
        assert f(FAKE_IN + off, FAKE_OUT, 4, 4, 4, 4) == B.Status.ERR_UNSUPPORTED
        assert f(FAKE_IN, FAKE_OUT + off, 4, 4, 4, 4) == B.Status.ERR_UNSUPPORTED
    # empty problems succeed without touching anything, even with NULL pointers
    assert f(0, 0, 0, 5, 5, 0) == B.Status.OK
    assert f(0, 0, 7, 0, 0, 7) == B.Status.OK


@pytest.mark.parametrize("fn", ["tr_transpose_batched_f32", "tr_transpose_batched_bf16"])
def test_batched_argument_errors(lib, fn):
    f = getattr(B, fn)
    assert f(FAKE_IN, FAKE_OUT, -1, 4, 4, 4, 4, 16, 16) == B.Status.ERR_BAD_DIM
    assert f(FAKE_IN, FAKE_OUT, 2, 4, 4, 4, 4, 15, 16) == B.Status.ERR_BAD_LD
    assert f(FAKE_IN, FAKE_OUT, 2, 4, 4, 4, 4, 16, 15) == B.Status.ERR_BAD_LD
    # planes may pack tighter than rows*ld when the last row is short (checked
    # with the planner, which validates without launching)
    dt = B.DType.F32 if fn.endswith("f32") else B.DType.BF16
    assert _plan(FAKE_IN, FAKE_OUT, dt, 2, 4, 3, 5, 4, 18, 12) > 0
    assert _plan(FAKE_IN, FAKE_OUT, dt, 2, 4, 3, 5, 4, 17, 12) == -B.Status.ERR_BAD_LD
    assert f(0, 0, 0, 4, 4, 4, 4, 16, 16) == B.Status.OK
    # overlap found through the last plane
    es = 4 if fn.endswith("f32") else 2
    assert f(FAKE_IN, FAKE_IN + es * 20, 2, 4, 4, 4, 4, 16, 16) == B.Status.ERR_OVERLAP


def test_copy_argument_errors(lib):
    assert B.tr_copy(0, FAKE_OUT, 16) == B.Status.ERR_NULL
    assert B.tr_copy(FAKE_IN, FAKE_IN + 8, 16) == B.Status.ERR_OVERLAP
    assert B.tr_copy(0, 0, 0) == B.Status.OK


def _plan(in_ptr, out_ptr, dtype, batch, rows, cols, ld_in, ld_out, si=0, so=0, **opt):
    a = B.make_args(in_ptr, out_ptr, dtype, batch, rows, cols, ld_in, ld_out, si, so)
    return B.tr_plan_variant(a, B.make_options(**opt) if opt else None)


def test_planner(lib):
    F32, BF16 = B.DType.F32, B.DType.BF16
    # AUTO takes the vectorised swizzled tile for every alignment class
    # (aligned, misaligned output pitch, misaligned base, batched)
    for case in [(FAKE_IN, FAKE_OUT, F32, 1, 8192, 8192, 8192, 8192),
                 (FAKE_IN, FAKE_OUT, BF16, 1, 16384, 16384, 16384, 16384),
                 (FAKE_IN, FAKE_OUT, F32, 64, 2048, 1536, 1536, 2048, 2048 * 1536, 1536 * 2048),
                 (FAKE_IN, FAKE_OUT, F32, 1, 12289, 7919, 7936, 12289),
                 (FAKE_IN + 4, FAKE_OUT, F32, 1, 64, 64, 64, 64),
                 (FAKE_IN, FAKE_OUT, BF16, 1, 4, 4, 4, 4),
                 (FAKE_IN, FAKE_OUT, F32, 2, 4, 4, 4, 4, 17, 16)]:
        assert _plan(*case) == B.Variant.TILE_VEC
    # explicit requests are honoured
    for v in B.Variant:
        if v != B.Variant.AUTO:
            assert _plan(FAKE_IN, FAKE_OUT, F32, 1, 64, 64, 64, 64, variant=v) == v
    # invalid arguments and options come back as negative statuses
    assert _plan(FAKE_IN, FAKE_OUT, F32, 1, -1, 4, 4, 4) == -B.Status.ERR_BAD_DIM
    assert _plan(FAKE_IN, FAKE_OUT, F32, 1, 4, 4, 4, 4, variant=9) == -B.Status.ERR_UNSUPPORTED
    assert _plan(FAKE_IN, FAKE_OUT, F32, 1, 4, 4, 4, 4, stages=1) == -B.Status.ERR_UNSUPPORTED
    assert _plan(FAKE_IN, FAKE_OUT, F32, 1, 4, 4, 4, 4, pad=5) == -B.Status.ERR_UNSUPPORTED
    assert _plan(FAKE_IN, FAKE_OUT, F32, 1, 4, 4, 4, 4, schedule=5) == -B.Status.ERR_UNSUPPORTED
    assert _plan(FAKE_IN, FAKE_OUT, 7, 1, 4, 4, 4, 4) == -B.Status.ERR_UNSUPPORTED


def _plan_ex(in_ptr, out_ptr, dtype, batch, rows, cols, ld_in, ld_out, si=0, so=0, **opt):
    a = B.make_args(in_ptr, out_ptr, dtype, batch, rows, cols, ld_in, ld_out, si, so)
    p = B.Plan()
    st = B.tr_plan_ex(a, B.make_options(**opt) if opt else None, p)
    return st, p


def test_plan_ex_reports_the_tile_auto_takes(lib):
    """AUTO's vector-tile shape and block size for each alignment class, as the
    header documents them (tile rows, tile cols, threads, vec_in, vec_out)."""
    F32, BF16 = B.DType.F32, B.DType.BF16
    cases = [
        ((F32, 1, 8192, 8192, 8192, 8192), (64, 64, 256, 1, 1)),                  # C2
        ((F32, 1, 12289, 7919, 7936, 12289), (128, 64, 256, 1, 0)),              # C3
        ((F32, 64, 2048, 1536, 1536, 2048, 2048 * 1536, 1536 * 2048), (64, 64, 256, 1, 1)),
        ((BF16, 1, 16384, 16384, 16384, 16384), (128, 128, 256, 1, 1)),          # C5
        ((F32, 1, 7919, 12289, 12289, 7936), (64, 128, 256, 0, 1)),              # C3 back
        ((BF16, 1, 16384, 16384, 16385, 16384), (64, 128, 128, 0, 1)),           # odd input
        ((BF16, 1, 16384, 16384, 16385, 16385), (64, 128, 128, 0, 0)),           # both odd
        ((BF16, 1, 16384, 16384, 16384, 16385), (128, 128, 256, 1, 0)),          # odd output
        ((F32, 2, 64, 64, 64, 64, 64 * 64 + 1, 64 * 64), (64, 128, 256, 0, 1)),  # plane pitch
    ]
    for args, want in cases:
        st, p = _plan_ex(FAKE_IN, FAKE_OUT, *args)
        assert st == B.Status.OK and p.variant == B.Variant.TILE_VEC, args
        assert (p.tile_rows, p.tile_cols, p.threads, p.vec_in, p.vec_out) == want, args
        assert p.schedule == 0
    st, p = _plan_ex(FAKE_IN + 4, FAKE_OUT, F32, 1, 64, 64, 64, 64)              # base pointer
    assert (p.tile_rows, p.tile_cols, p.threads, p.vec_in, p.vec_out) == (64, 128, 256, 0, 1)


def test_plan_ex_reports_requests_and_refusals(lib):
    F32, BF16, V = B.DType.F32, B.DType.BF16, B.Variant
    # a block size set by the caller keeps bf16's 128x128 tile for a misaligned input
    st, p = _plan_ex(FAKE_IN, FAKE_OUT, BF16, 1, 4096, 4096, 4097, 4096, variant=V.TILE_VEC,
                     threads=256)
    assert (st, p.tile_rows, p.tile_cols, p.threads) == (B.Status.OK, 128, 128, 256)
    # explicit shapes and the prefetching schedule are reported as requested
    st, p = _plan_ex(FAKE_IN, FAKE_OUT, F32, 1, 64, 64, 64, 64, variant=V.TILE_VEC,
                     tile_rows=128, tile_cols=32, schedule=2)
    assert (st, p.tile_rows, p.tile_cols, p.threads, p.schedule) == (B.Status.OK, 128, 32, 256, 2)
    st, p = _plan_ex(FAKE_IN, FAKE_OUT, F32, 1, 64, 64, 64, 64, variant=V.TILE_VEC, tile_rows=128)
    assert (p.tile_rows, p.tile_cols) == (128, 64)
    # the other variants carry no tile shape
    for v in (V.TMA, V.TILE_PAD, V.NAIVE_ROW, V.NAIVE_COL):
        st, p = _plan_ex(FAKE_IN, FAKE_OUT, F32, 1, 64, 64, 64, 64, variant=v)
        assert st == B.Status.OK and p.variant == v and (p.tile_rows, p.threads) == (0, 0)
        assert (p.vec_in, p.vec_out) == (1, 1)
    # refusals match tr_transpose_ex's argument checks
    assert _plan_ex(FAKE_IN, FAKE_OUT, F32, 1, 64, 64, 65, 64, variant=V.TMA)[0] == \
        B.Status.ERR_UNSUPPORTED
    assert _plan_ex(FAKE_IN, FAKE_OUT, F32, 1, 64, 64, 64, 64, variant=V.TILE_VEC,
                    schedule=3)[0] == B.Status.ERR_UNSUPPORTED
    assert _plan_ex(FAKE_IN, FAKE_OUT, F32, 1, 4, 5, 4, 4)[0] == B.Status.ERR_BAD_LD
    assert _plan_ex(FAKE_IN + 2, FAKE_OUT, F32, 1, 4, 4, 4, 4)[0] == B.Status.ERR_UNSUPPORTED
    assert _plan_ex(FAKE_IN, FAKE_OUT, F32, 1, 4, 4, 4, 4, pad=5)[0] == B.Status.ERR_UNSUPPORTED
    a = B.make_args(FAKE_IN, FAKE_OUT, F32, 1, 4, 4, 4, 4)
    assert B.tr_plan_ex(a, None, None) == B.Status.ERR_NULL


def test_ex_rejects_bad_options_and_reserved_fields(lib):
    a = B.make_args(FAKE_IN, FAKE_OUT, B.DType.F32, 1, 4, 4, 4, 4)
    assert B.tr_transpose_ex(a, B.make_options(variant=42)) == B.Status.ERR_UNSUPPORTED
    o = B.make_options(threads=64)
    assert B.tr_transpose_ex(a, o) == B.Status.ERR_UNSUPPORTED
    # the TMA load pipelines (schedules 3 and 4) are refused for the LSU tile,
    # on the host, before any CUDA call
    for sched in (3, 4):
        o = B.make_options(B.Variant.TILE_VEC, schedule=sched)
        assert B.tr_transpose_ex(a, o) == B.Status.ERR_UNSUPPORTED
    a.reserved = 1
    assert B.tr_transpose_ex(a, None) == B.Status.ERR_UNSUPPORTED
    assert B.tr_transpose_ex(B.make_args(0, 0, B.DType.F32, 0, 0, 0, 0, 0)) == B.Status.OK
    assert B.load().tr_transpose_ex(None, None) == B.Status.ERR_NULL


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(B.LibraryMissing):
        B.load(str(tmp_path / "nope.so"))
    monkeypatch.setattr(B, "_lib", None)


@pytest.mark.parametrize("fn", ["tr_transpose_inplace_f32", "tr_transpose_inplace_bf16"])
def test_inplace_argument_errors(lib, fn):
    f = getattr(B, fn)
    assert f(FAKE_IN, -1, 4, 4, 16) == B.Status.ERR_BAD_DIM
    assert f(FAKE_IN, 1, -4, 4, 16) == B.Status.ERR_BAD_DIM
    assert f(0, 1, 4, 4, 16) == B.Status.ERR_NULL
    assert f(FAKE_IN, 1, 5, 4, 16) == B.Status.ERR_BAD_LD
    assert f(FAKE_IN, 2, 4, 4, 15) == B.Status.ERR_BAD_LD
    assert f(FAKE_IN, 1, 1 << 40, 1 << 40, 0) == B.Status.ERR_BAD_DIM
    es = 4 if fn.endswith("f32") else 2
    for off in range(1, es):
        assert f(FAKE_IN + off, 1, 4, 4, 16) == B.Status.ERR_UNSUPPORTED
    assert f(0, 0, 4, 4, 16) == B.Status.OK and f(0, 3, 0, 0, 0) == B.Status.OK


def test_operand_tiles_argument_errors(lib):
    f = B.tr_operand_tiles_f32
    assert f(FAKE_IN, FAKE_OUT, -1, 16, 16, 128, 16) == B.Status.ERR_BAD_DIM
    assert f(FAKE_IN, FAKE_OUT, 128, 16, 16, 96, 16) == B.Status.ERR_UNSUPPORTED
    assert f(FAKE_IN, FAKE_OUT, 128, 16, 16, 128, 12) == B.Status.ERR_UNSUPPORTED
    assert f(FAKE_IN, FAKE_OUT, 128, 16, 16, 128, 16, 9) == B.Status.ERR_UNSUPPORTED
    assert f(FAKE_IN, FAKE_OUT, 100, 16, 16, 128, 16) == B.Status.ERR_UNSUPPORTED
    assert f(FAKE_IN + 4, FAKE_OUT, 128, 16, 16, 128, 16) == B.Status.ERR_UNSUPPORTED
    assert f(FAKE_IN, FAKE_OUT, 128, 16, 18, 128, 16) == B.Status.ERR_UNSUPPORTED
    assert f(FAKE_IN, FAKE_OUT + 2, 128, 16, 16, 128, 16) == B.Status.ERR_UNSUPPORTED
    assert f(FAKE_IN, FAKE_OUT, 128, 16, 8, 128, 16) == B.Status.ERR_BAD_LD
    assert f(0, FAKE_OUT, 128, 16, 16, 128, 16) == B.Status.ERR_NULL
    assert f(FAKE_IN, FAKE_IN + 64, 128, 16, 16, 128, 16) == B.Status.ERR_OVERLAP
    assert f(0, 0, 0, 16, 16, 128, 16) == B.Status.OK


def test_bank_probe_argument_errors(lib):
    assert B.tr_bank_probe(4, 1, 1, FAKE_OUT) == B.Status.ERR_UNSUPPORTED
    assert B.tr_bank_probe(0, -1, 1, FAKE_OUT) == B.Status.ERR_BAD_DIM
    assert B.tr_bank_probe(0, 1, 1, 0) == B.Status.ERR_NULL
    assert B.tr_bank_probe(0, 1, 1, FAKE_OUT + 2) == B.Status.ERR_UNSUPPORTED
    assert B.tr_bank_probe(0, 1, 0, 0) == B.Status.OK


def test_selftest_argument_errors_on_host(lib):
    assert B.tr_selftest_bounded_wait(0, 0) == B.Status.ERR_BAD_DIM
    assert B.tr_selftest_bounded_wait(1, -5) == B.Status.ERR_BAD_DIM


def test_plan_ex_against_the_documented_rules(lib):
    """Random pointers, shapes and pitches: the planner's aligned sides and
    AUTO's tile equal a restatement of the header's rules (a side allows
    16-byte accesses when its base, row pitch and, for batch > 1, plane pitch
    are multiples of 16 bytes; then the tile follows the table in tr_options)."""
    import numpy as np
    rng = np.random.default_rng(7)

    def aligned(base, ld, stride, batch, es):
        return base % 16 == 0 and (ld * es) % 16 == 0 and (batch == 1 or (stride * es) % 16 == 0)

    def auto_tile(es, in16, out16):
        v = 16 // es
        if not in16 and es == 2:
            return 64, 128, 128
        if not out16:
            return 128, 16 * v, 256
        if not in16:
            return 16 * v, 128, 256
        return 16 * v, 16 * v, 256

    for _ in range(3000):
        dt = B.DType.F32 if rng.random() < 0.5 else B.DType.BF16
        es = 4 if dt == B.DType.F32 else 2
        batch = int(rng.choice([1, 1, 2, 5]))
        rows, cols = int(rng.integers(1, 5000)), int(rng.integers(1, 5000))
        ld_in, ld_out = cols + int(rng.integers(0, 20)), rows + int(rng.integers(0, 20))
        si = (rows - 1) * ld_in + cols + int(rng.integers(0, 40))
        so = (cols - 1) * ld_out + rows + int(rng.integers(0, 40))
        base_in = FAKE_IN + es * int(rng.integers(0, 8))
        base_out = FAKE_OUT + es * int(rng.integers(0, 8))
        st, p = _plan_ex(base_in, base_out, dt, batch, rows, cols, ld_in, ld_out, si, so)
        assert st == B.Status.OK
        in16 = aligned(base_in, ld_in, si, batch, es)
        out16 = aligned(base_out, ld_out, so, batch, es)
        assert (p.vec_in, p.vec_out) == (in16, out16)
        assert p.variant == B.Variant.TILE_VEC
        assert (p.tile_rows, p.tile_cols, p.threads) == auto_tile(es, in16, out16)


def test_release_build_makes_no_bounds_checks(lib):
    """The release library has no bounds checks: both debug entry points say so
    on the host, without a CUDA call, and a NULL report is an argument error."""
    rep = B.BoundsReport(refused=5)
    assert B.tr_debug_bounds(rep) == B.Status.ERR_UNSUPPORTED
    assert rep.refused == 0
    assert "TR_DEBUG" in B.tr_last_error()
    assert B.tr_debug_bounds(None) == B.Status.ERR_NULL
    assert B.tr_debug_bounds_selftest(0x10000) == B.Status.ERR_UNSUPPORTED
