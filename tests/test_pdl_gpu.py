"""Back-to-back dependent launches (programmatic dependent launch).

Every transpose and copy kernel may be scheduled while the previous kernel in
the stream is still running, and waits at its start until that kernel has
completed.  These tests chain dependent calls with no host synchronisation in
between: A -> B then B -> A, many times, which exercises both a read of the
previous kernel's output (B) and a write over the previous kernel's input (A).
Any missing or misplaced wait shows up as a corrupted A.
"""
from __future__ import annotations

import pytest

from shared_memory_tiled_gb300 import binding as B

pytestmark = pytest.mark.gpu

V = B.Variant
KINDS = [dict(variant=V.AUTO), dict(variant=V.TILE_VEC), dict(variant=V.TILE_PAD, pad=1),
         dict(variant=V.NAIVE_ROW), dict(variant=V.TMA), dict(variant=V.TMA, schedule=1),
         dict(variant=V.TMA, schedule=3), dict(variant=V.TMA, schedule=4)]


def _pingpong(a, b, rows, cols, dt, kw, rounds):
    fwd = B.make_args(a.data_ptr(), b.data_ptr(), dt, 1, rows, cols, cols, rows)
    bwd = B.make_args(b.data_ptr(), a.data_ptr(), dt, 1, cols, rows, rows, cols)
    opts = B.make_options(**kw)
    for _ in range(rounds):
        B.check(B.tr_transpose_ex(fwd, opts))
        B.check(B.tr_transpose_ex(bwd, opts))


@pytest.mark.parametrize("kw", KINDS, ids=lambda k: "-".join(f"{v}" for v in k.values()))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_transpose_pingpong(kw, dtype):
    import torch
    rows, cols = 3072, 2048 + 64
    tdt = torch.int32 if dtype == "f32" else torch.int16
    dt = B.DType.F32 if dtype == "f32" else B.DType.BF16
    g = torch.Generator(device="cuda").manual_seed(11)
    lo, hi = (-2**31, 2**31 - 1) if dtype == "f32" else (-2**15, 2**15 - 1)
    a = torch.randint(lo, hi, (rows * cols,), dtype=tdt, device="cuda", generator=g)
    ref = a.clone()
    b = torch.empty_like(a)
    _pingpong(a, b, rows, cols, dt, kw, rounds=15)
    torch.cuda.synchronize()
    assert torch.equal(a, ref)
    assert torch.equal(b.view(cols, rows), ref.view(rows, cols).t())


def test_chain_through_copy_inplace_and_a_torch_kernel():
    import torch
    n = 4096
    a = torch.randint(-2**31, 2**31 - 1, (n * n,), dtype=torch.int32, device="cuda")
    ref = a.clone()
    b = torch.empty_like(a)
    c = torch.empty_like(a)
    args_ab = B.make_args(a.data_ptr(), b.data_ptr(), B.DType.F32, 1, n, n, n, n)
    for _ in range(10):
        B.check(B.tr_copy(a.data_ptr(), c.data_ptr(), n * n * 4))          # c = a
        B.check(B.tr_transpose_ex(args_ab))                                # b = a^T
        B.check(B.tr_transpose_inplace_f32(b.data_ptr(), 1, n, n, n * n))  # b = a
        c.add_(1)                                                          # c = a + 1 (torch)
        B.check(B.tr_copy(c.data_ptr(), a.data_ptr(), n * n * 4))          # a = a + 1
        B.check(B.tr_transpose_inplace_f32(a.data_ptr(), 1, n, n, n * n))  # a = (a + 1)^T
        B.check(B.tr_transpose_inplace_f32(a.data_ptr(), 1, n, n, n * n))  # a = a + 1
    torch.cuda.synchronize()
    assert torch.equal(a, ref + 10)
    assert torch.equal(b, ref + 9)


def test_every_pair_of_kernels_back_to_back():
    """A -> B with one variant, B -> A with another, for every ordered pair:
    persistent TMA grids followed by one-tile-per-block grids and back."""
    import torch
    rows, cols = 1536, 2048 + 64
    a = torch.randint(-2**31, 2**31 - 1, (rows * cols,), dtype=torch.int32, device="cuda")
    ref = a.clone()
    b = torch.empty_like(a)
    fwd = B.make_args(a.data_ptr(), b.data_ptr(), B.DType.F32, 1, rows, cols, cols, rows)
    bwd = B.make_args(b.data_ptr(), a.data_ptr(), B.DType.F32, 1, cols, rows, rows, cols)
    opts = [B.make_options(**kw) for kw in KINDS]
    for o1 in opts:
        for o2 in opts:
            B.check(B.tr_transpose_ex(fwd, o1))
            B.check(B.tr_transpose_ex(bwd, o2))
    torch.cuda.synchronize()
    assert torch.equal(a, ref)
    assert torch.equal(b.view(cols, rows), ref.view(rows, cols).t())
