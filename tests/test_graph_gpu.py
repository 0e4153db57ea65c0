"""The library's calls inside a captured CUDA graph.

Every transpose and copy call is an ordinary stream launch (with programmatic
stream serialization), so a sequence of calls can be captured once and
replayed; the first call of each configuration on a device sets its kernel
attributes, so the test makes those calls before capturing.
"""
from __future__ import annotations

import pytest

from shared_memory_tiled_gb300 import binding as B

pytestmark = pytest.mark.gpu

V = B.Variant
KINDS = [dict(variant=V.AUTO), dict(variant=V.TILE_PAD, pad=1), dict(variant=V.TMA),
         dict(variant=V.TMA, schedule=1), dict(variant=V.TMA, schedule=3),
         dict(variant=V.TMA, schedule=4)]


def test_chain_replays_from_a_graph():
    import torch
    rows, cols = 2048, 2048 + 64
    n = 1024
    s = torch.cuda.Stream()
    a = torch.randint(-2**31, 2**31 - 1, (rows * cols,), dtype=torch.int32, device="cuda")
    ref = a.clone()
    b = torch.empty_like(a)
    sq = torch.randint(-2**31, 2**31 - 1, (n * n,), dtype=torch.int32, device="cuda")
    sq_ref = sq.clone()
    c = torch.empty_like(sq)
    fwd = B.make_args(a.data_ptr(), b.data_ptr(), B.DType.F32, 1, rows, cols, cols, rows,
                      stream=s.cuda_stream)
    bwd = B.make_args(b.data_ptr(), a.data_ptr(), B.DType.F32, 1, cols, rows, rows, cols,
                      stream=s.cuda_stream)
    opts = [B.make_options(**kw) for kw in KINDS]

    def sequence():
        for o in opts:
            B.check(B.tr_transpose_ex(fwd, o))
            B.check(B.tr_transpose_ex(bwd, o))
        B.check(B.tr_transpose_inplace_f32(sq.data_ptr(), 1, n, n, n * n, s.cuda_stream))
        B.check(B.tr_copy(sq.data_ptr(), c.data_ptr(), n * n * 4, s.cuda_stream))
        B.check(B.tr_transpose_inplace_f32(sq.data_ptr(), 1, n, n, n * n, s.cuda_stream))

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sequence()  # every configuration once, outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sequence()
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a, ref)
    assert torch.equal(b.view(cols, rows), ref.view(rows, cols).t())
    assert torch.equal(sq, sq_ref)
    assert torch.equal(c.view(n, n), sq_ref.view(n, n).t())
