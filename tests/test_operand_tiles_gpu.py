"""GPU parity of the transposed operand-tile stage against the oracle, for
every supported tile shape and padding (the page's rule, none, and others)."""
import numpy as np
import pytest

import oracle
from gpu_util import first_mismatch, from_device, to_device
from shared_memory_tiled_gb300 import binding as B

pytestmark = pytest.mark.gpu

SHAPES = [(128, 8), (128, 16), (128, 32), (64, 8), (64, 16), (64, 32)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()


@pytest.mark.parametrize("bm,bk", SHAPES)
def test_operand_tiles(bm, bk):
    import torch
    m, k = 3 * bm, 5 * bk
    for lda in (k, k + 4, k + 20):
        a = np.random.default_rng(bm * 100 + bk + lda).integers(
            0, 1 << 32, (m - 1) * lda + k, dtype=np.uint64).astype(np.uint32)
        want = np.zeros(m * k, dtype=np.uint32)
        oracle.operand_tiles(a, want, m=m, k=k, lda=lda, bm=bm, bk=bk)
        for pad in (-1, 0, 1, 2, 4):
            da, pa = to_device(a)
            dout, po = to_device(np.full(m * k, 0xFFFFFFFF, dtype=np.uint32))
            B.check(B.tr_operand_tiles_f32(pa, po, m, k, lda, bm, bk, pad))
            torch.cuda.synchronize()
            got = from_device(dout, m * k, 0, np.uint32)
            assert np.array_equal(got, want), f"{(bm, bk, lda, pad)}: {first_mismatch(got, want)}"


def test_operand_tiles_large():
    import torch
    m, k = 4096, 4096
    a = np.random.default_rng(7).integers(0, 1 << 32, m * k, dtype=np.uint64).astype(np.uint32)
    want = np.zeros(m * k, dtype=np.uint32)
    oracle.operand_tiles(a, want, m=m, k=k, lda=k, bm=128, bk=16)
    da, pa = to_device(a)
    dout, po = to_device(np.zeros(m * k, dtype=np.uint32))
    B.check(B.tr_operand_tiles_f32(pa, po, m, k, k, 128, 16, -1))
    torch.cuda.synchronize()
    assert np.array_equal(from_device(dout, m * k, 0, np.uint32), want)


def test_operand_tiles_refusals():
    assert B.tr_operand_tiles_f32(16, 1 << 40, 128, 16, 16, 96, 16, 0) == B.Status.ERR_UNSUPPORTED
    assert B.tr_operand_tiles_f32(16, 1 << 40, 100, 16, 16, 128, 16, 0) == B.Status.ERR_UNSUPPORTED
    assert B.tr_operand_tiles_f32(20, 1 << 40, 128, 16, 16, 128, 16, 0) == B.Status.ERR_UNSUPPORTED
    assert B.tr_operand_tiles_f32(16, 16, 128, 16, 16, 128, 16, 0) == B.Status.ERR_OVERLAP
    assert B.tr_operand_tiles_f32(0, 0, 0, 16, 16, 128, 16, 0) == B.Status.OK
