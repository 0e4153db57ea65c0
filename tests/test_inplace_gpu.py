"""GPU parity of the in-place square transpose against the CPU oracle's
pairwise-swap loop, bit for bit, padding included."""
import numpy as np
import pytest

import oracle
from gpu_util import first_mismatch, from_device, to_device
from shared_memory_tiled_gb300 import binding as B
from shared_memory_tiled_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()


def run_gpu(x, batch, n, ld, stride, off=0):
    import torch
    buf, ptr = to_device(x, off)
    f = B.tr_transpose_inplace_f32 if x.dtype == np.uint32 else B.tr_transpose_inplace_bf16
    B.check(f(ptr, batch, n, ld, stride))
    torch.cuda.synchronize()
    return from_device(buf, x.size, off, x.dtype.type)


def case(dt, batch, n, pad, ppad, seed):
    ld = n + pad
    stride = n * ld + ppad
    size = batch * stride
    x = np.random.default_rng(seed).integers(0, np.iinfo(dt).max, size, dtype=dt, endpoint=True)
    return x, ld, stride


@pytest.mark.parametrize("dt", [np.uint32, np.uint16], ids=["f32", "bf16"])
def test_inplace_shapes(dt):
    al = 16 // np.dtype(dt).itemsize
    for batch, n, pad, ppad in [(1, 1, 0, 0), (1, 7, 0, 0), (1, 64, 0, 0), (1, 65, al, 0),
                                (3, 128, 0, 0), (2, 200, 3, 5), (1, 257, al, 0),
                                (1, 1000, 0, 0), (2, 300, 2 * al, 4 * al), (1, 129, 1, 0)]:
        x, ld, stride = case(dt, batch, n, pad, ppad, seed=n + batch)
        want = oracle.transpose_inplace(x.copy(), batch=batch, n=n, ld=ld, stride=stride)
        for off in (0, 1):
            got = run_gpu(x, batch, n, ld, stride, off)
            assert np.array_equal(got, want), f"{(batch, n, pad, ppad, off)}: {first_mismatch(got, want)}"


@pytest.mark.parametrize("name", ["c2", "c5"])
def test_inplace_full_size(name):
    w = W.WORKLOADS[name]
    x = W.make_input(w)
    want = oracle.transpose_inplace(x.copy(), n=w.rows, ld=w.ld_in)
    got = run_gpu(x, 1, w.rows, w.ld_in, w.rows * w.ld_in)
    assert np.array_equal(got, want), first_mismatch(got, want)


def test_inplace_twice_is_identity_on_device():
    import torch
    x = torch.randn(4, 513, 513, device="cuda")
    y = x.clone()
    B.transpose_(y)
    assert torch.equal(y, x.transpose(1, 2))
    B.transpose_(y)
    assert torch.equal(y, x)
