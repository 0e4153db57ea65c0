"""Seeded random sweep of transpose configurations against the oracle.

Each case draws an element type, a batch count, a shape, row pitches (dense,
padded by a few elements -- usually breaking 16-byte alignment -- or padded up
to a 16-byte multiple), plane gaps, base-pointer offsets and a variant with its
options, and compares the whole output buffer with the oracle bit for bit
(pitch padding and plane gaps included: they must keep their prefill)."""
from __future__ import annotations

import numpy as np
import pytest

import pins
from fuzz_cases import U16, U32, draw
from gpu_util import first_mismatch, gpu_out, oracle_out
from shared_memory_tiled_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()
    yield
    assert B.tr_device_status() == B.Status.OK, "a bounded in-kernel wait ran out"


@pytest.mark.parametrize("seed", range(6))
def test_random_configurations(seed):
    rng = np.random.default_rng(1000 + seed)
    for k in range(150):
        dtype, geo, in_off, out_off, opt = draw(rng)
        batch, rows, cols, ld_in, ld_out, si, so = geo
        x, prefill, _ = pins.alloc_case(dtype, batch, rows, cols, ld_in, ld_out, si, so,
                                        seed=int(rng.integers(1 << 30)))
        want = oracle_out(x, prefill, *geo)
        got = gpu_out(x, prefill, *geo, in_off=in_off, out_off=out_off, **opt)
        assert np.array_equal(got, want), \
            f"case {k}: {np.dtype(dtype).name} {geo} offsets {in_off}/{out_off} {opt}: " \
            f"{first_mismatch(got, want)}"


@pytest.mark.parametrize("seed", range(3))
def test_random_inplace_configurations(seed):
    """The in-place square transpose over random sizes, pitches, plane gaps and
    base offsets, against the oracle's pairwise swaps."""
    import oracle
    import torch
    from gpu_util import from_device, to_device
    rng = np.random.default_rng(2000 + seed)
    for k in range(60):
        dt = U32 if rng.random() < 0.5 else U16
        vec = 4 if dt is U32 else 8
        batch = int(rng.choice([1, 1, 2, 3]))
        n = int(rng.integers(1, 600))
        c = rng.random()
        ld = n if c < 0.4 else n + int(rng.integers(1, 9)) if c < 0.75 else n + (-n) % vec
        stride = n * ld + (int(rng.integers(0, 17)) if batch > 1 else 0)
        off = int(rng.choice([0, 0, 1, 3]))
        x = rng.integers(0, np.iinfo(dt).max, batch * stride, dtype=dt, endpoint=True)
        want = oracle.transpose_inplace(x.copy(), batch=batch, n=n, ld=ld, stride=stride)
        buf, ptr = to_device(x, off)
        f = B.tr_transpose_inplace_f32 if dt is U32 else B.tr_transpose_inplace_bf16
        B.check(f(ptr, batch, n, ld, stride))
        torch.cuda.synchronize()
        got = from_device(buf, x.size, off, dt)
        assert np.array_equal(got, want), \
            f"case {k}: {np.dtype(dt).name} batch {batch} n {n} ld {ld} stride {stride} " \
            f"offset {off}: {first_mismatch(got, want)}"
