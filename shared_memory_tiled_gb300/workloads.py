"""Seeded synthetic inputs for the transpose workloads.

This module is shared by the tests, the benchmark and the oracle-side checks.
It holds none of the transpose's arithmetic: it only names the workloads
(shape, pitch, element type, value distribution, seed) and fills host buffers
with their input values.  Every value it produces comes from numpy's PCG64
generator (``numpy.random.default_rng(seed)``) or from the element's own
linear index, in row-major logical order, batch plane by batch plane.

Pitch padding (the elements between ``cols`` and ``ld_in`` of each input row,
and between batch planes) is filled with a NaN sentinel that the value
distributions below can never produce, so a test can tell whether any padding
element leaked into the output.

The workloads follow the five configurations the library is measured on:

* ``c1_index``   fp32 1024x1024, every element holds its own linear index
  (exact below 2**24) -- the exact check of "Shared memory and the bank
  conflict", section "The barrier";
* ``c1_uniform`` the same shape, uniform[-1, 1) from seed 0;
* ``c2``         fp32 8192x8192 (256 MiB), uniform[-1, 1) from seed 1;
* ``c3``         fp32 12289x7919 with input row pitch 7936, N(0, 1) from seed 2;
* ``c4``         batched fp32 [64, 2048, 1536] -> [64, 1536, 2048], uniform from seed 3;
* ``c5``         bf16 16384x16384 (512 MiB), uniform random 16-bit patterns
  from seed 4 (NaN and Inf patterns included);
* ``c3_back``    c3's transpose back: 7919x12289 with input pitch 12289 (rows
  start at every 4-byte offset from a 16-byte boundary) and output pitch 7936.
* ``c5_oddin``   c5 with input pitch 16385 (bf16 rows start at every 2-byte
  offset from a 16-byte boundary), output dense.
* ``c5_oddout``  c5 with output pitch 16385; ``c5_oddboth`` with both pitches
  16385; ``c2_oddout`` c2 with output pitch 8193.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# NaN bit patterns used only to fill padding.  Uniform[-1,1) and N(0,1) fp32
# draws are finite, so these never occur as data in the fp32 workloads.
IN_PAD_U32 = np.uint32(0x7FC0DEAD)
OUT_PAD_U32 = np.uint32(0xFFC0BEEF)
IN_PAD_U16 = np.uint16(0x7FAD)
OUT_PAD_U16 = np.uint16(0xFFBE)

ESIZE = {"f32": 4, "bf16": 2}
BITS_DTYPE = {"f32": np.uint32, "bf16": np.uint16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One transpose problem: ``batch`` planes of ``rows`` x ``cols`` inputs.

    All pitches are in elements.  ``ld_in``/``ld_out`` are the row pitches of
    the input (rows x cols) and output (cols x rows) planes; ``stride_in`` and
    ``stride_out`` are the plane pitches.
    """
    name: str
    dtype: str            # "f32" or "bf16"
    rows: int
    cols: int
    ld_in: int
    ld_out: int
    batch: int = 1
    stride_in: int = 0    # 0 means rows * ld_in
    stride_out: int = 0   # 0 means cols * ld_out
    dist: str = "uniform" # "index", "uniform", "normal" or "bits"
    seed: int = 0

    @property
    def esize(self) -> int:
        return ESIZE[self.dtype]

    @property
    def sin(self) -> int:
        return self.stride_in or self.rows * self.ld_in

    @property
    def sout(self) -> int:
        return self.stride_out or self.cols * self.ld_out

    @property
    def in_elems(self) -> int:
        """Elements of the input buffer: whole planes, pitch padding included."""
        return self.batch * self.sin

    @property
    def out_elems(self) -> int:
        return self.batch * self.sout

    @property
    def logical_elems(self) -> int:
        return self.batch * self.rows * self.cols

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes read plus bytes written: every logical element once each way."""
        return 2 * self.esize * self.logical_elems

    def scaled(self, name: str, **kw) -> "Workload":
        return dataclasses.replace(self, name=name, **kw)


WORKLOADS = {
    "c1_index": Workload("c1_index", "f32", 1024, 1024, 1024, 1024, dist="index"),
    "c1_uniform": Workload("c1_uniform", "f32", 1024, 1024, 1024, 1024, dist="uniform", seed=0),
    "c2": Workload("c2", "f32", 8192, 8192, 8192, 8192, dist="uniform", seed=1),
    "c3": Workload("c3", "f32", 12289, 7919, 7936, 12289, dist="normal", seed=2),
    "c4": Workload("c4", "f32", 2048, 1536, 1536, 2048, batch=64, dist="uniform", seed=3),
    "c5": Workload("c5", "bf16", 16384, 16384, 16384, 16384, dist="bits", seed=4),
    # c3 transposed back: the odd pitch is now on the input side
    "c3_back": Workload("c3_back", "f32", 7919, 12289, 12289, 7936, dist="normal", seed=2),
    # c5 with the odd pitch on the input side
    "c5_oddin": Workload("c5_oddin", "bf16", 16384, 16384, 16385, 16384, dist="bits", seed=4),
    # c5 with an odd output pitch (shifted stores), and with both pitches odd
    "c5_oddout": Workload("c5_oddout", "bf16", 16384, 16384, 16384, 16385, dist="bits", seed=4),
    "c5_oddboth": Workload("c5_oddboth", "bf16", 16384, 16384, 16385, 16385, dist="bits", seed=4),
    # c2 with an odd output pitch
    "c2_oddout": Workload("c2_oddout", "f32", 8192, 8192, 8192, 8193, dist="uniform", seed=1),
}

DESCRIPTION = {
    "c1_index": "fp32 1024x1024 row-major, in[i][j] = float(i*1024+j), ld = cols",
    "c1_uniform": "fp32 1024x1024 row-major, uniform[-1,1) seed 0, ld = cols",
    "c2": "fp32 8192x8192 (256 MiB) square, uniform[-1,1) seed 1, ld = cols",
    "c3": "fp32 12289x7919 rectangular, N(0,1) seed 2, ld_in = 7936, output dense",
    "c4": "batched fp32 [64,2048,1536] -> [64,1536,2048], uniform[-1,1) seed 3, contiguous",
    "c5": "bf16 16384x16384 (512 MiB) square, uniform random u16 bits seed 4",
    "c3_back": "fp32 7919x12289 (c3's output shape), input pitch 12289, output pitch 7936, N(0,1) seed 2",
    "c5_oddin": "bf16 16384x16384, input pitch 16385, output dense, uniform random u16 bits seed 4",
    "c5_oddout": "bf16 16384x16384, input dense, output pitch 16385, uniform random u16 bits seed 4",
    "c5_oddboth": "bf16 16384x16384, input and output pitch 16385, uniform random u16 bits seed 4",
    "c2_oddout": "fp32 8192x8192, input dense, output pitch 8193, uniform[-1,1) seed 1",
}


def logical_values(w: Workload) -> np.ndarray:
    """The ``batch*rows*cols`` logical input values as raw bits, row-major order."""
    n = w.logical_elems
    if w.dist == "index":
        if w.dtype == "f32":
            if n > (1 << 24):
                # Past 2**24 a float no longer holds every integer exactly: use
                # the index itself as the bit pattern instead.
                return np.arange(n, dtype=np.uint32)
            return np.arange(n, dtype=np.float32).view(np.uint32)
        return (np.arange(n, dtype=np.uint32) & 0xFFFF).astype(np.uint16)
    rng = np.random.default_rng(w.seed)
    if w.dist == "uniform":
        if w.dtype != "f32":
            raise ValueError("uniform draws are defined for fp32 workloads")
        v = rng.random(n, dtype=np.float32)
        v *= np.float32(2.0)
        v -= np.float32(1.0)
        return v.view(np.uint32)
    if w.dist == "normal":
        if w.dtype != "f32":
            raise ValueError("normal draws are defined for fp32 workloads")
        return rng.standard_normal(n, dtype=np.float32).view(np.uint32)
    if w.dist == "bits":
        if w.dtype == "bf16":
            return rng.integers(0, 65536, n, dtype=np.uint16)
        return rng.integers(0, 1 << 32, n, dtype=np.uint32)
    raise ValueError(f"unknown distribution {w.dist!r}")


def make_input(w: Workload) -> np.ndarray:
    """Flat input buffer (raw bits) of ``w.in_elems`` elements, padding = sentinel."""
    vals = logical_values(w)
    dt = BITS_DTYPE[w.dtype]
    if w.ld_in == w.cols and w.sin == w.rows * w.cols:
        return vals.astype(dt, copy=False)
    buf = np.full(w.in_elems, IN_PAD_U32 if dt is np.uint32 else IN_PAD_U16, dtype=dt)
    planes = buf.reshape(w.batch, w.sin)
    src = vals.reshape(w.batch, w.rows, w.cols)
    for b in range(w.batch):
        body = planes[b, : w.rows * w.ld_in].reshape(w.rows, w.ld_in)
        body[:, : w.cols] = src[b]
    return buf


def make_output(w: Workload) -> np.ndarray:
    """Flat output buffer of ``w.out_elems`` elements, prefilled with the output sentinel."""
    dt = BITS_DTYPE[w.dtype]
    return np.full(w.out_elems, OUT_PAD_U32 if dt is np.uint32 else OUT_PAD_U16, dtype=dt)


def random_bits(n: int, dtype: str, seed: int) -> np.ndarray:
    """``n`` uniformly random raw bit patterns of the given element type."""
    rng = np.random.default_rng(seed)
    if dtype == "bf16":
        return rng.integers(0, 65536, n, dtype=np.uint16)
    return rng.integers(0, 1 << 32, n, dtype=np.uint32)
