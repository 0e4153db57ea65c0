"""Reader for the hand-written transpose fixtures in ``tests/golden``."""
from __future__ import annotations

import glob
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_transpose_fixture(path):
    """Return (params, in_tokens, out_tokens) with tokens as lists of rows."""
    params, blocks, cur = {}, {"in": [], "out": []}, None
    with open(path) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line in ("in", "out"):
                cur = line
                continue
            if cur is None:
                toks = line.split()
                params.update({toks[k]: int(toks[k + 1]) for k in range(0, len(toks), 2)})
            else:
                blocks[cur].append(line.split())
    return params, blocks["in"], blocks["out"]


def fixture_arrays(path, dtype, pad_in, pad_out):
    """Build flat input/expected-output arrays; P and Q become the given sentinels."""
    p, rows_in, rows_out = read_transpose_fixture(path)
    conv = lambda t, pad: pad if t in ("P", "Q") else int(t)
    x = np.array([conv(t, pad_in) for r in rows_in for t in r], dtype=dtype)
    y = np.array([conv(t, pad_out) for r in rows_out for t in r], dtype=dtype)
    assert x.size == p["batch"] * p["stride_in"], path
    assert y.size == p["batch"] * p["stride_out"], path
    return p, x, y


def transpose_fixtures():
    return sorted(glob.glob(os.path.join(GOLDEN_DIR, "transpose_*.txt")))


def inplace_fixtures():
    return sorted(glob.glob(os.path.join(GOLDEN_DIR, "inplace_*.txt")))
