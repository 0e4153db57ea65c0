"""The column-read microbenchmark computes its closed-form folds, and the
unpadded column read is slower than the padded and swizzled ones."""
import numpy as np
import pytest

from shared_memory_tiled_gb300 import binding as B
from shared_memory_tiled_gb300 import probe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()


def test_probe_results_and_ordering():
    times = {}
    for layout in range(4):
        ms, ok = probe.run(layout, reps=2048, blocks=152 * 4, trials=5)
        assert ok, f"layout {layout} fold differs from its closed form"
        times[layout] = ms
    assert times[0] > 4 * times[1] and times[0] > 4 * times[2]


def test_probe_rejects_bad_arguments():
    assert B.tr_bank_probe(7, 1, 1, 0) == B.Status.ERR_UNSUPPORTED
    assert B.tr_bank_probe(0, -1, 1, 0) == B.Status.ERR_BAD_DIM
    assert B.tr_bank_probe(0, 1, 1, 0) == B.Status.ERR_NULL
    assert B.tr_bank_probe(0, 1, 0, 0) == B.Status.OK
