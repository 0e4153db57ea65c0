"""The seeded input generators (no GPU)."""
import numpy as np

from shared_memory_tiled_gb300 import workloads as W


def test_sizes_and_bytes():
    c = W.WORKLOADS
    assert c["c1_index"].algorithmic_bytes == 8_388_608
    assert c["c2"].algorithmic_bytes == 536_870_912
    assert c["c3"].algorithmic_bytes == 778_532_728
    assert c["c4"].algorithmic_bytes == 1_610_612_736
    assert c["c5"].algorithmic_bytes == 1_073_741_824
    assert c["c3"].in_elems == 12289 * 7936 and c["c3"].out_elems == 7919 * 12289
    assert c["c4"].sin == 2048 * 1536 == c["c4"].sout


def test_deterministic_and_seeded():
    w = W.WORKLOADS["c1_uniform"]
    a, b = W.make_input(w), W.make_input(w)
    assert np.array_equal(a, b)
    other = W.make_input(w.scaled("x", seed=99))
    assert not np.array_equal(a, other)
    f = a.view(np.float32)
    assert f.min() >= -1.0 and f.max() < 1.0


def test_index_values_exact():
    w = W.WORKLOADS["c1_index"]
    x = W.make_input(w).view(np.float32)
    assert np.array_equal(x, np.arange(1024 * 1024, dtype=np.float64).astype(np.float32))
    assert x[-1] == 1024 * 1024 - 1


def test_pitch_padding_holds_sentinel():
    w = W.WORKLOADS["c3"].scaled("small", rows=5, cols=7, ld_in=10, ld_out=5)
    x = W.make_input(w).reshape(5, 10)
    assert np.all(x[:, 7:] == W.IN_PAD_U32)
    assert np.all(np.isfinite(x[:, :7].view(np.float32)))


def test_bits_cover_nan_patterns():
    w = W.WORKLOADS["c5"].scaled("small", rows=256, cols=256, ld_in=256, ld_out=256)
    x = W.make_input(w)
    nan = ((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0)
    assert nan.any()
