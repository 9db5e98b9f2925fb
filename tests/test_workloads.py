"""The seeded input generators: deterministic, and shaped as stated."""
import numpy as np

from fp8_fine_grained_17_b300 import workloads as wl


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -0.0], dtype=np.float32)
    b = wl.bf16_bits(x)
    assert list(b) == [0x3F80, 0x3F80, 0x3F82, 0x8000]
    assert np.array_equal(wl.bits_to_f32(b), np.array([1.0, 1.0, 1.0 + 2.0 ** -6, -0.0], np.float32))


def test_dense_deterministic_and_outliers():
    d1 = wl.dense("t", 64, 128, 2048, seed=3, outlier_scale=50.0)
    d2 = wl.dense("t", 64, 128, 2048, seed=3, outlier_scale=50.0)
    assert np.array_equal(d1.a_bits, d2.a_bits) and np.array_equal(d1.w_bits, d2.w_bits)
    assert len(d1.outlier_cols) == 10
    a = wl.bits_to_f32(d1.a_bits)
    mask = np.zeros(2048, bool)
    mask[d1.outlier_cols] = True
    assert np.abs(a[:, mask]).mean() > 30 * np.abs(a[:, ~mask]).mean()
    w = wl.bits_to_f32(d1.w_bits)
    assert 0.015 < w.std() < 0.025


def test_moe_routing():
    c = wl.moe_routing(0)
    assert c.shape == (32,) and c.min() >= 0 and c.max() <= 8192
    assert np.array_equal(c, wl.moe_routing(0))
    small = wl.moe(seed=0, N=128, K=128, counts=[2, 0, 3])
    assert list(small.offsets) == [0, 2, 2, 5]
    assert small.a_bits.shape == (5, 128) and small.w_bits.shape == (3, 128, 128)
