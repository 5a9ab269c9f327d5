"""Pins for the oracle's micro-step accumulation (deg/zero.py collect / reduce_scatter)."""
import math

import numpy as np

from oracle.accum import accumulate


def test_exact_closed_form():
    parts = [np.full(10, 0.5, np.float32) for _ in range(4)]
    assert np.array_equal(accumulate(parts), np.full(10, 2.0, np.float32))
    assert np.array_equal(accumulate([np.arange(5, dtype=np.float32)]), np.arange(5, dtype=np.float32))


def test_order_is_sequential_fp32():
    # 1 + 2^-24 + 2^-24: sequentially each tiny part rounds away; the other order keeps them
    parts = [np.array([1.0], np.float32), np.array([2 ** -24], np.float32), np.array([2 ** -24], np.float32)]
    assert accumulate(parts)[0] == np.float32(1.0)
    assert accumulate(parts[::-1])[0] == np.float32(1.0 + 2 ** -23)


def test_close_to_exact_sum():
    rng = np.random.default_rng(0)
    parts = [rng.normal(0, 1e-3, 1000).astype(np.float32) for _ in range(4)]
    exact = np.array([math.fsum(float(p[i]) for p in parts) for i in range(1000)])
    got = accumulate(parts).astype(np.float64)
    scale = np.sum([np.abs(p.astype(np.float64)) for p in parts], axis=0)
    assert np.all(np.abs(got - exact) <= 3 * 2.0 ** -24 * scale)
