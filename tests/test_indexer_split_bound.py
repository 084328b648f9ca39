"""The split-product term of the tensor-core indexer scores' error bound, on
the CPU: with x1 = bf16(x) and x2 = bf16(x - x1) (round to nearest even, as
the split kernel does), the three products q1.k1 + q1.k2 + q2.k1 differ
from the exact <q, k> by at most 3.02 * 2^-16 * sum_d |q_d k_d|, and every
split term is exact as claimed (x - x1 in fp32, |x - x1 - x2| <= 2^-16 |x|)."""

import numpy as np
import pytest


def bf16_rne(x):
    """fp32 -> the nearest bf16 (ties to even), returned as fp32."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((b >> 16) & 1)
    return ((b + bias) & 0xFFFF0000).astype(np.uint32).view(np.float32)


def split(x):
    x = np.asarray(x, dtype=np.float32)
    x1 = bf16_rne(x)
    r = (x - x1).astype(np.float32)                  # exact in fp32
    x2 = bf16_rne(r)
    return x1, x2, r


@pytest.mark.parametrize("scale", [1e-3, 1.0, 37.0, 1e4])
def test_split_terms_are_exact_and_small(scale):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * scale).astype(np.float32)
    x1, x2, r = split(x)
    # x - x1 computed in fp32 equals the exact difference
    assert np.array_equal(r.astype(np.float64), x.astype(np.float64) - x1.astype(np.float64))
    resid = np.abs(x.astype(np.float64) - x1 - x2.astype(np.float64))
    assert np.all(resid <= 2.0 ** -16 * np.abs(x.astype(np.float64)))


@pytest.mark.parametrize("D,scale", [(128, 1.0), (128, 0.01), (64, 300.0)])
def test_three_products_within_the_split_bound(D, scale):
    rng = np.random.default_rng(11 + D)
    n = 4000
    q = (rng.standard_normal((n, D)) * scale).astype(np.float32)
    k = (rng.standard_normal((n, D)) * rng.uniform(0.1, 10.0, (n, 1))).astype(np.float32)
    # a few rows with heavy cancellation: k nearly orthogonal to q
    k[:50] -= (np.sum(q[:50] * k[:50], axis=1, keepdims=True) /
               np.sum(q[:50] * q[:50], axis=1, keepdims=True) * q[:50]).astype(np.float32)
    q1, q2, _ = split(q)
    k1, k2, _ = split(k)
    f = lambda a: a.astype(np.float64)
    exact = np.sum(f(q) * f(k), axis=1)
    three = np.sum(f(q1) * f(k1) + f(q1) * f(k2) + f(q2) * f(k1), axis=1)
    mag = np.sum(np.abs(f(q) * f(k)), axis=1)
    err = np.abs(three - exact)
    assert np.all(err <= 3.02 * 2.0 ** -16 * mag)
    # the bound is not vacuous: the error reaches a visible share of it
    assert err.max() > 0.01 * 2.0 ** -16 * mag[np.argmax(err)]
