"""Pins for the FP64 row-operator oracle (softmax, RMSNorm, LayerNorm).

Each check is fixed by mathematics, not by retyping the oracle's formula:
closed forms for special rows, exact invariances on dyadic inputs, and an
independent implementation (numpy's vectorised float64 routines, a
different summation order) on random rows.
"""
import math

import numpy as np
import pytest

import oracle


def _rng(seed=0):
    return np.random.default_rng(seed)


def _dyadic(rows, width, seed):
    return (_rng(seed).integers(-64, 65, (rows, width)) / 16.0).astype(np.float32)


# ---- softmax -----------------------------------------------------------------------

def test_softmax_rows_sum_to_one_and_are_positive():
    x = _rng(1).standard_normal((9, 1000)).astype(np.float32) * 5
    y = oracle.softmax(x)
    assert np.all(y > 0)
    assert np.allclose(y.sum(1), 1.0, rtol=0, atol=1e-14)


def test_softmax_constant_row_is_uniform():
    for w in (1, 7, 8191):
        y = oracle.softmax(np.full((2, w), -3.25, np.float32))
        assert np.all(y == 1.0 / w)


def test_softmax_two_elements_closed_form():
    a, b = 0.75, -1.5
    y = oracle.softmax(np.array([[a, b]], np.float32))
    assert y[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(b - a)), rel=1e-15)
    assert y[0, 1] == pytest.approx(1.0 / (1.0 + math.exp(a - b)), rel=1e-15)


def test_softmax_is_shift_invariant_bit_for_bit():
    x = _dyadic(4, 33, 2)
    assert np.array_equal(oracle.softmax(x), oracle.softmax(x + np.float32(7.5)))


def test_softmax_dominant_entry_and_no_overflow():
    y = oracle.softmax(np.array([[0.0, -1000.0, 3.0e38]], np.float32))
    assert y[0, 2] == 1.0 and y[0, 0] == 0.0 and y[0, 1] == 0.0


def test_softmax_matches_numpy_float64():
    x = _rng(3).standard_normal((17, 513)).astype(np.float32)
    x64 = x.astype(np.float64)
    e = np.exp(x64 - x64.max(1, keepdims=True))
    ref = e / e.sum(1, keepdims=True)
    assert np.max(np.abs(oracle.softmax(x) - ref) / ref) < 1e-14


# ---- RMSNorm -----------------------------------------------------------------------

def test_rmsnorm_constant_row_closed_form():
    c, eps = -2.5, 1e-5
    y = oracle.rmsnorm(np.full((1, 10), c, np.float32), eps=eps)
    assert np.allclose(y, c / math.sqrt(c * c + eps), rtol=1e-15, atol=0)


def test_rmsnorm_scale_invariant_with_zero_eps_and_linear_in_gamma():
    x = _dyadic(3, 40, 4)
    g = _rng(5).standard_normal(40).astype(np.float32)
    assert np.array_equal(oracle.rmsnorm(x, eps=0.0), oracle.rmsnorm(np.float32(2) * x, eps=0.0))
    assert np.array_equal(2 * oracle.rmsnorm(x, g), oracle.rmsnorm(x, np.float32(2) * g))


def test_rmsnorm_mean_square_of_output():
    x = _rng(6).standard_normal((5, 4096)).astype(np.float32)
    eps = 1e-3
    ms = np.mean(x.astype(np.float64) ** 2, axis=1)
    y = oracle.rmsnorm(x, eps=eps)
    assert np.allclose(np.mean(y ** 2, axis=1), ms / (ms + eps), rtol=1e-13)


def test_rmsnorm_matches_numpy_float64():
    x = _rng(7).standard_normal((11, 777)).astype(np.float32)
    g = _rng(8).standard_normal(777).astype(np.float32)
    x64 = x.astype(np.float64)
    ref = x64 / np.sqrt(np.mean(x64 * x64, axis=1, keepdims=True) + 1e-5) * g.astype(np.float64)
    assert np.max(np.abs(oracle.rmsnorm(x, g) - ref)) < 1e-13


# ---- LayerNorm ---------------------------------------------------------------------

def test_layernorm_constant_row_gives_beta():
    b = _rng(9).standard_normal(12).astype(np.float32)
    g = _rng(10).standard_normal(12).astype(np.float32)
    y = oracle.layernorm(np.full((3, 12), 4.125, np.float32), g, b)
    assert np.array_equal(y, np.broadcast_to(b.astype(np.float64), (3, 12)))


def test_layernorm_shift_invariant_on_power_of_two_width():
    x = _dyadic(4, 64, 11)   # sums and means are exact in double
    assert np.array_equal(oracle.layernorm(x), oracle.layernorm(x + np.float32(-3.0)))


def test_layernorm_output_moments():
    x = _rng(12).standard_normal((6, 2048)).astype(np.float32) * 3 + 1
    eps = 1e-2
    v = np.var(x.astype(np.float64), axis=1)
    y = oracle.layernorm(x, eps=eps)
    assert np.allclose(y.mean(1), 0.0, atol=1e-13)
    assert np.allclose(y.var(1), v / (v + eps), rtol=1e-12)


def test_layernorm_matches_numpy_float64():
    x = _rng(13).standard_normal((9, 1001)).astype(np.float32)
    g = _rng(14).standard_normal(1001).astype(np.float32)
    b = _rng(15).standard_normal(1001).astype(np.float32)
    x64 = x.astype(np.float64)
    mu = x64.mean(1, keepdims=True)
    ref = (x64 - mu) / np.sqrt(x64.var(1, keepdims=True) + 1e-5) * g + b
    assert np.max(np.abs(oracle.layernorm(x, g, b) - ref)) < 1e-12


def test_row_operators_reject_bad_shapes():
    with pytest.raises(ValueError):
        oracle.softmax(np.zeros(5, np.float32))
    with pytest.raises(ValueError):
        oracle.rmsnorm(np.zeros((2, 5), np.float32), np.zeros(4, np.float32))
