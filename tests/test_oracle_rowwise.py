"""Pins for the oracle's standalone row softmax and layer normalisation.

Each pin comes from the mathematics of the definition (closed forms,
invariants, special cases) or from an independent library routine (torch's
fp64 softmax and layer_norm on the CPU), never from a re-typed copy of the
oracle's own formula.
"""
import numpy as np
import pytest
import torch


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_softmax_rows_sum_to_one_and_match_torch(oracle_mod):
    x = rnd((7, 333), 1, 3.0)
    y = oracle_mod.softmax_rows(x)
    np.testing.assert_allclose(y.sum(-1), 1.0, atol=1e-13)
    np.testing.assert_allclose(y, torch.softmax(torch.from_numpy(x), -1).numpy(), rtol=1e-13, atol=1e-300)


def test_softmax_closed_forms(oracle_mod):
    # constant row: uniform; two entries: logistic of the difference
    y = oracle_mod.softmax_rows(np.full((2, 5), 3.25))
    np.testing.assert_array_equal(y, np.full((2, 5), 0.2))
    a, b = 1.5, -0.75
    y = oracle_mod.softmax_rows(np.array([[a, b]]))
    np.testing.assert_allclose(y[0], [1 / (1 + np.exp(b - a)), 1 / (1 + np.exp(a - b))], rtol=1e-15)


def test_softmax_shift_invariance_and_large_values(oracle_mod):
    x = np.round(rnd((3, 50), 2, 4.0))
    y0 = oracle_mod.softmax_rows(x)
    np.testing.assert_allclose(oracle_mod.softmax_rows(x + 17.0), y0, rtol=1e-14)
    # values far beyond exp's range: only a max-subtracted evaluation stays finite
    y = oracle_mod.softmax_rows(x + 2000.0)
    assert np.isfinite(y).all()
    np.testing.assert_allclose(y, y0, rtol=1e-14)


def test_layernorm_matches_torch(oracle_mod):
    x = rnd((6, 257), 3, 2.0) + 1.5
    g, b = rnd(257, 4), rnd(257, 5)
    y = oracle_mod.layernorm_rows(x, g, b, 1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (257,), torch.from_numpy(g), torch.from_numpy(b), 1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_layernorm_moments_closed_form(oracle_mod):
    """gamma = 1, beta = 0: each output row has mean 0 and mean square var / (var + eps)."""
    x = rnd((4, 100), 6, 0.3)
    eps = 0.01
    y = oracle_mod.layernorm_rows(x, np.ones(100), np.zeros(100), eps)
    var = x.var(-1)
    np.testing.assert_allclose(y.mean(-1), 0.0, atol=1e-14)
    np.testing.assert_allclose((y * y).mean(-1), var / (var + eps), rtol=1e-12)


def test_layernorm_constant_row_and_affine_invariance(oracle_mod):
    g, b = rnd(30, 7), rnd(30, 8)
    y = oracle_mod.layernorm_rows(np.full((2, 30), -4.5), g, b, 1e-3)
    np.testing.assert_array_equal(y, np.tile(b, (2, 1)))  # x - mean = 0 exactly
    x = rnd((3, 30), 9)
    y0 = oracle_mod.layernorm_rows(x, g, b, 0.0)
    np.testing.assert_allclose(oracle_mod.layernorm_rows(2.5 * x - 7.0, g, b, 0.0), y0, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("N", [1, 2])
def test_tiny_rows(oracle_mod, N):
    x = rnd((2, N), 10)
    np.testing.assert_allclose(oracle_mod.softmax_rows(x).sum(-1), 1.0, atol=1e-15)
    y = oracle_mod.layernorm_rows(x, np.full(N, 2.0), np.full(N, 0.5), 1e-6)
    if N == 1:
        np.testing.assert_array_equal(y, np.full((2, 1), 0.5))
    else:  # two values: normalised to -1, +1 (times sqrt(var / (var + eps)))
        var = x.var(-1, keepdims=True)
        np.testing.assert_allclose(np.abs(y - 0.5), np.broadcast_to(2.0 * np.sqrt(var / (var + 1e-6)), y.shape), rtol=1e-12)
