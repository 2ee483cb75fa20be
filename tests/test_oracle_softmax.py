"""Pins for the oracle's safe softmax (CPU only).

Each check comes from outside the oracle: a closed form, an invariant the
mathematics fixes, brute force with math.exp, or torch's own float64 softmax.
"""

import math

import numpy as np
import scipy.special
import pytest
import torch

import oracle

EPS = np.finfo(np.float64).eps


def test_constant_row_closed_form():
    # All entries equal: every weight is 1/n, m = s*c, l = n.
    n, c, s = 37, 2.5, 0.75
    y, m, l = oracle.softmax_rows(np.full((1, n), c), scale=s)
    assert m[0] == s * c
    assert l[0] == pytest.approx(n, rel=4 * EPS)
    np.testing.assert_allclose(y, np.full((1, n), 1.0 / n), rtol=4 * EPS)


def test_log_integers_closed_form():
    # x_j = ln(j+1): exp(x_j - m) = (j+1)/n, so y_j = (j+1) / sum(1..n).
    n = 6
    x = np.log(np.arange(1, n + 1, dtype=np.float64))[None, :]
    y, m, l = oracle.softmax_rows(x)
    total = n * (n + 1) / 2
    np.testing.assert_allclose(y[0], np.arange(1, n + 1) / total, rtol=8 * EPS)
    assert m[0] == pytest.approx(math.log(n), rel=2 * EPS)
    assert l[0] == pytest.approx(total / n, rel=8 * EPS)


def test_shift_invariance():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((5, 50))
    y0, m0, l0 = oracle.softmax_rows(x)
    y1, m1, l1 = oracle.softmax_rows(x + 3.0)
    np.testing.assert_allclose(y1, y0, rtol=1e-13, atol=0)
    np.testing.assert_allclose(m1, m0 + 3.0, rtol=1e-15)
    np.testing.assert_allclose(l1, l0, rtol=1e-13)


def test_normaliser_bounds_and_sum_to_one():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((64, 300)) * 10
    y, m, l = oracle.softmax_rows(x)
    assert np.all(l >= 1.0) and np.all(l <= x.shape[1])
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=1e-13)
    # the maximum entry has weight exactly 1/l
    j = x.argmax(axis=1)
    np.testing.assert_allclose(y[np.arange(64), j], 1.0 / l, rtol=4 * EPS)


def test_one_hot_dominant_row():
    # Gaps beyond ~745 make every other term underflow to 0 in float64.
    x = np.zeros((1, 9))
    x[0, 4] = 800.0
    y, m, l = oracle.softmax_rows(x)
    assert l[0] == 1.0
    assert m[0] == 800.0
    assert y[0, 4] == 1.0 and np.count_nonzero(y) == 1


def test_scale_multiplies_logits():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((3, 20)).astype(np.float32)
    y, m, l = oracle.softmax_rows(x, scale=0.125)
    y2, m2, l2 = oracle.softmax_rows(x.astype(np.float64) * 0.125)
    np.testing.assert_array_equal(m, m2)
    np.testing.assert_allclose(y, y2, rtol=0, atol=0)


def test_brute_force_small():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((4, 7)) * 3
    s = 0.9
    y, m, l = oracle.softmax_rows(x, scale=s)
    for r in range(4):
        mm = max(s * v for v in x[r])
        ll = sum(math.exp(s * v - mm) for v in x[r])
        assert m[r] == mm
        assert l[r] == pytest.approx(ll, rel=8 * EPS)
        for j in range(7):
            assert y[r, j] == pytest.approx(math.exp(s * x[r, j] - mm) / ll, rel=8 * EPS)


def test_matches_torch_float64_softmax():
    g = torch.Generator().manual_seed(15)
    x = torch.randn(33, 129, generator=g, dtype=torch.float64) * 10
    y, m, l = oracle.softmax_rows(x.numpy(), scale=0.5)
    ref = torch.softmax(x * 0.5, dim=1).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-300)
    # scipy, not torch.logsumexp: on float64 CPU tensors the latter was seen
    # to return results 1.6e-10 off (relative) in a few percent of processes
    lse = scipy.special.logsumexp((x * 0.5).numpy(), axis=1)
    np.testing.assert_allclose(m + np.log(l), lse, rtol=1e-13)


def test_masked_entries_and_empty_row():
    x = np.array([[0.0, -np.inf, 1.0], [-np.inf, -np.inf, -np.inf]])
    y, m, l = oracle.softmax_rows(x)
    e = math.e
    np.testing.assert_allclose(y[0], [1 / (1 + e), 0.0, e / (1 + e)], rtol=4 * EPS)
    assert m[1] == -np.inf and l[1] == 0.0
    assert np.all(y[1] == 0.0) and not np.any(np.isnan(y))


def test_naive_normaliser_overflows_at_scale_1000():
    # curionode "The Online Softmax": e^1000 is infinite; double overflows past e^709.
    assert math.isinf(oracle.naive_normaliser([709.0])) is False
    assert math.isinf(oracle.naive_normaliser([710.0]))
    rng = np.random.default_rng(16)
    x = rng.standard_normal(64)
    assert math.isfinite(oracle.naive_normaliser(x))
    assert not math.isfinite(oracle.naive_normaliser(x, scale=1000.0))
