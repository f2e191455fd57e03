"""Pins for the oracle's gated-MLP epilogue (h = silu(g) * u), independent of
its own code: known values of the logistic function, scipy's expit, a
numerical check of the slope bound the tolerance uses, and a dense fp64
numpy matmul of the masked gate and up matrices."""
import math

import numpy as np
import pytest
import scipy.special

import oracle


def test_silu_known_values():
    # silu(g) = g * logistic(g); logistic(1) = e / (e + 1)
    e = math.e
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(e / (e + 1.0), rel=1e-15)
    assert oracle.silu(-1.0) == pytest.approx(-1.0 / (e + 1.0), rel=1e-15)
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu(-40.0)) < 1e-15
    assert oracle.silu(-1000.0) == 0.0  # exp overflow: the limit


def test_silu_matches_scipy_expit():
    g = np.random.default_rng(3).standard_normal(10000) * 8
    np.testing.assert_allclose(oracle.silu(g), g * scipy.special.expit(g), rtol=1e-13,
                               atol=1e-300)


def test_silu_slope_stays_below_the_bound():
    rng = np.random.default_rng(5)
    a = rng.uniform(-30, 30, 200000)
    b = a + rng.uniform(-1e-3, 1e-3, a.size)
    slope = np.abs(oracle.silu(a) - oracle.silu(b)) / np.abs(a - b)
    assert slope.max() <= oracle.SILU_LIPSCHITZ
    assert slope.max() > 1.09  # the bound is tight, not loose


@pytest.mark.parametrize("N,M,B", [(2, 4, 1), (1, 4, 3), (4, 8, 2), (2, 8, 8)])
def test_gate_up_matches_dense_numpy(N, M, B):
    rng = np.random.default_rng(N * 100 + M * 10 + B)
    rows, K = 37, 64
    def case():
        W = (rng.standard_normal((rows, K)) * 0.05).astype(np.float16)
        m = np.zeros((rows, K // M, M), dtype=np.uint8)
        for r in range(rows):
            for g in range(K // M):
                m[r, g, rng.choice(M, N, replace=False)] = 1
        return W, m.reshape(rows, K)
    Wg, mg = case()
    Wu, mu = case()
    x = rng.standard_normal((B, K)).astype(np.float16)
    h, bound = oracle.gate_up_silu(Wg, mg, Wu, mu, x)
    g = x.astype(np.float64) @ (Wg.astype(np.float64) * mg).T
    u = x.astype(np.float64) @ (Wu.astype(np.float64) * mu).T
    expect = g / (1.0 + np.exp(-g)) * u
    np.testing.assert_allclose(h, expect, rtol=1e-12, atol=1e-15)
    assert (bound > 0).all()


def test_gate_up_bound_covers_tolerated_errors():
    """A g and u perturbed by exactly the SpMV tolerance stay inside the bound."""
    rng = np.random.default_rng(11)
    rows, K = 64, 128
    Wg = (rng.standard_normal((rows, K)) * 0.05).astype(np.float16)
    Wu = (rng.standard_normal((rows, K)) * 0.05).astype(np.float16)
    ones = np.ones((rows, K), dtype=np.uint8)
    x = rng.standard_normal((1, K)).astype(np.float16)
    h, bound = oracle.gate_up_silu(Wg, ones, Wu, ones, x)
    g, sg = oracle.spmv_dense(Wg, ones, x)
    u, su = oracle.spmv_dense(Wu, ones, x)
    for sgn_g in (-1, 1):
        for sgn_u in (-1, 1):
            g2 = g + sgn_g * (1e-3 * sg + 1e-6)
            u2 = u + sgn_u * (1e-3 * su + 1e-6)
            h2 = oracle.silu(g2) * u2
            assert (np.abs(h2 - h) <= bound).all()


def test_gate_up_all_ones_closed_form():
    """Every weight kept and 1, x all ones: g = u = K, h = silu(K) K."""
    rows, K = 3, 16
    W = np.ones((rows, K), dtype=np.float16)
    m = np.ones((rows, K), dtype=np.uint8)
    x = np.full((1, K), 0.25, dtype=np.float16)
    h, _ = oracle.gate_up_silu(W, m, W, m, x)
    s = K * 0.25
    np.testing.assert_allclose(h, np.full((1, rows), s * s / (1 + math.exp(-s))), rtol=1e-15)
