"""Pins for the oracle's calibration accumulation (H += X^T X over tokens),
independent of its C loops: numpy's matmul, one-hot and rank-one closed
forms, symmetry and additivity over token batches."""
import numpy as np

import oracle


def _x(T, K, seed):
    return np.random.default_rng(seed).standard_normal((T, K)).astype(np.float16)


def test_matches_numpy_matmul():
    X = _x(37, 24, 1)
    H, S = oracle.calib_accumulate(X)
    Xd = X.astype(np.float64)
    np.testing.assert_allclose(H, Xd.T @ Xd, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S, np.abs(Xd).T @ np.abs(Xd), rtol=1e-13, atol=1e-13)


def test_one_hot_tokens_count_features():
    """Token t = e_{f(t)}: H is diagonal with the number of tokens per feature."""
    K, f = 8, [0, 3, 3, 7, 3]
    X = np.zeros((len(f), K), dtype=np.float16)
    for t, k in enumerate(f):
        X[t, k] = 1
    H, _ = oracle.calib_accumulate(X)
    assert np.array_equal(H, np.diag([1, 0, 0, 3, 0, 0, 0, 1]).astype(float))


def test_single_token_is_an_outer_product_and_h0_is_kept():
    x = np.array([[1, -2, 0.5, 4]], dtype=np.float16)
    H0 = np.arange(16, dtype=np.float64).reshape(4, 4)
    H, _ = oracle.calib_accumulate(x, H0)
    xd = x[0].astype(np.float64)
    assert np.array_equal(H, H0 + np.outer(xd, xd))


def test_symmetric_and_additive_over_batches():
    X = _x(50, 16, 2)
    H, _ = oracle.calib_accumulate(X)
    assert np.array_equal(H, H.T)
    H1, _ = oracle.calib_accumulate(X[:20])
    H2, _ = oracle.calib_accumulate(X[20:], H1)
    np.testing.assert_allclose(H2, H, rtol=1e-14, atol=1e-14)
