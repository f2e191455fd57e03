"""Pins for the oracle's score-driven N:M mask selection, independent of its
C loops: a numpy sort route (lexsort by score, then position), every ordering
of distinct scores in a group, ties, and the magnitude special case."""
import itertools

import numpy as np
import pytest

import oracle


def _np_select(W16, N, M, scale=None):
    """Sort route: fp32 scores (numpy's IEEE single multiply), per group
    the N first positions of a stable order by (-score, position)."""
    s = np.abs(W16.astype(np.float32))
    if scale is not None:
        s = s * scale.astype(np.float32)[None, :]
    rows, K = W16.shape
    mask = np.zeros((rows, K), dtype=np.uint8)
    pos = np.arange(M)
    for r in range(rows):
        for g in range(K // M):
            sg = s[r, g * M:(g + 1) * M]
            order = np.lexsort((pos, -sg))
            mask[r, g * M + order[:N]] = 1
    return mask


@pytest.mark.parametrize("N,M", [(2, 4), (1, 4), (3, 4), (4, 8), (2, 8), (1, 8), (4, 4)])
@pytest.mark.parametrize("scaled", [False, True])
def test_select_matches_numpy_sort(N, M, scaled):
    rng = np.random.default_rng(N * 31 + M + scaled)
    rows, K = 23, 96
    W = (rng.standard_normal((rows, K)) * 0.02).astype(np.float16)
    scale = (rng.uniform(0.1, 10.0, K)).astype(np.float32) if scaled else None
    assert np.array_equal(oracle.select_mask(W, N, M, scale), _np_select(W, N, M, scale))


@pytest.mark.parametrize("N", [1, 2, 3])
def test_every_ordering_of_a_group(N):
    """Distinct magnitudes in every order: the N largest are kept."""
    vals = np.array([0.5, 1.0, 2.0, 4.0], dtype=np.float16)
    perms = list(itertools.permutations(range(4)))
    W = np.stack([vals[list(p)] for p in perms])
    mask = oracle.select_mask(W, N, 4)
    for row, p in zip(mask, perms):
        kept = sorted(vals[list(p)][row.astype(bool)].tolist())
        assert kept == sorted(vals.tolist())[4 - N:]


def test_ties_go_to_the_lower_position():
    W = np.full((2, 8), 0.25, dtype=np.float16)
    W[1, :] = np.array([-0.0, 0.0, 0.0, -0.0, 1, 1, 1, 1], dtype=np.float16)
    m = oracle.select_mask(W, 2, 4)
    assert m.tolist() == [[1, 1, 0, 0, 1, 1, 0, 0], [1, 1, 0, 0, 1, 1, 0, 0]]


def test_scale_changes_the_choice():
    """|w| prefers positions 2 and 3; a large scale on 0 and 1 reverses it."""
    W = np.array([[0.1, 0.2, 0.3, 0.4]], dtype=np.float16)
    assert oracle.select_mask(W, 2, 4).tolist() == [[0, 0, 1, 1]]
    scale = np.array([100.0, 100.0, 1.0, 1.0], dtype=np.float32)
    assert oracle.select_mask(W, 2, 4, scale).tolist() == [[1, 1, 0, 0]]


def test_unit_scale_and_no_scale_agree_with_magnitude_rule():
    rng = np.random.default_rng(9)
    W = (rng.standard_normal((17, 64)) * 0.02).astype(np.float16)
    m0 = oracle.select_mask(W, 2, 4)
    assert np.array_equal(m0, oracle.select_mask(W, 2, 4, np.ones(64, np.float32)))
    assert np.array_equal(m0, oracle.topn_mask(W, 2, 4))
    assert (m0.reshape(17, 16, 4).sum(-1) == 2).all()
