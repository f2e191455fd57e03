"""Pins for the CPU oracle, independent of the oracle's own code.

Each check reaches the expected value by a different route than the oracle's
loops: numpy's binary16 conversion, numpy boolean-mask gathers and bit
packing, a dense fp64 numpy matmul of the masked matrix, hand-worked examples
(tests/golden/), closed forms and invariants.  A dropped term, a wrong bit
order, a shifted value index or a transposed operand in the oracle fails at
least one of them.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import scalar_twin
from tests.golden_examples import load_examples

PATTERNS = [(2, 4), (4, 8), (1, 4), (2, 8), (3, 4), (1, 8), (4, 4), (8, 8), (5, 8)]


def _rand_case(rows, K, N, M, seed, B=1):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((rows, K)) * 0.02).astype(np.float16)
    mask = np.zeros((rows, K // M, M), dtype=np.uint8)
    for r in range(rows):
        for g in range(K // M):
            mask[r, g, rng.choice(M, N, replace=False)] = 1
    mask = mask.reshape(rows, K)
    x = rng.standard_normal((B, K)).astype(np.float16)
    return W, mask, x


def _np_expected_pack(W, mask):
    """Library route: boolean gather (row-major, increasing k) and
    little-endian bit packing."""
    rows, K = W.shape
    keep = mask.astype(bool)
    vals = np.stack([W[r][keep[r]] for r in range(rows)]).view(np.uint16)
    nbytes = ((K + 31) // 32) * 4
    packed = np.packbits(keep, axis=1, bitorder="little")
    padded = np.zeros((rows, nbytes), dtype=np.uint8)
    padded[:, :packed.shape[1]] = packed
    words = padded.view("<u4")
    return vals, words


def _np_expected_y(W, mask, x):
    Wm = np.where(mask.astype(bool), W.astype(np.float64), 0.0)
    P = Wm[None, :, :] * x.astype(np.float64)[:, None, :]
    return P.sum(axis=2), np.abs(P).sum(axis=2)


# ---------------------------------------------------------------- binary16

def test_half_decode_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signs of zero are kept
    assert np.signbit(got[0x8000]) and not np.signbit(got[0x0000])


# ---------------------------------------------------------------- golden

@pytest.mark.parametrize("ex", load_examples(), ids=lambda e: e.name)
def test_pack_matches_hand_worked_examples(ex):
    W, mask = ex.W_arr, ex.mask_arr
    values, masks, bad = oracle.pack(W, mask, ex.N, ex.M)
    assert bad == ex.bad
    assert np.array_equal(values, ex.values_arr.view(np.uint16))
    assert np.array_equal(masks, ex.masks_arr)
    K = W.shape[1]
    for x, y, s in ex.cases:
        yd, sd = oracle.spmv_dense(W, mask, x)
        yp, sp = oracle.spmv_packed(values, masks, K, ex.N, ex.M, x)
        assert np.array_equal(yd[0], np.array(y)), (yd, y)
        assert np.array_equal(sd[0], np.array(s))
        assert np.array_equal(yp[0], np.array(y))
        assert np.array_equal(sp[0], np.array(s))


@pytest.mark.parametrize("ex", [e for e in load_examples() if e.bad == 0],
                         ids=lambda e: e.name)
def test_unpack_matches_hand_worked_examples(ex):
    W, mask = ex.W_arr, ex.mask_arr
    back = oracle.unpack(ex.values_arr, ex.masks_arr, W.shape[1], ex.N, ex.M)
    expect = np.where(mask.astype(bool), W.view(np.uint16), np.uint16(0))
    assert np.array_equal(back, expect)


# ---------------------------------------------------------------- pack

@pytest.mark.parametrize("N,M", [(2, 4), (4, 8)])
def test_pack_every_group_mask_exhaustively(N, M):
    """All C(M,N) masks of a group (6 for 2:4, 70 for 4:8), one per row,
    with distinct weights per position."""
    combos = list(itertools.combinations(range(M), N))
    rows = len(combos)
    K = 4 * M  # four groups per row; the tested mask sits in group 1
    W = (np.arange(rows * K, dtype=np.float64).reshape(rows, K) / 8 + 1).astype(np.float16)
    mask = np.zeros((rows, K), dtype=np.uint8)
    for r, c in enumerate(combos):
        for g in range(K // M):
            sel = c if g == 1 else tuple(range(N))
            for q in sel:
                mask[r, g * M + q] = 1
    values, masks, bad = oracle.pack(W, mask, N, M)
    ev, em = _np_expected_pack(W, mask)
    assert bad == 0
    assert np.array_equal(values, ev)
    assert np.array_equal(masks, em)


@pytest.mark.parametrize("N,M", PATTERNS)
@pytest.mark.parametrize("rows,K", [(1, 8), (3, 24), (17, 96), (33, 200), (64, 256)])
def test_pack_matches_numpy_gather_and_bitpack(N, M, rows, K):
    if K % M:
        pytest.skip("K must be a multiple of M")
    W, mask, _ = _rand_case(rows, K, N, M, seed=rows * 1000 + K + 10 * N + M)
    values, masks, bad = oracle.pack(W, mask, N, M)
    ev, em = _np_expected_pack(W, mask)
    assert bad == 0
    assert values.shape == (rows, K * N // M)
    assert np.array_equal(values, ev)
    assert np.array_equal(masks, em)
    # exactly N ones per group, read back from the packed words
    bits = np.unpackbits(masks.view(np.uint8), axis=1, bitorder="little")[:, :K]
    assert np.all(bits.reshape(rows, K // M, M).sum(-1) == N)
    assert np.all(bits[:, K:] == 0) if bits.shape[1] > K else True


def test_pack_counts_invalid_groups():
    rng = np.random.default_rng(7)
    rows, K, N, M = 5, 64, 2, 4
    W, mask, _ = _rand_case(rows, K, N, M, seed=3)
    mask = mask.copy()
    mask[0, 0:4] = [1, 1, 1, 0]      # N+1 ones
    mask[2, 8:12] = [0, 0, 0, 1]     # N-1 ones
    mask[4, 60:64] = [0, 0, 0, 0]    # none
    _, _, bad = oracle.pack(W, mask, N, M)
    assert bad == 3
    _, _, bad = oracle.pack(W, np.ones_like(mask), N, M)
    assert bad == rows * K // M
    del rng


def test_pack_copies_bits_of_special_values():
    rows, K, N, M = 1, 8, 2, 4
    W = np.array([[0x8000, 0x7C00, 0xFC00, 0x0001, 0x7BFF, 0x8001, 0x3C00, 0x0000]],
                 dtype=np.uint16)
    mask = np.array([[1, 1, 0, 0, 0, 1, 0, 1]], dtype=np.uint8)
    values, masks, bad = oracle.pack(W, mask, N, M)
    assert bad == 0
    assert values.tolist() == [[0x8000, 0x7C00, 0x8001, 0x0000]]
    assert masks.tolist() == [[0b10100011]]


@pytest.mark.parametrize("N,M", PATTERNS)
def test_unpack_inverts_pack(N, M):
    rows, K = 19, 8 * M * 3
    W, mask, _ = _rand_case(rows, K, N, M, seed=N * 31 + M)
    values, masks, _ = oracle.pack(W, mask, N, M)
    back = oracle.unpack(values, masks, K, N, M)
    expect = np.where(mask.astype(bool), W.view(np.uint16), np.uint16(0))
    assert np.array_equal(back, expect)


# ---------------------------------------------------------------- spmv

@pytest.mark.parametrize("N,M", PATTERNS)
@pytest.mark.parametrize("B", [1, 2, 3, 8])
def test_spmv_matches_dense_numpy_matmul(N, M, B):
    rows, K = 37, 16 * M
    W, mask, x = _rand_case(rows, K, N, M, seed=B * 100 + N * 10 + M, B=B)
    ey, es = _np_expected_y(W, mask, x)
    yd, sd = oracle.spmv_dense(W, mask, x)
    values, masks, _ = oracle.pack(W, mask, N, M)
    yp, sp = oracle.spmv_packed(values, masks, K, N, M, x)
    scale = np.abs(es) + 1e-300
    assert np.all(np.abs(yd - ey) <= 1e-12 * scale)
    assert np.all(np.abs(sd - es) <= 1e-12 * scale)
    # same k order in both oracle routes: identical results
    assert np.array_equal(yd, yp) and np.array_equal(sd, sp)


def test_spmv_all_ones_gives_kept_row_sums():
    rows, K, N, M = 24, 128, 2, 4
    W, mask, _ = _rand_case(rows, K, N, M, seed=11)
    x = np.ones((1, K), dtype=np.float16)
    y, _ = oracle.spmv_dense(W, mask, x)
    keep = mask.astype(bool)
    sums = np.array([W[r][keep[r]].astype(np.float64).sum() for r in range(rows)])
    assert np.allclose(y[0], sums, rtol=1e-13, atol=0)


def test_spmv_one_hot_picks_a_column_of_the_masked_matrix():
    rows, K, N, M = 16, 64, 4, 8
    W, mask, _ = _rand_case(rows, K, N, M, seed=12)
    values, masks, _ = oracle.pack(W, mask, N, M)
    for k in (0, 1, 7, 31, 32, 63):
        x = np.zeros((1, K), dtype=np.float16)
        x[0, k] = 1
        y, _ = oracle.spmv_packed(values, masks, K, N, M, x)
        col = np.where(mask[:, k] != 0, W[:, k].astype(np.float64), 0.0)
        assert np.array_equal(y[0], col)


@pytest.mark.parametrize("N,M", [(2, 4), (4, 8), (1, 4), (2, 8)])
def test_spmv_small_integers_are_exact(N, M):
    rng = np.random.default_rng(N + M)
    rows, K = 40, 32 * M
    W = rng.integers(-8, 9, size=(rows, K)).astype(np.float16)
    _, mask, _ = _rand_case(rows, K, N, M, seed=5)
    x = rng.integers(-8, 9, size=(3, K)).astype(np.float16)
    Wi = np.where(mask.astype(bool), W.astype(np.int64), 0)
    ey = x.astype(np.int64) @ Wi.T
    values, masks, _ = oracle.pack(W, mask, N, M)
    y, _ = oracle.spmv_packed(values, masks, K, N, M, x)
    assert np.array_equal(y, ey.astype(np.float64))


def test_spmv_is_linear_in_x():
    rows, K, N, M = 30, 256, 2, 4
    W, mask, x = _rand_case(rows, K, N, M, seed=21, B=2)
    a = np.float16(0.5)
    x3 = (a * x[0].astype(np.float32) + x[1].astype(np.float32)).astype(np.float16)
    # use the fp16-rounded combination and compare against the fp64 identity
    y, s = oracle.spmv_dense(W, mask, x)
    y3, s3 = oracle.spmv_dense(W, mask, x3[None, :])
    # rounding of x3 to fp16 perturbs each product by <= 2^-11 relative
    lin = 0.5 * y[0] + y[1]
    bound = 2.0 ** -11 * (0.5 * s[0] + s[1]) + 1e-12
    assert np.all(np.abs(y3[0] - lin) <= bound)


@pytest.mark.parametrize("M", [4, 8])
def test_dense_pattern_equals_plain_matvec(M):
    rows, K = 21, 64
    rng = np.random.default_rng(M)
    W = rng.standard_normal((rows, K)).astype(np.float16)
    mask = np.ones((rows, K), dtype=np.uint8)
    x = rng.standard_normal((1, K)).astype(np.float16)
    values, masks, bad = oracle.pack(W, mask, M, M)
    assert bad == 0 and np.array_equal(values, W.view(np.uint16))
    y, _ = oracle.spmv_packed(values, masks, K, M, M, x)
    ref = W.astype(np.float64) @ x[0].astype(np.float64)
    assert np.allclose(y[0], ref, rtol=1e-13, atol=1e-15)


def test_spmv_row_range_and_strides():
    rows, K, N, M = 50, 96, 2, 4
    W, mask, x = _rand_case(rows, K, N, M, seed=9, B=2)
    xpad = np.zeros((2, K + 8), dtype=np.float16)
    xpad[:, :K] = x
    y_all, _ = oracle.spmv_dense(W, mask, x)
    y_part, _ = oracle.spmv_dense(W, mask, xpad, row_begin=10, row_end=20)
    assert np.array_equal(y_part[:, 10:20], y_all[:, 10:20])
    assert np.all(np.isnan(y_part[:, :10])) and np.all(np.isnan(y_part[:, 20:]))


# ---------------------------------------------------------------- twins

@pytest.mark.parametrize("N,M", [(2, 4), (4, 8), (1, 4), (2, 8), (3, 4)])
def test_c_oracle_agrees_with_python_scalar_twin(N, M):
    rows, K = 5, 8 * M
    W, mask, x = _rand_case(rows, K, N, M, seed=77 + N, B=2)
    Wb = W.view(np.uint16).tolist()
    vals_py, words_py, bad_py = scalar_twin.pack(Wb, mask.tolist(), N, M)
    values, masks, bad = oracle.pack(W, mask, N, M)
    assert bad == bad_py == 0
    assert values.tolist() == vals_py and masks.tolist() == words_py
    assert oracle.unpack(values, masks, K, N, M).tolist() == scalar_twin.unpack(
        vals_py, words_py, K, N, M)
    y_py, s_py = scalar_twin.spmv(vals_py, words_py, K, N, M, x.view(np.uint16).tolist())
    y, s = oracle.spmv_packed(values, masks, K, N, M, x)
    assert np.array_equal(y, np.array(y_py)) and np.array_equal(s, np.array(s_py))


def test_topn_mask_rule():
    """N largest |w| per group, ties to the lower k; checked against a sort."""
    rng = np.random.default_rng(3)
    rows, K = 12, 64
    W = rng.integers(-3, 4, size=(rows, K)).astype(np.float16)  # many ties
    W[0, 0:4] = [np.float16(-0.0), 0.0, 0.0, -0.0]
    for N, M in [(2, 4), (4, 8), (1, 4), (2, 8)]:
        mask = oracle.topn_mask(W, N, M)
        a = np.abs(W.astype(np.float64)).reshape(rows, K // M, M)
        ref = np.zeros_like(a, dtype=np.uint8)
        for r in range(rows):
            for g in range(K // M):
                order = sorted(range(M), key=lambda q: (-a[r, g, q], q))
                ref[r, g, order[:N]] = 1
        assert np.array_equal(mask, ref.reshape(rows, K))
