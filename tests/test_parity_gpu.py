"""GPU parity: libnm against the CPU oracle, element by element.

nm_pack must equal oracle.pack byte for byte.  nm_spmv / nm_spmv_batched must
satisfy |y - y_ref| <= 1e-3 * sum_k |w_k x_k| + 1e-6 per element, y_ref and
the sum from the oracle in fp64 (fp32 accumulation over K terms plus one
fp16 rounding of y stays well inside this bound).  Inputs come from the
seeded generator (nm_synth) and reach the oracle as host copies; nothing the
oracle reads comes from libnm.
"""
import ctypes

import numpy as np
import pytest
import torch

import nm_synth
import oracle
from sparse_spmv_memory_02_b300 import nm

pytestmark = pytest.mark.gpu
DEV = "cuda"

FAST = [(2, 4), (4, 8), (1, 4), (2, 8), (4, 4), (1, 8), (8, 8)]
GENERIC = [(3, 4), (3, 8), (5, 8), (7, 8)]


def _np16(t):
    return t.detach().cpu().numpy().view(np.uint16)


def _inputs(rows, K, N, M, B, seed, device=DEV):
    W = nm_synth.weights(rows, K, seed, device)
    mask = nm_synth.random_mask(rows, K, N, M, seed + 1, device) if N < M else \
        torch.ones(rows, K, dtype=torch.uint8, device=device)
    x = nm_synth.activations(K, B, seed + 2, True, device) if K else \
        torch.zeros(B, 0, dtype=torch.float16, device=device)
    return W, mask, x


def _pack_and_check(W, mask, N, M):
    A = nm.nm_pack(W, mask, N, M)
    torch.cuda.synchronize()
    ev, em, bad = oracle.pack(_np16(W), mask.cpu().numpy(), N, M)
    assert bad == 0
    assert np.array_equal(_np16(A.values), ev)
    assert np.array_equal(A.masks.cpu().numpy().view(np.uint32), em)
    return A


def _check_y(y, W, mask, x, rows=None):
    """Compare y [B][rows] (or a subset of rows) with the oracle."""
    Wn, mn, xn = _np16(W), mask.cpu().numpy(), _np16(x)
    yr, sr = oracle.spmv_dense(Wn, mn, xn)
    yg = y.detach().double().cpu().numpy().reshape(yr.shape)
    ok = oracle.within_tolerance(yg, yr, sr)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        msg = ["b=%d row=%d gpu=%r ref=%r s=%r" % (b, r, yg[b, r], yr[b, r], sr[b, r])
               for b, r in bad]
        pytest.fail("%d/%d outside tolerance: %s" % ((~ok).sum(), ok.size, "; ".join(msg)))
    return yr, sr


def _guarded(shape, dtype, pad=64):
    """Tensor view with canary regions on both sides (detect stray writes)."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), float("nan") if dtype != torch.int32 else -7,
                     dtype=dtype, device=DEV)
    if dtype == torch.float16:
        buf.view(torch.int16)[:] = 0x7E5A  # distinctive NaN payload
    view = buf[pad:pad + n].view(shape)
    return buf, view, pad


def _guards_intact(buf, pad):
    g = torch.cat([buf[:pad], buf[-pad:]])
    if buf.dtype == torch.float16:
        return bool((g.view(torch.int16) == 0x7E5A).all())
    return bool(torch.isnan(g).all())


# ------------------------------------------------------------------ pack

@pytest.mark.parametrize("N,M", FAST + GENERIC)
@pytest.mark.parametrize("rows,K", [(1, 8), (37, 96), (300, 1000), (65, 4112)])
def test_pack_unpack_bit_exact(N, M, rows, K):
    if K % M:
        pytest.skip("K must be a multiple of M")
    W, mask, _ = _inputs(rows, K, N, M, 1, seed=rows + K + N * 7 + M)
    A = _pack_and_check(W, mask, N, M)
    back = nm.nm_unpack(A)
    torch.cuda.synchronize()
    assert np.array_equal(_np16(back), oracle.unpack(_np16(A.values),
                                                     A.masks.cpu().numpy().view(np.uint32),
                                                     K, N, M))


def test_pack_special_bit_patterns():
    rows, K, N, M = 4, 64, 2, 4
    bits = np.array([0x8000, 0x0000, 0x7C00, 0xFC00, 0x0001, 0x7BFF, 0x7E01, 0x3C00],
                    dtype=np.uint16)
    W = torch.from_numpy(np.tile(bits, (rows, K // 8)).view(np.float16)).to(DEV)
    mask = nm_synth.random_mask(rows, K, N, M, 3, DEV)
    _pack_and_check(W, mask, N, M)


def test_pack_golden_examples():
    from tests.golden_examples import load_examples
    for ex in load_examples():
        W = torch.from_numpy(ex.W_arr.copy()).to(DEV)
        mask = torch.from_numpy(ex.mask_arr.copy()).to(DEV)
        if ex.bad:
            with pytest.raises(nm.NMError) as e:
                nm.nm_pack(W, mask, ex.N, ex.M)
            assert e.value.status == nm.NM_ERR_BAD_MASK
            continue
        A = nm.nm_pack(W, mask, ex.N, ex.M)
        assert np.array_equal(_np16(A.values), ex.values_arr.view(np.uint16))
        assert np.array_equal(A.masks.cpu().numpy().view(np.uint32), ex.masks_arr)
        for x, y, s in ex.cases:
            xt = torch.from_numpy(x.copy()).to(DEV)
            yg = nm.nm_spmv(A, xt, y_dtype=torch.float32)
            assert np.array_equal(yg.double().cpu().numpy(), np.array(y))


@pytest.mark.parametrize("where", ["excess", "missing", "empty"])
def test_pack_rejects_bad_masks(where):
    rows, K, N, M = 16, 128, 2, 4
    W, mask, _ = _inputs(rows, K, N, M, 1, seed=5)
    mask = mask.clone()
    if where == "excess":
        mask[3, 8:12] = 1
    elif where == "missing":
        mask[15, 124:128] = torch.tensor([0, 0, 1, 0], dtype=torch.uint8)
    else:
        mask[0, 0:4] = 0
    with pytest.raises(nm.NMError) as e:
        nm.nm_pack(W, mask, N, M)
    assert e.value.status == nm.NM_ERR_BAD_MASK
    assert "1 group" in str(e.value)


# ------------------------------------------------------------------ spmv

BATCH_CASES = [(1, torch.float16), (1, torch.float32), (2, torch.float32), (3, torch.float16),
               (5, torch.float32), (8, torch.float16)]


@pytest.mark.parametrize("N,M", FAST + GENERIC)
@pytest.mark.parametrize("rows,K", [(1, 64), (37, 1024), (300, 3000), (129, 4112)])
@pytest.mark.parametrize("B,ydt", BATCH_CASES, ids=lambda v: str(v))
def test_spmv_matches_oracle(N, M, rows, K, B, ydt):
    if K % M:
        pytest.skip("K must be a multiple of M")
    W, mask, x = _inputs(rows, K, N, M, B, seed=rows * 3 + K + B + N * 11 + M)
    A = _pack_and_check(W, mask, N, M)
    ybuf, y, pad = _guarded((B, rows), ydt)
    if B == 1:
        nm.nm_spmv(A, x[0], y[0])
    else:
        nm.nm_spmv_batched(A, x, y)
    torch.cuda.synchronize()
    assert _guards_intact(ybuf, pad)
    _check_y(y, W, mask, x)


@pytest.mark.parametrize("N,M,K,B", [(2, 4, 40960, 1), (2, 4, 17408, 2), (2, 4, 14336, 8),
                                     (4, 8, 40960, 1), (1, 4, 81920, 1), (2, 8, 36864, 3)])
def test_spmv_several_k_tiles(N, M, K, B):
    """K long enough that a row needs more than one K tile of the block."""
    rows = 77
    W, mask, x = _inputs(rows, K, N, M, B, seed=K + B)
    A = _pack_and_check(W, mask, N, M)
    y = nm.nm_spmv_batched(A, x, y_dtype=torch.float32)
    torch.cuda.synchronize()
    _check_y(y, W, mask, x)


@pytest.mark.parametrize("N,M", FAST + [(3, 4)])
def test_spmv_small_integers_exact(N, M):
    rows, K, B = 203, 2048, 4
    W = nm_synth.small_int_weights(rows, K, seed=N * M, device=DEV)
    mask = nm_synth.random_mask(rows, K, N, M, 9, DEV) if N < M else \
        torch.ones(rows, K, dtype=torch.uint8, device=DEV)
    x = nm_synth.small_int_weights(B, K, seed=99, device=DEV)
    A = _pack_and_check(W, mask, N, M)
    y = nm.nm_spmv_batched(A, x, y_dtype=torch.float32)
    yr, _ = oracle.spmv_dense(_np16(W), mask.cpu().numpy(), _np16(x))
    assert np.array_equal(y.double().cpu().numpy(), yr)


def test_spmv_strided_batch():
    rows, K, N, M, B = 150, 2048, 2, 4, 4
    W, mask, _ = _inputs(rows, K, N, M, B, seed=17)
    A = _pack_and_check(W, mask, N, M)
    xs = nm_synth.activations(K, B, seed=18, device=DEV, ld=K + 64)   # ldx = K + 64
    ybig = torch.full((B, rows + 50), 123.0, dtype=torch.float32, device=DEV)
    y = ybig[:, :rows]                                                  # ldy = rows + 50
    nm.nm_spmv_batched(A, xs[:, :K], y)
    torch.cuda.synchronize()
    assert torch.all(ybig[:, rows:] == 123.0)
    _check_y(y, W, mask, xs[:, :K].contiguous())


def test_spmv_empty_and_degenerate():
    # K == 0: y is zeroed (strided, batch 3)
    A = nm.PackedMatrix(torch.empty(5, 0, dtype=torch.float16, device=DEV),
                        torch.empty(5, 0, dtype=torch.int32, device=DEV), 5, 0, 2, 4)
    ybig = torch.full((3, 8), 7.0, dtype=torch.float32, device=DEV)
    x = torch.zeros(3, 8, dtype=torch.float16, device=DEV)
    nm.nm_spmv_batched(A, x, ybig[:, :5])
    torch.cuda.synchronize()
    assert torch.all(ybig[:, :5] == 0) and torch.all(ybig[:, 5:] == 7.0)
    # rows == 0: nothing happens
    W = torch.empty(0, 64, dtype=torch.float16, device=DEV)
    A0 = nm.nm_pack(W, torch.empty(0, 64, dtype=torch.uint8, device=DEV), 2, 4)
    nm.nm_spmv(A0, torch.zeros(64, dtype=torch.float16, device=DEV))
    # K == M: one group per row
    Wt, mask, x = _inputs(33, 4, 2, 4, 1, seed=4)
    A1 = _pack_and_check(Wt, mask, 2, 4)
    _check_y(nm.nm_spmv(A1, x[0], y_dtype=torch.float32)[None], Wt, mask, x)


def test_spmv_rejects_misaligned_x():
    rows, K = 16, 256
    W, mask, x = _inputs(rows, K, 2, 4, 1, seed=6)
    A = nm.nm_pack(W, mask, 2, 4)
    xb = torch.zeros(K + 8, dtype=torch.float16, device=DEV)
    with pytest.raises(nm.NMError) as e:
        nm.nm_spmv(A, xb[1:K + 1])
    assert e.value.status == nm.NM_ERR_INVALID_ARG


def test_spmv_cuda_graph_capture_and_replay():
    rows, K, N, M = 512, 4096, 2, 4
    W, mask, x = _inputs(rows, K, N, M, 1, seed=8)
    A = _pack_and_check(W, mask, N, M)
    y = torch.empty(rows, dtype=torch.float32, device=DEV)
    nm.nm_spmv(A, x[0], y)  # warm-up outside capture
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            nm.nm_spmv(A, x[0], y)
            # pack synchronises and must refuse a capturing stream
            with pytest.raises(nm.NMError):
                nm.nm_pack(W, mask, N, M)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    y1 = y.clone()
    _check_y(y1[None], W, mask, x)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y1)  # deterministic


def test_spmv_is_deterministic():
    rows, K = 1000, 14336
    W, mask, x = _inputs(rows, K, 2, 4, 2, seed=12)
    A = nm.nm_pack(W, mask, 2, 4)
    y1 = nm.nm_spmv_batched(A, x, y_dtype=torch.float32)
    y2 = nm.nm_spmv_batched(A, x, y_dtype=torch.float32)
    assert torch.equal(y1, y2)


def test_raw_c_abi_call():
    """nm_spmv through ctypes with raw device pointers and a non-default stream."""
    rows, K, N, M = 96, 512, 2, 4
    W, mask, x = _inputs(rows, K, N, M, 1, seed=10)
    A = nm.nm_pack(W, mask, N, M)
    y = torch.empty(rows, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    desc = nm.nm_matrix(rows, K, N, M, A.values.data_ptr(), A.masks.data_ptr())
    torch.cuda.synchronize()
    st = nm.lib().nm_spmv(ctypes.byref(desc), x.data_ptr(), y.data_ptr(), nm.NM_F32,
                          s.cuda_stream)
    assert st == nm.NM_OK
    s.synchronize()
    _check_y(y[None], W, mask, x)
