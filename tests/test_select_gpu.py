"""GPU parity of nm_select_mask and nm_prune_pack against the oracle: the
mask bit-exact (both sides decide with the same fp32 scores), the packed
arrays bit-exact against the oracle's pack of the oracle's mask."""
import numpy as np
import pytest
import torch

import nm_synth
import oracle
from sparse_spmv_memory_02_b300 import nm

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _np16(t):
    return t.detach().cpu().numpy().view(np.uint16)


def _inputs(rows, K, seed, scaled, ties=False):
    if ties:  # small integers: many equal magnitudes within a group
        W = nm_synth.small_int_weights(rows, K, seed, -3, 3, DEV)
    else:
        W = nm_synth.weights(rows, K, seed, DEV)
    scale = None
    if scaled:
        g = torch.Generator(device=DEV).manual_seed(seed + 1)
        scale = torch.rand(K, generator=g, device=DEV) * 4 + 0.05
        if ties:
            scale = torch.round(scale)  # integer scales keep products exact and tied
    return W, scale


SHAPES = [(1, 8), (7, 40), (149, 4096), (300, 5120), (64, 14336), (33, 1000), (5, 24)]


@pytest.mark.parametrize("N,M", [(2, 4), (1, 4), (3, 4), (4, 8), (2, 8), (1, 8), (4, 4), (5, 8)])
@pytest.mark.parametrize("scaled", [False, True])
@pytest.mark.parametrize("ties", [False, True])
def test_select_mask_bit_exact(N, M, scaled, ties):
    for rows, K in SHAPES:
        if K % M:
            continue
        W, scale = _inputs(rows, K, rows + K + N + M, scaled, ties)
        mask = nm.nm_select_mask(W, N, M, scale)
        torch.cuda.synchronize()
        ref = oracle.select_mask(_np16(W), N, M, None if scale is None else scale.cpu().numpy())
        assert np.array_equal(mask.cpu().numpy(), ref), (rows, K)


@pytest.mark.parametrize("N,M", [(2, 4), (1, 4), (4, 8), (2, 8), (1, 8), (3, 4), (8, 8)])
@pytest.mark.parametrize("scaled", [False, True])
def test_prune_pack_bit_exact(N, M, scaled):
    for rows, K in SHAPES:
        if K % M:
            continue
        W, scale = _inputs(rows, K, rows * 3 + K + N, scaled, ties=(rows % 2 == 1))
        A = nm.nm_prune_pack(W, N, M, scale)
        torch.cuda.synchronize()
        Wn = _np16(W)
        mref = oracle.select_mask(Wn, N, M, None if scale is None else scale.cpu().numpy())
        vref, wref, bad = oracle.pack(Wn, mref, N, M)
        assert bad == 0
        assert np.array_equal(_np16(A.values), vref), (rows, K)
        assert np.array_equal(A.masks.cpu().numpy().view(np.uint32), wref), (rows, K)


def test_prune_pack_equals_select_then_pack_and_feeds_spmv():
    W, scale = _inputs(1000, 4096, 5, True)
    A = nm.nm_prune_pack(W, 2, 4, scale)
    B = nm.nm_pack(W, nm.nm_select_mask(W, 2, 4, scale), 2, 4)
    torch.cuda.synchronize()
    assert torch.equal(A.values.view(torch.int16), B.values.view(torch.int16))
    assert torch.equal(A.masks, B.masks)
    x = nm_synth.activations(4096, 1, 6, True, DEV)[0]
    assert torch.equal(nm.nm_spmv(A, x), nm.nm_spmv(B, x))


def test_select_graph_capture_and_empty():
    W, _ = _inputs(64, 512, 3, False)
    mask = torch.empty(64, 512, dtype=torch.uint8, device=DEV)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            nm.nm_select_mask(W, 2, 4, mask=mask)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(mask.cpu().numpy(), oracle.select_mask(_np16(W), 2, 4))
    e = torch.empty(0, 64, dtype=torch.float16, device=DEV)
    assert nm.nm_select_mask(e, 2, 4).shape == (0, 64)
    assert nm.nm_prune_pack(e, 2, 4).rows == 0


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("rows,batch", [(4096, 1), (4096, 4), (8192, 8)],
                         ids=["row_kernel_b1", "row_kernel_b4", "tensor_cores_b8"])
def test_prune_pack_then_spmv_without_sync(graph, rows, batch):
    """nm_prune_pack followed at once by an SpMV on the same stream (no host
    synchronisation, eager or in one CUDA graph): the SpMV, whose weight
    copies may start before its dependence wait (the row kernel, and at batch
    8 with 56 rows per SM the sparse tensor-core product), must read the
    arrays the prune-pack just wrote, not what the buffers held before."""
    K, N, M = 4096, 2, 4
    W, scale = _inputs(rows, K, 11, True)
    W_old, _ = _inputs(rows, K, 12, False)
    A = nm.nm_prune_pack(W_old, N, M)  # the buffers first hold another matrix
    x = nm_synth.activations(K, batch, 13, True, DEV)
    y = torch.empty(batch, rows, dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()

    def run():
        nm.nm_prune_pack(W, N, M, scale, values=A.values, masks=A.masks)
        nm.nm_spmv_batched(A, x, y)

    if graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                run()
        torch.cuda.current_stream().wait_stream(side)
        nm.nm_prune_pack(W_old, N, M, values=A.values, masks=A.masks)  # stale again
        g.replay()
    else:
        run()
    torch.cuda.synchronize()
    Wn = _np16(W)
    mref = oracle.select_mask(Wn, N, M, scale.cpu().numpy())
    pick = np.arange(0, rows, 7)  # every 7th row against the oracle
    yr, sr = oracle.spmv_dense(Wn[pick], mref[pick], _np16(x))
    assert oracle.within_tolerance(y[:, pick].double().cpu().numpy(), yr, sr).all()
    assert nm.nm_device_errors() == 0
