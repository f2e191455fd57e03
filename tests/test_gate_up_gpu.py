"""GPU parity of nm_spmv_gate_up_silu (h = silu(gate x) * (up x) in one pass
over both matrices) against the oracle's fp64 reference and its derived
error bound (oracle.gate_up_silu)."""
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


def _pair(rows, K, N, M, B, seed):
    Wg = nm_synth.weights(rows, K, seed, DEV)
    Wu = nm_synth.weights(rows, K, seed + 1, DEV)
    mg, mu = nm_synth.topn_mask(Wg, N, M), nm_synth.topn_mask(Wu, N, M)
    x = nm_synth.activations(K, B, seed + 500, True, DEV)
    return Wg, mg, Wu, mu, x


def _check(h, Wg, mg, Wu, mu, x, rows_idx=None):
    if rows_idx is not None:
        it = torch.from_numpy(rows_idx).to(DEV)
        Wg, mg, Wu, mu = Wg[it], mg[it], Wu[it], mu[it]
        h = h[..., it]
    href, bound = oracle.gate_up_silu(_np16(Wg), mg.cpu().numpy(), _np16(Wu), mu.cpu().numpy(),
                                      _np16(x))
    hg = h.detach().double().cpu().numpy().reshape(href.shape)
    ok = np.abs(hg - href) <= bound
    assert ok.all(), "%d/%d outside the bound, first at %s" % (
        (~ok).sum(), ok.size, np.argwhere(~ok)[:3].tolist())


@pytest.mark.parametrize("rows,K,N,M,B", [
    (1, 128, 2, 4, 1), (5, 128, 1, 8, 1), (149, 4096, 2, 4, 1), (300, 4096, 2, 4, 2),
    (77, 1024, 1, 4, 2), (200, 2048, 4, 8, 3), (129, 512, 2, 8, 8), (333, 5120, 2, 4, 4),
    (64, 8192, 2, 4, 8),     # x of 8 vectors exceeds one tile: K tiles with carried sums
    (90, 14336, 4, 8, 1), (40, 2048, 4, 4, 1), (40, 2048, 8, 8, 2)])
@pytest.mark.parametrize("h_dtype", [torch.float16, torch.float32])
def test_gate_up_silu_matches_oracle(rows, K, N, M, B, h_dtype):
    Wg, mg, Wu, mu, x = _pair(rows, K, N, M, B, seed=rows * 7 + K + N + M + B)
    G, U = nm.nm_pack(Wg, mg, N, M), nm.nm_pack(Wu, mu, N, M)
    h = nm.nm_spmv_gate_up_silu(G, U, x if B > 1 else x[0], h_dtype=h_dtype)
    torch.cuda.synchronize()
    assert nm.nm_device_errors() == 0
    _check(h, Wg, mg, Wu, mu, x)


def test_gate_up_silu_llama8b_shape_sampled():
    """The Llama-3.1-8B-shaped gate/up pair (14336 x 4096, 2:4), batch 1,
    checked on sampled rows; also captured in a CUDA graph and replayed."""
    wl = nm_synth.WORKLOADS["llama31_8b_block"]
    rows, K = 14336, 4096
    Wg, mg, Wu, mu, x = _pair(rows, K, 2, 4, 1, seed=2004)
    G, U = nm.nm_pack(Wg, mg, 2, 4), nm.nm_pack(Wu, mu, 2, 4)
    h = torch.full((rows,), float("nan"), dtype=torch.float16, device=DEV)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    nm.nm_spmv_gate_up_silu(G, U, x[0], h)  # load the kernel before capture
    torch.cuda.synchronize()
    h.fill_(float("nan"))
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            nm.nm_spmv_gate_up_silu(G, U, x[0], h)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert nm.nm_device_errors() == 0
    idx = np.sort(np.random.default_rng(0).choice(rows, 256, replace=False))
    _check(h, Wg, mg, Wu, mu, x, rows_idx=idx)
    del wl


def test_gate_up_silu_equals_separate_products():
    """The fused epilogue and silu applied to two separate nm_spmv results
    agree to fp32 rounding (same kernels' sums, different launch)."""
    rows, K = 500, 4096
    Wg, mg, Wu, mu, x = _pair(rows, K, 2, 4, 1, seed=77)
    G, U = nm.nm_pack(Wg, mg, 2, 4), nm.nm_pack(Wu, mu, 2, 4)
    h = nm.nm_spmv_gate_up_silu(G, U, x[0], h_dtype=torch.float32)
    g = nm.nm_spmv(G, x[0], y_dtype=torch.float32)
    u = nm.nm_spmv(U, x[0], y_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = torch.nn.functional.silu(g.double()) * u.double()
    # both within the oracle bound; their difference only from summation order
    _check(h, Wg, mg, Wu, mu, x)
    assert torch.allclose(h.double(), ref, rtol=1e-3, atol=1e-5)


def test_gate_up_silu_empty_and_zero_k():
    G0 = nm.PackedMatrix(torch.empty(0, 64, dtype=torch.float16, device=DEV),
                         torch.empty(0, 4, dtype=torch.int32, device=DEV), 0, 128, 2, 4)
    x = torch.zeros(128, dtype=torch.float16, device=DEV)
    h = torch.empty(0, dtype=torch.float16, device=DEV)
    nm.nm_spmv_gate_up_silu(G0, G0, x, h)
    # K == 0: every sum is empty, h = silu(0) * 0 = 0
    Gk = nm.PackedMatrix(torch.empty(8, 0, dtype=torch.float16, device=DEV),
                         torch.empty(8, 0, dtype=torch.int32, device=DEV), 8, 0, 2, 4)
    h = torch.full((8,), 7.0, dtype=torch.float16, device=DEV)
    nm.nm_spmv_gate_up_silu(Gk, Gk, torch.zeros(8, dtype=torch.float16, device=DEV), h)
    torch.cuda.synchronize()
    assert (h == 0).all()
