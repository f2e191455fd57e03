"""GPU parity of nm_calib_accumulate (H += X^T X on the tensor cores) against
the oracle's fp64 accumulation, with the tolerance of
oracle.calib_within_tolerance."""
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


def _x(T, K, seed, ld=None):
    x = nm_synth.activations(K, T, seed, True, DEV, ld=ld)  # [T][ld], outlier channels
    return x


@pytest.mark.parametrize("T,K", [(1, 8), (64, 128), (100, 200), (448, 256), (513, 1000),
                                 (2048, 512), (33, 1024), (128, 4096)])
def test_calib_matches_oracle(T, K):
    X = _x(T, K, T + K)
    H0 = torch.randn(K, K, generator=torch.Generator(device=DEV).manual_seed(K), device=DEV)
    H = H0.clone()
    nm.nm_calib_accumulate(X, H)
    torch.cuda.synchronize()
    assert nm.nm_device_errors() == 0
    Href, S = oracle.calib_accumulate(_np16(X), H0.double().cpu().numpy())
    ok = oracle.calib_within_tolerance(H.cpu().numpy(), Href, S)
    assert ok.all(), "%d/%d outside tolerance, first at %s" % (
        (~ok).sum(), ok.size, np.argwhere(~ok)[:3].tolist())


def test_calib_strided_inputs_and_batches_add_up():
    T, K, ldx, ldh = 300, 264, 272, 268
    X = _x(T, K, 5, ld=ldx)
    Hbuf = torch.zeros(K, ldh, device=DEV)
    nm.nm_calib_accumulate(X[:120, :K], Hbuf[:, :K])   # two batches of tokens
    nm.nm_calib_accumulate(X[120:, :K], Hbuf[:, :K])
    torch.cuda.synchronize()
    assert (Hbuf[:, K:] == 0).all()  # the padding columns are never touched
    Href, S = oracle.calib_accumulate(_np16(X[:, :K].contiguous()))
    ok = oracle.calib_within_tolerance(Hbuf[:, :K].cpu().numpy(), Href, S)
    assert ok.all(), (~ok).sum()


def test_calib_large_k_sampled_features():
    """K = 14336 (the down projection's input), 512 decode tokens, checked on
    256 sampled features (rows and columns of H)."""
    T, K = 512, 14336
    X = _x(T, K, 11)
    H = nm.nm_calib_accumulate(X)
    torch.cuda.synchronize()
    assert nm.nm_device_errors() == 0
    F = np.sort(np.random.default_rng(0).choice(K, 256, replace=False))
    Ft = torch.from_numpy(F).to(DEV)
    Href, S = oracle.calib_accumulate(_np16(X[:, Ft].contiguous()))
    Hs = H[Ft][:, Ft].cpu().numpy()
    ok = oracle.calib_within_tolerance(Hs, Href, S)
    assert ok.all(), (~ok).sum()
    # H and its transpose sum the same products (in tiles mirrored across the diagonal)
    assert torch.allclose(H, H.T, rtol=1e-5, atol=1e-3)


def test_calib_graph_capture():
    T, K = 256, 512
    X = _x(T, K, 3)
    H = torch.zeros(K, K, device=DEV)
    nm.nm_calib_accumulate(X, H)  # load before capture
    torch.cuda.synchronize()
    H.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            nm.nm_calib_accumulate(X, H)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    g.replay()  # accumulates twice
    torch.cuda.synchronize()
    Href, S = oracle.calib_accumulate(_np16(X))
    ok = oracle.calib_within_tolerance(H.cpu().numpy(), 2 * Href, 2 * S)
    assert ok.all(), (~ok).sum()
