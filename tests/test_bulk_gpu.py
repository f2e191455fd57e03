"""GPU parity of the bulk-staged SpMV kernels (the path every pattern with
8 % N == 0 and K a multiple of 128 takes: the row-per-warp kernel at batch 1
and 2, the chunk-column kernel at larger batches) against the CPU oracle.

The shapes stress the kernel's schedule: fewer rows than CTAs, row counts
that leave a ragged last stage, K tiles that do not divide the row, every
batch size, and forced tunings (run in child processes, because the tuning
is read once per process) that make rows span several K tiles, shrink the
ring to two slots or one row per stage, and switch programmatic dependent
launch off.  Consecutive dependent calls (the output of one call is the
input of the next) check that a call reads x only after the previous kernel
has written it.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import nm_synth
import oracle
from sparse_spmv_memory_02_b300 import nm

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FAST = [(2, 4), (4, 8), (1, 4), (2, 8), (4, 4), (1, 8), (8, 8)]


def _np16(t):
    return t.detach().cpu().numpy().view(np.uint16)


def _case(rows, K, N, M, B, seed):
    W = nm_synth.weights(rows, K, seed, DEV)
    mask = nm_synth.topn_mask(W, N, M)
    x = nm_synth.activations(K, B, seed + 500, True, DEV)
    return W, mask, x


def _check(y, W, mask, x):
    yr, sr = oracle.spmv_dense(_np16(W), mask.cpu().numpy(), _np16(x))
    yg = y.detach().double().cpu().numpy().reshape(yr.shape)
    ok = oracle.within_tolerance(yg, yr, sr)
    assert ok.all(), "%d/%d outside tolerance, first at %s" % (
        (~ok).sum(), ok.size, np.argwhere(~ok)[:3].tolist())


@pytest.mark.parametrize("N,M", FAST)
@pytest.mark.parametrize("rows,K", [(1, 128), (7, 1024), (149, 4096), (300, 5120),
                                    (600, 14336)])
@pytest.mark.parametrize("B", [1, 2, 3, 5, 8])
def test_bulk_matches_oracle(N, M, rows, K, B):
    W, mask, x = _case(rows, K, N, M, B, seed=rows + K + 13 * N + M + 101 * B)
    A = nm.nm_pack(W, mask, N, M)
    ydt = torch.float32 if B % 2 else torch.float16
    y = torch.full((B, rows), float("nan"), dtype=ydt, device=DEV)
    if B == 1:
        nm.nm_spmv(A, x[0], y[0])
    else:
        nm.nm_spmv_batched(A, x, y)
    torch.cuda.synchronize()
    _check(y, W, mask, x)


def test_bulk_model_shapes_sampled_rows():
    """Decode-layer shapes of the 8B block at batch 1, checked on a sample of
    rows (the oracle computes those rows only)."""
    g = np.random.default_rng(0)
    for rows, K in [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]:
        W, mask, x = _case(rows, K, 2, 4, 1, seed=rows + K)
        A = nm.nm_pack(W, mask, 2, 4)
        y = nm.nm_spmv(A, x[0], y_dtype=torch.float16)
        torch.cuda.synchronize()
        pick = np.sort(g.choice(rows, 256, replace=False))
        idx = torch.from_numpy(pick).to(DEV)
        _check(y[idx][None], W[idx], mask[idx], x)
    assert nm.nm_device_errors() == 0


def test_dependent_chain_reads_x_after_previous_call():
    """y_i = A_i y_{i-1}: each call's x is the previous call's output.  The
    chain run back to back must equal the same calls run one at a time with a
    full synchronisation between them (the kernel is deterministic)."""
    K = 4096
    mats, bufs = [], [nm_synth.activations(K, 1, 7, True, DEV)[0] * 0.05]
    for i in range(12):
        W = nm_synth.weights(K, K, 900 + i, DEV, std=0.02)
        mats.append(nm.nm_pack(W, nm_synth.topn_mask(W, 2, 4), 2, 4))
        bufs.append(torch.full((K,), float("nan"), dtype=torch.float16, device=DEV))
    torch.cuda.synchronize()
    for i, A in enumerate(mats):
        nm.nm_spmv(A, bufs[i], bufs[i + 1])
    torch.cuda.synchronize()
    chained = [b.clone() for b in bufs]
    for i, A in enumerate(mats):
        out = torch.full((K,), float("nan"), dtype=torch.float16, device=DEV)
        nm.nm_spmv(A, chained[i], out)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), chained[i + 1].view(torch.int16)), i
    assert torch.isfinite(chained[-1].float()).all()


def test_dependent_chain_in_cuda_graph():
    K, rows = 2048, 2048
    W1 = nm_synth.weights(rows, K, 31, DEV)
    W2 = nm_synth.weights(rows, rows, 32, DEV)
    A1 = nm.nm_pack(W1, nm_synth.topn_mask(W1, 2, 4), 2, 4)
    A2 = nm.nm_pack(W2, nm_synth.topn_mask(W2, 2, 4), 2, 4)
    x = nm_synth.activations(K, 1, 33, True, DEV)[0]
    h = torch.empty(rows, dtype=torch.float16, device=DEV)
    y = torch.empty(rows, dtype=torch.float32, device=DEV)
    nm.nm_spmv(A1, x, h)
    nm.nm_spmv(A2, h, y)
    torch.cuda.synchronize()
    ref = y.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            nm.nm_spmv(A1, x, h)
            nm.nm_spmv(A2, h, y)
    for _ in range(3):
        h.fill_(float("nan"))
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref)


# ------------------------------------------------------------------ groups

def _group_case(shapes, K, N, M, B, shared_x, seed):
    mats, Ws, masks, xs = [], [], [], []
    x0 = nm_synth.activations(K, B, seed + 500, True, DEV)
    for i, rows in enumerate(shapes):
        W = nm_synth.weights(rows, K, seed + i, DEV)
        mask = nm_synth.topn_mask(W, N, M)
        Ws.append(W)
        masks.append(mask)
        mats.append(nm.nm_pack(W, mask, N, M))
        xs.append(x0 if shared_x else nm_synth.activations(K, B, seed + 600 + i, True, DEV))
    return mats, Ws, masks, xs


@pytest.mark.parametrize("shapes,K,N,M,B,shared", [
    ((4096, 1024, 1024), 4096, 2, 4, 1, True),     # q/k/v of the 8B block
    ((700, 300, 1), 4096, 2, 4, 1, False),
    ((1500, 1500), 4096, 2, 4, 2, True),             # gate/up, batch 2
    ((333, 77, 250, 4, 5, 6, 7, 900), 1024, 4, 8, 1, False),  # 8 matrices
    ((512, 640), 14336, 2, 4, 1, True),              # rows span several K tiles
    ((300, 200), 5120, 1, 4, 2, False),
])
def test_group_matches_oracle(shapes, K, N, M, B, shared):
    mats, Ws, masks, xs = _group_case(shapes, K, N, M, B, shared, seed=sum(shapes) + K + B)
    xin = [x[0] for x in xs] if B == 1 else xs
    ys = [torch.full((A.rows,) if B == 1 else (B, A.rows), float("nan"),
                     dtype=torch.float32, device=DEV) for A in mats]
    nm.nm_spmv_group(mats, xin, ys)
    torch.cuda.synchronize()
    for y, W, mask, x in zip(ys, Ws, masks, xs):
        _check(y if B > 1 else y[None], W, mask, x)
    assert nm.nm_device_errors() == 0


@pytest.mark.parametrize("K,B", [(4112, 1), (1024, 3), (4096, 8)])
def test_group_falls_back_to_single_launches(K, B):
    """Shapes the fused launch does not take (K not a multiple of 128, batch
    above 2) still give every product."""
    mats, Ws, masks, xs = _group_case((100, 37, 260), K, 2, 4, B, False, seed=K + B)
    ys = nm.nm_spmv_group(mats, xs if B > 1 else [x[0] for x in xs], y_dtype=torch.float32)
    torch.cuda.synchronize()
    for y, W, mask, x in zip(ys, Ws, masks, xs):
        _check(y if B > 1 else y[None], W, mask, x)


def test_group_with_empty_member_and_graph_capture():
    mats, Ws, masks, xs = _group_case((400, 300), 4096, 2, 4, 1, True, seed=5)
    empty = nm.nm_pack(torch.empty(0, 4096, dtype=torch.float16, device=DEV),
                       torch.empty(0, 4096, dtype=torch.uint8, device=DEV), 2, 4)
    ye = torch.empty(0, dtype=torch.float32, device=DEV)
    y0 = torch.empty(400, dtype=torch.float32, device=DEV)
    y1 = torch.empty(300, dtype=torch.float32, device=DEV)
    nm.nm_spmv_group([mats[0], empty, mats[1]], [xs[0][0]] * 3, [y0, ye, y1])
    torch.cuda.synchronize()
    _check(y0[None], Ws[0], masks[0], xs[0])
    _check(y1[None], Ws[1], masks[1], xs[1])
    ref0, ref1 = y0.clone(), y1.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            nm.nm_spmv_group(mats, [xs[0][0]] * 2, [y0, y1])
    for _ in range(2):
        y0.fill_(float("nan"))
        y1.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y0, ref0) and torch.equal(y1, ref1)


def test_device_error_word_is_clear():
    assert nm.nm_device_errors(clear=False) == 0
    assert nm.nm_device_errors(clear=True) == 0


_CHILD = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import nm_synth, oracle
from sparse_spmv_memory_02_b300 import nm
fails = []
for (rows, K, N, M, B) in json.loads(sys.argv[2]):
    W = nm_synth.weights(rows, K, rows + K, "cuda")
    mask = nm_synth.topn_mask(W, N, M)
    x = nm_synth.activations(K, B, rows + 3, True, "cuda")
    A = nm.nm_pack(W, mask, N, M)
    y = nm.nm_spmv_batched(A, x, y_dtype=torch.float32)
    torch.cuda.synchronize()
    Wn = W.cpu().numpy().view(np.uint16); xn = x.cpu().numpy().view(np.uint16)
    yr, sr = oracle.spmv_dense(Wn, mask.cpu().numpy(), xn)
    ok = oracle.within_tolerance(y.double().cpu().numpy(), yr, sr)
    if not ok.all():
        fails.append([rows, K, N, M, B, int((~ok).sum())])
# a fused group of three matrices sharing x
K, N, M = 4096, 2, 4
Ws = [nm_synth.weights(r, K, r, "cuda") for r in (300, 100, 57)]
ms = [nm_synth.topn_mask(W, N, M) for W in Ws]
As = [nm.nm_pack(W, m, N, M) for W, m in zip(Ws, ms)]
x = nm_synth.activations(K, 1, 9, True, "cuda")
ys = nm.nm_spmv_group(As, [x[0]] * 3, y_dtype=torch.float32)
torch.cuda.synchronize()
for W, m, y in zip(Ws, ms, ys):
    yr, sr = oracle.spmv_dense(W.cpu().numpy().view(np.uint16), m.cpu().numpy(),
                               x.cpu().numpy().view(np.uint16))
    ok = oracle.within_tolerance(y.double().cpu().numpy()[None], yr, sr)
    if not ok.all():
        fails.append(["group", W.shape[0], int((~ok).sum())])
errs = nm.nm_device_errors()
print(json.dumps({"fails": fails, "errors": errs}))
"""


@pytest.mark.parametrize("tune", ["warps=2,cpl=1,rows=0", "warps=3,cpl=2,R=1,rows=0",
                                  "ring=4096,rows=0", "R=3,ring=20000,rows=0", "pdl=0",
                                  "ctas=2,warps=4", "stage=1024,rows=0", "rows_R=1",
                                  "rows_R=4,rows_warps=3", "rows_xtile=1024", "rows_ring=4096",
                                  "rows_warps=1,rows_xtile=2048,rows_task=512", "ctas=2",
                                  "rows_pair=1", "rows_task=512", "rows_pre=1",
                                  "rows_xtile=4096,rows_task=1000,rows_pre=1",
                                  "rows_pair=1,rows_pre=2"])
def test_bulk_forced_tunings(tune):
    cases = [(5, 4096, 2, 4, 1), (301, 8192, 2, 4, 2), (77, 14336, 4, 8, 1),
             (150, 5120, 1, 4, 1), (64, 3072, 2, 8, 3), (33, 1024, 4, 4, 8)]
    env = dict(os.environ, NM_BULK_TUNE=tune)
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT, json.dumps(cases)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["fails"] == [] and out["errors"] == 0, out
