"""GPU parity of the tensor-core 2:4 products (tcgen05: A expanded into
tensor memory, or the packed values as the sparse operand of
tcgen05.mma.sp) against the CPU oracle.

The path is taken by default for 2:4 products from batch 3-5 on large enough
layers (the routing rule in nm_api.cu); the forced tuning ``tc=1`` (read once per process, so
run in a child) makes every 2:4 product with K a multiple of 128 and at most
256 rows per CTA take it.  Shapes cover one row, fewer rows than SMs, ragged
row splits, one and two 128-row MMA tiles (the second partial), the largest
split that still fits (256 rows per CTA), splits just past it and K not a
multiple of 128 (both fall back to the CUDA-core kernels), fp16 and fp32 y,
x and y with row strides wider than the matrix, and for the sparse-operand
product the K split: layers of at most one 128-row tile a SM give each tile
to a cluster of 2-8 CTAs, each a share of K's slabs (even and uneven shares,
a partial last tile, batch 1-8).
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

_CHILD = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import nm_synth, oracle
from sparse_spmv_memory_02_b300 import nm
g = np.random.default_rng(1)
nsm = torch.cuda.get_device_properties(0).multi_processor_count
fails = []
for (rows, K, B, wide, f32) in json.loads(sys.argv[2]):
    rows = rows if rows > 0 else -rows * nsm     # negative: rows per SM
    W = nm_synth.weights(rows, K, rows + K, "cuda")
    mask = nm_synth.topn_mask(W, 2, 4)
    A = nm.nm_pack(W, mask, 2, 4)
    xs = nm_synth.activations(K + (64 if wide else 0), B, rows + 3, True, "cuda")
    x = xs[:, :K]
    ydt = torch.float32 if f32 else torch.float16
    ybuf = torch.full((B, rows + (40 if wide else 0)), float("nan"), dtype=ydt, device="cuda")
    y = ybuf[:, :rows]
    nm.nm_spmv_batched(A, x, y)
    torch.cuda.synchronize()
    if wide and not torch.isnan(ybuf[:, rows:].float()).all():
        fails.append([rows, K, B, "wrote past ldy"])
    pick = np.arange(rows) if rows <= 1024 else np.sort(g.choice(rows, 512, replace=False))
    idx = torch.from_numpy(pick).to("cuda")
    Wn = W[idx].cpu().numpy().view(np.uint16)
    xn = x.contiguous().cpu().numpy().view(np.uint16)
    yr, sr = oracle.spmv_dense(Wn, mask[idx].cpu().numpy(), xn)
    yg = y[:, idx].double().cpu().numpy()
    ok = oracle.within_tolerance(yg, yr, sr)
    if not ok.all():
        fails.append([rows, K, B, int((~ok).sum())])
print(json.dumps({"fails": fails, "errors": nm.nm_device_errors()}))
"""

# (rows, K, batch, wide strides, fp32 y); rows < 0 means -rows per SM
CASES = [
    (1, 128, 8, False, True),
    (149, 1024, 8, True, True),
    (300, 256, 8, False, False),
    (4096, 4096, 8, True, True),
    (28672, 512, 8, False, True),     # two tiles, the second partial
    (-256, 384, 8, False, True),      # 256 rows a CTA: both tiles full
    (-257, 256, 8, False, True),      # 257 rows a CTA: CUDA-core kernels
    (37000, 384, 8, True, False),
    (3000, 4000, 8, False, True),     # K not a multiple of 128
    (5000, 2048, 5, False, True),     # batch 5 (x padded to 16 rows)
    # the sparse-operand product's K split (clusters of CTAs sharing a tile)
    (1000, 896, 4, False, True),      # clusters of 7, 7 slabs: one slab each
    (1000, 640, 3, True, False),      # clusters of 5; last tile 104 rows
    (4100, 1152, 8, False, True),     # clusters of 4 over 9 slabs (3, 2, 2, 2)
    (8192, 1024, 1, False, True),     # batch 1, clusters of 2
    # more than 8 vectors (the tensor-core path only): 16-column split sums
    # up to batch 16, then N = 32 MMAs without the split
    (1000, 896, 12, True, True),
    (8192, 1024, 16, False, False),
    (149, 1024, 9, False, True),
    (4096, 4096, 24, True, True),
    (28672, 512, 32, False, True),    # two tiles a CTA, N = 32
]


@pytest.mark.parametrize("tune", ["tc=1,tc_sp=0", "tc=1,tc_sp=1", "tc=1,tc_sp=1,sp_split=0"],
                         ids=["expanded", "sparse_operand", "sparse_operand_unsplit"])
def test_tensor_core_path_forced(tune):
    """Every case through the tensor-core product, A either expanded into
    tensor memory or taken as the sparse operand of tcgen05.mma.sp (with
    and without the K split across a cluster)."""
    env = dict(os.environ, NM_BULK_TUNE=tune)
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT, json.dumps(CASES)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["fails"] == [] and out["errors"] == 0, out


@pytest.mark.parametrize("rows,K,B", [(28672, 8192, 16), (8192, 8192, 16), (8192, 4096, 32)])
def test_tensor_core_path_above_batch_8(rows, K, B):
    """Above 8 vectors only the tensor-core path runs: sampled rows of the
    70B-shaped gate and of split layers against the oracle, at batch 16 (the
    16-column split sums) and 32 (N = 32 MMAs)."""
    W = nm_synth.weights(rows, K, 90 + B, DEV)
    mask = nm_synth.topn_mask(W, 2, 4)
    A = nm.nm_pack(W, mask, 2, 4)
    x = nm_synth.activations(K, B, 91 + B, True, DEV)
    y = nm.nm_spmv_batched(A, x, y_dtype=torch.float32)
    torch.cuda.synchronize()
    g = np.random.default_rng(B)
    pick = np.sort(g.choice(rows, 256, replace=False))
    idx = torch.from_numpy(pick).to(DEV)
    yr, sr = oracle.spmv_dense(W[idx].cpu().numpy().view(np.uint16), mask[idx].cpu().numpy(),
                               x.cpu().numpy().view(np.uint16))
    ok = oracle.within_tolerance(y[:, idx].double().cpu().numpy(), yr, sr)
    assert ok.all(), "%d/%d outside tolerance" % ((~ok).sum(), ok.size)
    assert nm.nm_device_errors() == 0


def _group_check(rows_list, K, B, seed):
    """nm_spmv_group over matrices of these rows, each with its own x, against
    the oracle on sampled rows of every member."""
    Ws, masks, mats, xs = [], [], [], []
    for i, rows in enumerate(rows_list):
        W = nm_synth.weights(rows, K, seed + i, DEV)
        mask = nm_synth.topn_mask(W, 2, 4)
        Ws.append(W)
        masks.append(mask)
        mats.append(nm.nm_pack(W, mask, 2, 4))
        xs.append(nm_synth.activations(K, B, seed + 50 + i, True, DEV))
    ys = nm.nm_spmv_group(mats, xs, y_dtype=torch.float32)
    torch.cuda.synchronize()
    g = np.random.default_rng(seed)
    for i, rows in enumerate(rows_list):
        pick = np.sort(g.choice(rows, min(rows, 192), replace=False))
        idx = torch.from_numpy(pick).to(DEV)
        yr, sr = oracle.spmv_dense(Ws[i][idx].cpu().numpy().view(np.uint16),
                                   masks[i][idx].cpu().numpy(), xs[i].cpu().numpy().view(np.uint16))
        ok = oracle.within_tolerance(ys[i][:, idx].double().cpu().numpy(), yr, sr)
        assert ok.all(), "member %d (%d rows): %d/%d outside tolerance" % (
            i, rows, (~ok).sum(), ok.size)
    assert nm.nm_device_errors() == 0


@pytest.mark.parametrize("B", [9, 16, 32])
@pytest.mark.parametrize("rows_list", [(8192, 1024, 1024), (300, 77, 250, 4, 5), (1000, 2048)],
                         ids=["qkv_shaped", "ragged5", "two"])
def test_group_in_one_tensor_core_launch(rows_list, B):
    """Above 8 vectors every 2:4 member takes the tensor-core product, so a
    group is one grouped launch of it (units of each matrix consecutive,
    each matrix its own maps, x and y): each member against the oracle."""
    _group_check(rows_list, 1024, B, 300 + B)


def test_group_70b_qkv_batch8_one_launch():
    """The 70B-shaped q/k/v (8192 + 1024 + 1024 rows, K = 8192) at batch 8:
    all three take the tensor cores, in one grouped launch."""
    _group_check((8192, 1024, 1024), 8192, 8, 77)


def test_batch_above_8_unsupported_where_the_tensor_cores_cannot_run():
    """257 rows per SM exceed the tensor-core product's two tiles: batch 9
    is refused (NM_ERR_UNSUPPORTED) before any launch, batch 8 runs on the
    CUDA cores."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    rows, K = 257 * nsm, 256
    W = nm_synth.weights(rows, K, 5, DEV)
    A = nm.nm_pack(W, nm_synth.topn_mask(W, 2, 4), 2, 4)
    x = nm_synth.activations(K, 9, 6, True, DEV)
    with pytest.raises(nm.NMError) as e:
        nm.nm_spmv_batched(A, x)
    assert e.value.status == nm.NM_ERR_UNSUPPORTED
    y = nm.nm_spmv_batched(A, x[:8])
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()


def test_tensor_core_path_default_on_70b_gate_batch8():
    """The gate projection of the 70B-shaped block (28672 x 8192) at batch 8
    takes the tensor-core path by default: sampled rows against the oracle,
    and a repeated call gives the same bits."""
    rows, K, B = 28672, 8192, 8
    W = nm_synth.weights(rows, K, 77, DEV)
    mask = nm_synth.topn_mask(W, 2, 4)
    A = nm.nm_pack(W, mask, 2, 4)
    x = nm_synth.activations(K, B, 78, True, DEV)
    y = nm.nm_spmv_batched(A, x, y_dtype=torch.float32)
    torch.cuda.synchronize()
    g = np.random.default_rng(3)
    pick = np.sort(g.choice(rows, 384, replace=False))
    idx = torch.from_numpy(pick).to(DEV)
    yr, sr = oracle.spmv_dense(W[idx].cpu().numpy().view(np.uint16), mask[idx].cpu().numpy(),
                               x.cpu().numpy().view(np.uint16))
    ok = oracle.within_tolerance(y[:, idx].double().cpu().numpy(), yr, sr)
    assert ok.all(), "%d/%d outside tolerance" % ((~ok).sum(), ok.size)
    assert nm.nm_device_errors() == 0
    y2 = nm.nm_spmv_batched(A, x, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
