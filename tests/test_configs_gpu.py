"""Parity at the benchmark's full sizes: the five workload configurations, in
the launch structure bench.py times (the step's layers replayed from one CUDA
graph, q/k/v and gate/up each fused into one grouped launch).

For every checked layer nm_pack must equal the oracle's pack byte for byte
over the whole matrix, and the SpMV must satisfy
|y - y_ref| <= 1e-3 * sum|w x| + 1e-6 on sampled rows (the oracle computes
those rows only, from the same seeded inputs regenerated on the GPU and
copied to the host; nothing the oracle reads comes from libnm).
"""
import numpy as np
import pytest
import torch

import bench
import nm_synth
import oracle
from sparse_spmv_memory_02_b300 import nm

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _np16(t):
    return t.detach().cpu().numpy().view(np.uint16)


def _check_layer(wl, L, N, M, batch, check_pack=True, nsample=192, seed=0):
    li = L["index"]
    layer = wl.layers[li % len(wl.layers)]
    W, mask, x = nm_synth.layer_inputs(wl, li, layer, N, M, batch, DEV)
    A = L["mats"][0]
    if check_pack:
        ev, em, bad = oracle.pack(_np16(W), mask.cpu().numpy(), N, M)
        assert bad == 0
        assert np.array_equal(_np16(A.values), ev), "%s: packed values differ" % L["name"]
        assert np.array_equal(A.masks.cpu().numpy().view(np.uint32), em), \
            "%s: packed masks differ" % L["name"]
    g = np.random.default_rng(seed + li)
    rows = layer.rows
    idx = np.sort(g.choice(rows, min(nsample, rows), replace=False))
    it = torch.from_numpy(idx).to(DEV)
    yr, sr = oracle.spmv_dense(_np16(W[it]), mask[it].cpu().numpy(), _np16(x))
    y = L["y"] if batch > 1 else L["y"][None]
    yg = y[:, it].double().cpu().numpy()
    ok = oracle.within_tolerance(yg, yr, sr)
    assert ok.all(), "%s: %d/%d sampled outputs outside tolerance" % (L["name"], (~ok).sum(),
                                                                       ok.size)


def _run_step(wl, N, M, batch, fused=True):
    layers = bench.build_workload(wl, N, M, batch, copies=1)
    for L in layers:
        L["y"].fill_(float("nan"))
    streams = bench.capture_step_graphs(layers, 1, fused=fused)
    streams[0].replay()
    torch.cuda.synchronize()
    assert nm.nm_device_errors() == 0
    return layers, streams[0]


def test_config1_single_1024_full():
    """1024 x 1024, 2:4, seed 0, batch 1: every output checked."""
    wl = nm_synth.WORKLOADS["single_1024"]
    layers, _ = _run_step(wl, 2, 4, 1)
    _check_layer(wl, layers[0], 2, 4, 1, nsample=1024)


@pytest.mark.parametrize("fused", [True, False])
def test_config2_llama31_8b_block(fused):
    wl = nm_synth.WORKLOADS["llama31_8b_block"]
    layers, stream = _run_step(wl, 2, 4, 1, fused=fused)
    assert stream.launches == (4 if fused else 7)
    for L in layers:
        _check_layer(wl, L, 2, 4, 1)


def test_config2_llama31_8b_block_forward_graph():
    """The headline's timed structure: several blocks (steps) in one CUDA
    graph rotating over packed copies.  After a replay every copy's last
    step has run; the outputs (written by the last step) must match the
    oracle, and the same replay again gives the same bits."""
    wl = nm_synth.WORKLOADS["llama31_8b_block"]
    layers = bench.build_workload(wl, 2, 4, 1, copies=2)
    streams = bench.capture_step_graphs(layers, 2, fused=True)
    g = bench.capture_multi_step(streams, 2, 5)
    for L in layers:
        L["y"].fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert nm.nm_device_errors() == 0
    first = [L["y"].clone() for L in layers]
    for L in layers:
        _check_layer(wl, L, 2, 4, 1, check_pack=False)
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a, L["y"]) for a, L in zip(first, layers))


@pytest.mark.parametrize("N,M", [(2, 4), (4, 8), (1, 4), (2, 8)])
def test_config3_qwen3_14b_mlp_pattern_sweep(N, M):
    wl = nm_synth.WORKLOADS["qwen3_14b_mlp"]
    layers, stream = _run_step(wl, N, M, 1)
    assert stream.launches == 2  # gate+up fused, down
    for L in layers:
        _check_layer(wl, L, N, M, 1)


@pytest.mark.parametrize("batch", [1, 2, 3, 4, 8])
def test_config4_llama33_70b_block_batched(batch):
    wl = nm_synth.WORKLOADS["llama33_70b_block"]
    layers, _ = _run_step(wl, 2, 4, batch)
    for L in layers:
        _check_layer(wl, L, 2, 4, batch, check_pack=(batch == 1), nsample=96)
    del layers
    torch.cuda.empty_cache()


def test_config5_qwen3_32b_stream():
    """All 64 blocks x 7 layers in one CUDA graph (256 launches); pack and
    sampled outputs checked on the first block and on layers spread over the
    stream."""
    wl = nm_synth.WORKLOADS["qwen3_32b_stream"]
    from sparse_spmv_memory_02_b300.stream import LayerStream
    layers = []
    x_by_source = {}
    for li, layer in wl.all_layers():
        W, mask, x = nm_synth.layer_inputs(wl, li, layer, 2, 4, 1, DEV)
        src = nm_synth.x_source(wl, li)
        x = x_by_source.setdefault(src, x[0])
        A = nm.nm_pack(W, mask, 2, 4)
        del W, mask
        y = torch.full((layer.rows,), float("nan"), dtype=torch.float16, device=DEV)
        layers.append(dict(name="%s.%d" % (layer.name, li // 7), index=li, mats=[A], x=x, y=y))
    s = LayerStream([L["mats"][0] for L in layers], [L["x"] for L in layers],
                    [L["y"] for L in layers], fuse_shared_input=True)
    assert s.launches == 64 * 4
    s.capture()
    for L in layers:
        L["y"].fill_(float("nan"))
    s.replay()
    torch.cuda.synchronize()
    assert nm.nm_device_errors() == 0
    for li in list(range(7)) + [60, 131, 222, 333, 447]:
        _check_layer(wl, layers[li], 2, 4, 1, check_pack=li < 7, nsample=64)
