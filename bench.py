#!/usr/bin/env python
"""Benchmark of the N:M SpMV decode path on one B300 (or N replicas).

A "step" is one decode token's pass over the linear layers of one decoder
block of the chosen workload (default: the Llama-3.1-8B-shaped block, 2:4,
batch 1: q, k, v, o, gate, up, down) -- seven nm_spmv calls replayed from one
CUDA graph.  Weights are synthetic (seeded N(0, 0.02), top-N |w| per group of
M along K) and resident in HBM; three packed copies of the block rotate from
step to step so that no step finds its weights in the 126 MB L2 (the
rotation set is about 740 MB).

Printed (rank 0, one JSON line): achieved GB/s of algorithmic bytes
(kept values + mask bits + x + y) over the timed steps, microseconds per call
per layer, the roofline of the SpMV kernel against the measured HBM peak,
the dense fp16 cuBLAS GEMV of the same shapes, an end-to-end figure through
the public API with host buffers, the CPU oracle as a reported baseline and
the SM clocks seen during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import nm_synth  # noqa: E402

METRIC = "N:M SpMV µs/call and achieved HBM GB/s (% of peak), batch-1 decode shapes"
FALLBACK_HBM_GBS = 6400.0

# DRAM bytes (read + write) per launch, averaged over the launches of one
# step, from an ncu capture of that step taken with the current kernels;
# workloads without an entry report null.
TRAFFIC_PER_LAUNCH = {
    ("llama31_8b_block", "2:4", 1, "fused"): 61.481e6,  # 12 launches of the fused step
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="llama31_8b_block", choices=sorted(nm_synth.WORKLOADS))
    p.add_argument("--pattern", default=None, help="N:M, default: the workload's first")
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--copies", type=int, default=3, help="rotating packed copies (L2 defeat)")
    p.add_argument("--graph-steps", type=int, default=32,
                   help="consecutive steps (decoder blocks) captured in one CUDA graph: 32 is "
                        "one forward of a 32-block model such as Llama-3.1-8B")
    p.add_argument("--profile-steps", type=int, default=50, help="calls per layer in the per-layer pass")
    p.add_argument("--launch", choices=["fused", "unfused", "fused_silu"], default="fused",
                   help="fused: layers reading the same input (q/k/v, gate/up) share one "
                        "nm_spmv_group launch; unfused: one nm_spmv launch per layer; "
                        "fused_silu: as fused, with gate/up one nm_spmv_gate_up_silu launch "
                        "writing silu(gate x) * (up x)")
    p.add_argument("--no-dense", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-prune", action="store_true", help="skip the mask-selection timing")
    p.add_argument("--no-calib", action="store_true", help="skip the calibration timing")
    p.add_argument("--no-crossover", action="store_true",
                   help="skip the batch crossover against 2:4 sparse tensor cores")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads (single layer, Qwen3-14B MLP pattern sweep, "
                        "Llama-3.3-70B block at batch 1/2/3/4/8, 448-layer Qwen3-32B stream)")
    p.add_argument("--calib-tokens", type=int, default=512,
                   help="decode-step tokens per nm_calib_accumulate call in the calibration timing")
    p.add_argument("--layer", default=None, metavar="ROWSxK",
                   help="time one product of this shape alone (pattern --pattern, default 2:4; "
                        "batch --batch) and print one JSON line; the workload options are ignored")
    p.add_argument("--calls", type=int, default=50, help="--layer: calls per timed sample")
    p.add_argument("--samples", type=int, default=20, help="--layer: timed samples")
    p.add_argument("--eager", action="store_true",
                   help="--layer: launch the calls eagerly instead of from a CUDA graph (for "
                        "profilers that replay single launches)")
    p.add_argument("--seed", type=int, default=4242, help="--layer: weight seed (x: seed + 500)")
    p.add_argument("--batches", default=None, help="--layer: comma-separated batch sizes")
    return p.parse_args(argv)


# ------------------------------------------------------------------ helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tc_peak():
    """Dense fp16 tensor peak in TFLOP/s: the measured cuBLAS bf16 burst figure
    (fp16 and bf16 share one rate), else the profiling fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (bf16 burst; fp16 runs at the same rate)"
    except Exception:
        return 1800.0, "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi samples (SM clock, reasons) while the GPU runs.  nvidia-smi
    writes them, timestamped, to a file that is read only when a summary is
    asked for: no Python thread runs beside the timed loops (one that woke
    every sample would take the GIL from the end-to-end loop's host thread)."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index, self.period_ms = index, period_ms
        self.proc, self.out = None, None

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=self.out, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    @property
    def samples(self):
        """(epoch seconds, [index, sm, max sm, power, active, 4 reasons]) each."""
        if self.out is None:
            return []
        self.out.seek(0)
        rows = []
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue  # a line nvidia-smi is still writing
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append((t, parts[1:]))
        return rows

    def wait_first(self, timeout: float = 3.0):
        """Block until nvidia-smi has printed a sample (its start-up is done,
        so it cannot stall the timed region), at most `timeout` seconds."""
        t_end = time.time() + timeout
        while self.proc is not None and not self.samples and time.time() < t_end:
            time.sleep(0.01)
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float, window: str = "timed region"):
        samples = self.samples
        sel = [p for t, p in samples if t0 <= t <= t1]
        if not sel:
            sel = [p for _, p in samples]
            window = "whole run (timed region shorter than the sampling period)"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "nvidia-smi unavailable"}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[1]) for p in sel if num(p[1]) is not None]
        mx = [num(p[2]) for p in sel if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in sel for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sel), "window": window}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def layer_list(wl):
    """Every layer of the workload's step (all blocks of a layer stream)."""
    return list(wl.all_layers())


def workload_bytes(wl, N, M, batch):
    return sum(layer.rows * (layer.K // M) * N * 2 + layer.rows * layer.K // 8
               + batch * layer.K * 2 + batch * layer.rows * 2 for _, layer in layer_list(wl))


# ------------------------------------------------------------------ workload

def build_workload(wl, N, M, batch, copies, device="cuda", keep_dense=False):
    """Generate, pack and replicate the layers of one step.  Returns a list of
    dicts: name, rows, K, mats (packed copies), x, y, dense (optional).
    Layers that read the same block input (q/k/v; gate/up) share one x
    tensor."""
    from sparse_spmv_memory_02_b300 import nm
    layers = []
    x_by_source = {}
    for li, layer in layer_list(wl):
        W, mask, x = nm_synth.layer_inputs(wl, li, layer, N, M, batch, device)
        src = nm_synth.x_source(wl, li)
        if src in x_by_source:
            x = x_by_source[src]
        else:
            x = x if batch > 1 else x[0]
            x_by_source[src] = x
        A = nm.nm_pack(W, mask, N, M)
        mats = [A] + [nm.PackedMatrix(A.values.clone(), A.masks.clone(), A.rows, A.K, N, M)
                      for _ in range(copies - 1)]
        dense = None
        if keep_dense:
            Wm = torch.where(mask.bool(), W, torch.zeros((), dtype=W.dtype, device=device))
            dense = [Wm] + [Wm.clone() for _ in range(copies - 1)]
        del W, mask
        y = torch.empty(batch, layer.rows, dtype=torch.float16, device=device)
        layers.append(dict(name=layer.name, rows=layer.rows, K=layer.K, mats=mats,
                           x=x, y=y if batch > 1 else y[0], dense=dense, index=li))
    torch.cuda.synchronize()
    return layers


def silu_pairs(layers):
    """(gate, up) index pairs of consecutive gate and up layers (one per
    decoder block)."""
    return [(i, i + 1) for i in range(len(layers) - 1)
            if layers[i]["name"] == "gate" and layers[i + 1]["name"] == "up"]


def step_bytes(layers, batch, silu=False):
    """Algorithmic bytes per layer call; with the gate/up SiLU epilogue the
    up layer reads no x of its own and writes no y (the pair writes one h)."""
    from sparse_spmv_memory_02_b300.stream import algorithmic_bytes
    out = [algorithmic_bytes(L["mats"][0], batch, 2) for L in layers]
    if silu:
        for _, ui in silu_pairs(layers):
            out[ui] -= batch * layers[ui]["K"] * 2 + batch * layers[ui]["rows"] * 2
    return out


def capture_step_graphs(layers, copies, fused, silu=False):
    from sparse_spmv_memory_02_b300.stream import LayerStream
    streams = []
    pairs = silu_pairs(layers) if silu else ()
    for c in range(copies):
        s = LayerStream([L["mats"][c] for L in layers], [L["x"] for L in layers],
                        [L["y"] for L in layers], fuse_shared_input=fused, silu_pairs=pairs)
        s.capture()
        streams.append(s)
    return streams


def time_steps(streams, copies, steps, warmup, world, samples=20):
    """Replays `steps` steps (rotating over the copies) after `warmup`
    untimed ones, in `samples` consecutive timed pieces (CUDA events on the
    replay stream around each piece, no gap between pieces).  Returns
    (total seconds, per-step seconds of every piece, wall t0, wall t1)."""
    for s in range(warmup):
        streams[s % copies].replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    samples = max(1, min(samples, steps))
    bounds = [round(i * steps / samples) for i in range(samples + 1)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(samples + 1)]
    t_wall0 = time.time()
    ev[0].record()
    for i in range(samples):
        for s in range(bounds[i], bounds[i + 1]):
            streams[s % copies].replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    per_step = [ev[i].elapsed_time(ev[i + 1]) * 1e-3 / max(1, bounds[i + 1] - bounds[i])
                for i in range(samples)]
    return ev[0].elapsed_time(ev[samples]) * 1e-3, per_step, t_wall0, t_wall1


def capture_multi_step(streams, copies, nsteps):
    """One CUDA graph of steps 0 .. nsteps - 1, step s on packed copy s % copies."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for s in range(nsteps):
                streams[s % copies].run_eager()
    torch.cuda.current_stream().wait_stream(side)
    return g


def time_graph_steps(streams, copies, per_graph, steps, warmup, world, samples=20):
    """As time_steps, with `per_graph` consecutive steps in each CUDA graph
    (a decode forward's blocks; the last replay takes the remainder), so the
    timed region runs exactly `steps` steps.  The timed pieces are whole
    replays."""
    per_graph = max(1, min(per_graph, steps))
    g = capture_multi_step(streams, copies, per_graph)
    rem = steps % per_graph
    reps = [(g, per_graph)] * (steps // per_graph)
    if rem:
        reps.append((capture_multi_step(streams, copies, rem), rem))
    for _ in range(-(-max(1, warmup) // per_graph)):
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    samples = max(1, min(samples, len(reps)))
    bounds = [round(i * len(reps) / samples) for i in range(samples + 1)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(samples + 1)]
    t_wall0 = time.time()
    ev[0].record()
    for i in range(samples):
        for r in range(bounds[i], bounds[i + 1]):
            reps[r][0].replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    per_step = [ev[i].elapsed_time(ev[i + 1]) * 1e-3
                / max(1, sum(n for _, n in reps[bounds[i]:bounds[i + 1]]))
                for i in range(samples)]
    return ev[0].elapsed_time(ev[samples]) * 1e-3, per_step, t_wall0, t_wall1


def layer_pass(layers, batch, reps, l2_bytes):
    """Each layer alone: a CUDA graph of `reps` calls that rotate over enough
    packed copies of the layer (> 3x L2) that every call streams its weights
    from HBM.  Returns per-layer mean microseconds per call."""
    from sparse_spmv_memory_02_b300 import nm
    out = []
    for L in layers:
        A = L["mats"][0]
        nbytes = A.nbytes
        ncopy = max(3, -(-3 * l2_bytes // nbytes))
        extra = [nm.PackedMatrix(A.values.clone(), A.masks.clone(), A.rows, A.K, A.N, A.M)
                 for _ in range(ncopy - len(L["mats"]))]
        mats = list(L["mats"]) + extra
        n = max(reps, len(mats))

        def run():
            for i in range(n):
                if L["x"].dim() == 1:
                    nm.nm_spmv(mats[i % len(mats)], L["x"], L["y"])
                else:
                    nm.nm_spmv_batched(mats[i % len(mats)], L["x"], L["y"])
        run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                run()
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(5):
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e-3 / n)
        out.append(statistics.median(times))
        del g, extra, mats
        torch.cuda.empty_cache()
    return out


def _graph_time(run, n):
    """Median seconds per call of `run` (n calls) replayed from a CUDA graph."""
    run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            run()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(5):
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e-3 / n)
    del g
    return statistics.median(times)


def pair_pass(gate, up, batch, reps, l2_bytes):
    """The gate/up pair alone, as one nm_spmv_group launch (two outputs) and
    as one nm_spmv_gate_up_silu launch (silu(gate x) * (up x)), each a CUDA
    graph of calls rotating over > 3x L2 of packed copies.  Returns
    {variant: (seconds per call, algorithmic bytes per call)}."""
    from sparse_spmv_memory_02_b300 import nm
    from sparse_spmv_memory_02_b300.stream import algorithmic_bytes
    G, U = gate["mats"][0], up["mats"][0]
    ncopy = max(3, -(-3 * l2_bytes // (G.nbytes + U.nbytes)))
    gs = [G] + [nm.PackedMatrix(G.values.clone(), G.masks.clone(), G.rows, G.K, G.N, G.M)
                for _ in range(ncopy - 1)]
    us = [U] + [nm.PackedMatrix(U.values.clone(), U.masks.clone(), U.rows, U.K, U.N, U.M)
                for _ in range(ncopy - 1)]
    n = max(reps, ncopy)
    x, yg, yu = gate["x"], gate["y"], up["y"]

    def run_group():
        for i in range(n):
            nm.nm_spmv_group([gs[i % ncopy], us[i % ncopy]], [x, x], [yg, yu])

    def run_silu():
        for i in range(n):
            nm.nm_spmv_gate_up_silu(gs[i % ncopy], us[i % ncopy], x, yg)

    b_group = algorithmic_bytes(G, batch, 2) + algorithmic_bytes(U, batch, 2)
    b_silu = b_group - batch * U.K * 2 - batch * U.rows * 2
    out = {"group": (_graph_time(run_group, n), b_group),
           "silu": (_graph_time(run_silu, n), b_silu)}
    del gs, us
    torch.cuda.empty_cache()
    return out


def prune_pass(wl, N, M, reps, l2_bytes):
    """nm_select_mask and nm_prune_pack on the dense fp16 weights of the
    block's largest layer, with an activation-norm column scale, each a CUDA
    graph of calls rotating over > 3x L2 of weight copies.  Returns
    {name: (seconds per call, algorithmic bytes per call)}."""
    from sparse_spmv_memory_02_b300 import nm
    li, layer = max(layer_list(wl)[:len(wl.layers)], key=lambda t: t[1].rows * t[1].K)
    rows, K = layer.rows, layer.K
    W0 = nm_synth.weights(rows, K, nm_synth.weight_seed(wl, li), "cuda")
    ncopy = max(2, -(-3 * l2_bytes // W0.numel() // 2))
    Ws = [W0] + [W0.clone() for _ in range(ncopy - 1)]
    x = nm_synth.activations(K, 64, nm_synth.x_seed(wl, li), wl.outliers, "cuda")
    scale = x.float().norm(dim=0).contiguous()  # column norms over 64 synthetic tokens
    mask = torch.empty(rows, K, dtype=torch.uint8, device="cuda")
    A = nm.nm_prune_pack(W0, N, M, scale)
    n = max(reps // 5, ncopy)

    def run_select():
        for i in range(n):
            nm.nm_select_mask(Ws[i % ncopy], N, M, scale, mask=mask)

    def run_prune():
        for i in range(n):
            nm.nm_prune_pack(Ws[i % ncopy], N, M, scale, values=A.values, masks=A.masks)

    wbytes = rows * K * 2 + K * 4
    out = {"select_mask": (_graph_time(run_select, n), wbytes + rows * K),
           "prune_pack": (_graph_time(run_prune, n), wbytes + A.nbytes),
           "shape": (layer.name, rows, K)}
    del Ws, W0, mask, A
    torch.cuda.empty_cache()
    return out


def calib_pass(wl, tokens, reps):
    """nm_calib_accumulate (H += X^T X on the tensor cores) for `tokens`
    decode-step inputs of each distinct layer-input width of the block.
    Returns {K: (seconds per call, flops, bytes)}: flops T K (K + 1), the
    symmetric rank-T update's count (the kernel computes the tiles on and
    above the diagonal and mirrors them); bytes the read-modify-write of H
    (8 K^2) plus X once."""
    from sparse_spmv_memory_02_b300 import nm
    out = {}
    for K in sorted({layer.K for layer in wl.layers}):
        X = nm_synth.activations(K, tokens, 77 + K, wl.outliers, "cuda")
        H = torch.zeros(K, K, dtype=torch.float32, device="cuda")
        n = max(3, reps // 10)

        def run():
            for _ in range(n):
                nm.nm_calib_accumulate(X, H)
        t = _graph_time(run, n)
        out[K] = (t, float(tokens) * K * (K + 1), 8.0 * K * K + 2.0 * tokens * K)
        del X, H
        torch.cuda.empty_cache()
    return out


def _eager_time(run, n, warmup=3):
    """Median seconds per call of `run` (n calls per sample), launched
    eagerly (library calls that may not be graph-capturable)."""
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(5):
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e-3 / n)
    return statistics.median(times)


def _libnm_kernel(rows, batch, K):
    """Which kernel libnm runs for a 2:4 product with K a multiple of 128
    (the library's routing rule, restated for the report; NM_BULK_TUNE tc=0/1
    and tc_sp=0 override it there and here)."""
    tune = dict(kv.split("=", 1) for kv in os.environ.get("NM_BULK_TUNE", "").split(",")
                if "=" in kv)
    tc, sp = int(tune.get("tc", "-1")), int(tune.get("tc_sp", "1"))
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    per_sm = (rows + nsm - 1) // nsm
    w = rows * K
    auto = ((batch >= 5 and w >= 4 << 20) or (batch in (3, 4) and w > 24_000_000)
            or (batch == 2 and w >= 128 << 20 and per_sm <= 128))
    if tc != 0 and per_sm <= 256 and (tc == 1 or auto):
        return ("tensor-core 2:4 product (tcgen05.mma.sp, packed values as the sparse operand)"
                if sp else "tensor-core 2:4 product (tcgen05, A expanded into tensor memory)")
    return "CUDA-core row kernel"


def crossover_pass(batches=(1, 2, 4, 8, 16, 32, 64)):
    """The batch at which a 2:4 sparse-tensor-core GEMM (cuSPARSELt through
    torch's semi-structured sparse tensors, a library comparator) overtakes
    this library, on the Llama-3.3-70B-shaped gate layer (28672 x 8192, 2:4):
    microseconds per product for libnm (batch <= 8; the CUDA-core row kernel,
    or at batch 8 the library's tensor-core 2:4 product), the sparse tensor
    cores and dense cuBLAS on the masked weights, all launched eagerly."""
    from sparse_spmv_memory_02_b300 import nm
    rows, K = 28672, 8192
    W = nm_synth.weights(rows, K, 4242, "cuda")
    mask = nm_synth.topn_mask(W, 2, 4)
    A = nm.nm_pack(W, mask, 2, 4)
    Wm = torch.where(mask.bool(), W, torch.zeros((), dtype=W.dtype, device="cuda"))
    del W, mask
    Ws, sparse_note = None, "cuSPARSELt 2:4 via torch.sparse.to_sparse_semi_structured"
    try:
        from torch.sparse import to_sparse_semi_structured
        Ws = to_sparse_semi_structured(Wm)
    except Exception as e:  # reported, not fatal: a comparator only
        sparse_note = "unavailable: %s" % str(e).splitlines()[0][:160]
    table = []
    n = 10
    for B in batches:
        X = nm_synth.activations(K, B, 900 + B, True, "cuda")
        Xt = X.t().contiguous()
        row = {"batch": B}
        if B <= nm.NM_MAX_BATCH_TC:  # a 2:4 layer: the tensor-core path takes up to 32
            try:
                row["libnm_kernel"] = _libnm_kernel(rows, B, K)
            except Exception as e:  # a label only: never costs the timing
                row["libnm_kernel"] = "unknown (%s)" % type(e).__name__
            y = torch.empty(B, rows, dtype=torch.float16, device="cuda")

            def ours():
                for _ in range(n):
                    nm.nm_spmv_batched(A, X, y)
            row["libnm_us"] = _eager_time(ours, n) * 1e6

        def dense():
            for _ in range(n):
                torch.mm(Wm, Xt)
        row["dense_cublas_us"] = _eager_time(dense, n) * 1e6
        if Ws is not None:
            try:
                def sparse():
                    for _ in range(n):
                        torch.mm(Ws, Xt)
                row["sparse_tc_us"] = _eager_time(sparse, n) * 1e6
            except Exception as e:
                row["sparse_tc_us"] = None
                row["sparse_tc_error"] = str(e).splitlines()[0][:160]
        table.append(row)
    del A, Wm, Ws
    torch.cuda.empty_cache()
    return {"layer": {"rows": rows, "K": K, "pattern": "2:4"}, "sparse_tc": sparse_note,
            "table": table}


def dense_pass(layers, copies, steps, warmup):
    """cuBLAS fp16 GEMV of W (dropped weights zeroed), same protocol."""
    n = len(layers)
    ys = [torch.empty_like(L["y"]) for L in layers]
    graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i, L in enumerate(layers):  # warm cuBLAS handles outside capture
                torch.matmul(L["dense"][c], L["x"].t() if L["x"].dim() > 1 else L["x"])
            with torch.cuda.graph(g, stream=side):
                for i, L in enumerate(layers):
                    if L["x"].dim() == 1:
                        torch.mv(L["dense"][c], L["x"], out=ys[i])
                    else:
                        ys[i].copy_(torch.matmul(L["x"], L["dense"][c].t()))
        torch.cuda.current_stream().wait_stream(side)
        graphs.append(g)
    for s in range(warmup):
        graphs[s % copies].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(steps):
        graphs[s % copies].replay()
    e1.record()
    torch.cuda.synchronize()
    dt = e0.elapsed_time(e1) * 1e-3 / steps
    dense_bytes = sum(L["rows"] * L["K"] * 2 for L in layers)
    del graphs
    return dt, dense_bytes, n


def e2e_pass(layers, copies, steps, warmup, fused, silu=False, per_graph=1):
    """Through the public API with host buffers, `per_graph` steps (decoder
    blocks) a forward, each block with its own input and output buffers.
    Every forward: all of its blocks' input vectors are copied from one
    pinned host buffer into one device buffer, the blocks' libnm launches
    run, all of their outputs are copied into one pinned host buffer -- the
    two copies captured together with the launches in one CUDA graph -- and
    the host waits for the outputs (a decode loop needs them before the next
    token).  Block i reads packed copy i % copies.  Returns (mean seconds per
    step, per-step seconds of every forward, h2d bytes per step, d2h bytes
    per step)."""
    from sparse_spmv_memory_02_b300.stream import LayerStream
    G = max(1, min(per_graph, steps))
    srcs = []
    for L in layers:
        if not any(L["x"] is t for t in srcs):
            srcs.append(L["x"])

    def layout(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += -(-t.numel() // 64) * 64  # keep every view 128-byte aligned
        return offs, n
    xoff, xn = layout(srcs)
    youts = [L["y"] for L in layers]
    yoff, yn = layout(youts)
    x_dev = torch.zeros(G * xn, dtype=torch.float16, device="cuda")
    y_dev = torch.zeros(G * yn, dtype=youts[0].dtype, device="cuda")
    blocks = []
    for i in range(G):
        xv = [x_dev[i * xn + o:i * xn + o + t.numel()].view(t.shape) for o, t in zip(xoff, srcs)]
        yv = [y_dev[i * yn + o:i * yn + o + t.numel()].view(t.shape) for o, t in zip(yoff, youts)]
        for v, t in zip(xv, srcs):
            v.copy_(t)
        xs = [xv[next(k for k, t in enumerate(srcs) if t is L["x"])] for L in layers]
        blocks.append(LayerStream([L["mats"][i % copies] for L in layers], xs, yv,
                                  fuse_shared_input=fused,
                                  silu_pairs=silu_pairs(layers) if silu else ()))
    x_host = x_dev.cpu().pin_memory()
    y_host = torch.empty(G * yn, dtype=y_dev.dtype).pin_memory()
    for b in blocks[:2]:
        b.run_eager()
    torch.cuda.synchronize()

    def forward_graph(n):
        # Inside one graph: the first two blocks' inputs are copied inline
        # (the first block needs its x at once), the other blocks' inputs in
        # one copy on a side stream that the third block waits for (two
        # blocks' compute covers it), and each block's outputs go down on
        # another side stream as soon as the block is done.  Measured (32
        # blocks of the 8B-shaped step): every input and output in one copy
        # each, before and after the blocks, 49.3 us a block; an event wait
        # before every block breaks the programmatic-dependent-launch chain
        # between blocks (49.5 us even without outputs); outputs a block at a
        # time overlap almost fully (45.2 against 44.9 us with no copies).
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                head = min(n, 2)
                up.wait_stream(side)
                down.wait_stream(side)
                x_dev[:head * xn].copy_(x_host[:head * xn], non_blocking=True)
                rest = None
                if n > head:
                    with torch.cuda.stream(up):
                        x_dev[head * xn:n * xn].copy_(x_host[head * xn:n * xn], non_blocking=True)
                        rest = torch.cuda.Event()
                        rest.record(up)
                for i in range(n):
                    if i == head and rest is not None:
                        side.wait_event(rest)
                    blocks[i].run_eager()
                    done = torch.cuda.Event()
                    done.record(side)
                    down.wait_event(done)
                    with torch.cuda.stream(down):
                        y_host[i * yn:(i + 1) * yn].copy_(y_dev[i * yn:(i + 1) * yn],
                                                          non_blocking=True)
                side.wait_stream(up)
                side.wait_stream(down)
        torch.cuda.current_stream().wait_stream(side)
        return g
    reps = [(forward_graph(G), G)] * (steps // G)
    if steps % G:
        reps.append((forward_graph(steps % G), steps % G))
    cur = torch.cuda.current_stream()
    for s in range(max(3, -(-warmup // G))):
        reps[0][0].replay()
        cur.synchronize()
    per = []
    t0 = time.perf_counter()
    for g, n in reps:
        ts = time.perf_counter()
        g.replay()
        cur.synchronize()
        per.append((time.perf_counter() - ts) / n)
    dt = (time.perf_counter() - t0) / steps
    h2d = sum(t.numel() * t.element_size() for t in srcs)
    d2h = sum(t.numel() * t.element_size() for t in youts)
    del reps
    return dt, per, h2d, d2h


# ------------------------------------------------------------------ configs

# The workloads every default run reports beside its headline step: the
# single 1024 x 1024 layer, the Qwen3-14B-shaped MLP at each pattern, the
# Llama-3.3-70B-shaped block at each batch and the 448-layer Qwen3-32B-shaped
# stream (the Llama-3.1-8B-shaped block is the headline itself).
CONFIG_SET = ([("1", "single_1024", "2:4", 1)] +
              [("3", "qwen3_14b_mlp", p, 1) for p in ("2:4", "4:8", "1:4", "2:8")] +
              [("4", "llama33_70b_block", "2:4", b) for b in (1, 2, 3, 4, 8)] +
              [("5", "qwen3_32b_stream", "2:4", 1)])
NOMINAL_HBM_GBS = 8000.0


def graph_of(run_step, nsteps):
    """One CUDA graph of run_step(0) .. run_step(nsteps - 1)."""
    for i in range(min(nsteps, 2)):
        run_step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(nsteps):
                run_step(i)
    torch.cuda.current_stream().wait_stream(side)
    return g


def replay_samples(g, nsteps, samples):
    """Per-step seconds of `samples` timed replays of a graph of nsteps steps."""
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(samples):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) * 1e-3 / nsteps)
    return out


def config_timing(wl_key, pattern, batch, l2, samples, dense=True):
    """One workload's decode step: its layers packed, q/k/v and gate/up each
    one grouped launch, replayed from a CUDA graph of several steps that
    rotate over enough packed copies (> 3x L2) that every step streams its
    weights from HBM; and the dense cuBLAS GEMV of the same step."""
    from sparse_spmv_memory_02_b300.stream import LayerStream
    wl = nm_synth.WORKLOADS[wl_key]
    N, M = map(int, pattern.split(":"))
    comp = sum(layer.rows * (layer.K // M) * N * 2 + layer.rows * layer.K // 8
               for _, layer in layer_list(wl))
    copies = int(min(400, max(1, -(-3 * l2 // comp))))
    layers = build_workload(wl, N, M, batch, copies, keep_dense=dense)
    step_b = sum(step_bytes(layers, batch))
    streams = [LayerStream([L["mats"][c] for L in layers], [L["x"] for L in layers],
                           [L["y"] for L in layers], fuse_shared_input=True)
               for c in range(copies)]
    # at least ~50 us of work a replay, and every copy once
    est = max(comp / 6e12, 2e-6)
    nsteps = int(max(copies, min(64, -(-50e-6 // est))))
    g = graph_of(lambda i: streams[i % copies].run_eager(), nsteps)
    per = replay_samples(g, nsteps, samples)
    del g
    p10, med, p90 = percentiles(per)
    out = {"config": None, "workload": wl_key, "pattern": pattern, "batch": batch,
           "layers": len(layers), "launches_per_step": streams[0].launches,
           "copies": copies, "steps_per_sample": nsteps, "samples": len(per),
           "algorithmic_bytes": step_b, "us_per_step": med * 1e6, "us_p10": p10 * 1e6,
           "us_p90": p90 * 1e6, "gbs": step_b / med / 1e9}
    if dense:
        ys = [torch.empty_like(L["y"]) for L in layers]

        def dense_step(i):
            c = i % copies
            for j, L in enumerate(layers):
                if L["x"].dim() == 1:
                    torch.mv(L["dense"][c], L["x"], out=ys[j])
                else:
                    torch.matmul(L["x"], L["dense"][c].t(), out=ys[j])
        gd = graph_of(dense_step, nsteps)
        dper = replay_samples(gd, nsteps, samples)
        del gd
        dmed = percentiles(dper)[1]
        dbytes = sum(L["rows"] * L["K"] * 2 for L in layers)
        out["dense_us_per_step"] = dmed * 1e6
        out["dense_gbs"] = dbytes / dmed / 1e9
        out["speedup_vs_dense"] = dmed / med
    del layers, streams
    torch.cuda.empty_cache()
    return out


def read_probe(samples=10, nbytes=8 << 30):
    """The library's read-only HBM stream over an 8 GiB buffer (> 60x L2):
    median GB/s of `samples` timed calls."""
    from sparse_spmv_memory_02_b300 import nm
    buf = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    buf.fill_(1)
    sink = torch.empty(1, dtype=torch.int32, device="cuda")
    nm.nm_probe_read_stream(buf, sink)
    torch.cuda.synchronize()
    ts = []
    for _ in range(samples):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        nm.nm_probe_read_stream(buf, sink)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    del buf
    torch.cuda.empty_cache()
    p10, med, p90 = percentiles(ts)
    return {"gbs": nbytes / med / 1e9, "gbs_p10": nbytes / p90 / 1e9,
            "gbs_p90": nbytes / p10 / 1e9, "bytes": nbytes, "samples": samples,
            "kernel": "nm_probe_read_stream (libnm): 16-byte loads, one 1024-thread CTA per SM"}


def configs_pass(l2, peak, read_gbs, samples=20, dense=True):
    out = []
    for cfg, wl_key, pattern, batch in CONFIG_SET:
        r = config_timing(wl_key, pattern, batch, l2, samples, dense=dense)
        r["config"] = cfg
        r["frac_of_measured_peak"] = r["gbs"] / peak
        r["frac_of_nominal_8tbs"] = r["gbs"] / NOMINAL_HBM_GBS
        r["frac_of_read_probe"] = r["gbs"] / read_gbs if read_gbs else None
        out.append(r)
    return out


# ------------------------------------------------------------------ oracle leg

def oracle_sample(wl, N, M, batch, row_fraction, device, max_layers=None):
    """Host copies for the oracle: the first ceil(rows * fraction) rows of
    every layer of one step (or of its first max_layers layers), packed by
    the oracle itself."""
    import oracle
    sample = []
    for li, layer in layer_list(wl)[:max_layers]:
        W, mask, x = nm_synth.layer_inputs(wl, li, layer, N, M, batch, device)
        r = max(1, int(round(layer.rows * row_fraction)))
        Wn = W[:r].cpu().numpy()
        mn = mask[:r].cpu().numpy()
        xn = x.cpu().numpy()
        del W, mask
        vals, masks, bad = oracle.pack(Wn, mn, N, M)
        assert bad == 0
        sample.append((vals, masks, layer.K, xn.view("uint16")))
    return sample


def run_oracle(sample, N, M, threads):
    """Row ranges of every layer spread over host threads (the oracle's
    arithmetic is untouched; ctypes releases the GIL).  Returns (seconds,
    algorithmic bytes)."""
    import numpy as np

    import oracle
    jobs, outs = [], []
    for vals, masks, K, x in sample:
        rows = vals.shape[0]
        B = x.shape[0]
        y = np.empty((B, rows))
        s = np.empty((B, rows))
        outs.append((y, s))
        step = max(1, (rows + threads - 1) // threads)
        for r0 in range(0, rows, step):
            jobs.append((vals, masks, K, x, y, s, r0, min(rows, r0 + step)))
    idx = [0]
    lock = threading.Lock()

    def worker():
        while True:
            with lock:
                if idx[0] >= len(jobs):
                    return
                j = jobs[idx[0]]
                idx[0] += 1
            vals, masks, K, x, y, s, r0, r1 = j
            oracle.spmv_packed_rows_into(vals, masks, K, N, M, x, y, s, r0, r1)

    t0 = time.perf_counter()
    ths = [threading.Thread(target=worker) for _ in range(threads)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    dt = time.perf_counter() - t0
    nbytes = 0
    for vals, masks, K, x in sample:
        rows, B = vals.shape[0], x.shape[0]
        nbytes += vals.size * 2 + rows * K // 8 + B * K * 2 + B * rows * 2
    return dt, nbytes


# ------------------------------------------------------------------ arms

def config_block(args, wl, N, M, copies, layers_desc):
    return {"workload": wl.key, "title": wl.title, "pattern": "%d:%d" % (N, M),
            "batch": args.batch, "layers": layers_desc,
            "l2": "rotating %d packed copies of the step's weights (> 3x the 126 MB L2)" % copies,
            "launch": "%s: %s" % ("one CUDA graph per %d steps (a %d-block forward)"
                                  % (args.graph_steps, args.graph_steps)
                                  if getattr(args, "graph_steps", 1) > 1
                                  else "one CUDA graph per step", {
                "fused": "q/k/v and gate/up each one nm_spmv_group launch (they read the same "
                         "input), o and down one nm_spmv launch each",
                "fused_silu": "q/k/v one nm_spmv_group launch, o and down one nm_spmv launch "
                              "each, gate/up one nm_spmv_gate_up_silu launch writing "
                              "silu(gate x) * (up x)",
                "unfused": "one nm_spmv launch per layer"}.get(getattr(args, "launch", ""),
                                                               "one nm_spmv launch per layer")),
            "weights": "synthetic N(0,0.02), top-N |w| per group of M along K",
            "activations": ("synthetic N(0,1), 1% outlier channels x20; q/k/v share one input "
                            "vector, gate/up another" if wl.outliers else "synthetic N(0,1)")}


def run_reference(args, world, rank):
    """The oracle as it stands, on the host cores, on the same workload."""
    if rank != 0:
        return
    wl = nm_synth.WORKLOADS[args.workload]
    N, M = map(int, (args.pattern or "%d:%d" % wl.patterns[0]).split(":"))
    device = "cuda" if torch.cuda.is_available() else "cpu"
    threads = min(host_cores(), 64)
    # each step: a bounded sample, the first rows of every layer of the first
    # block, about 16 MB of packed weights (a few ms to tens of ms of CPU work)
    blk = len(wl.layers)
    blk_bytes = sum(layer.rows * (layer.K // M) * N * 2 + layer.rows * layer.K // 8
                    for _, layer in layer_list(wl)[:blk])
    frac = min(1.0, 16e6 / blk_bytes)
    sample = oracle_sample(wl, N, M, args.batch, frac, device, max_layers=blk)
    for _ in range(args.warmup):
        run_oracle(sample, N, M, threads)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = run_oracle(sample, N, M, threads)
        tot_t += dt
        tot_b += nb
    gbs = tot_b / tot_t / 1e9
    desc = [{"name": L.name, "rows": L.rows, "K": L.K} for _, L in layer_list(wl)]
    out = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": tot_t / max(1, args.steps) * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": config_block(args, wl, N, M, 0, desc),
           "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                            "sample": "per step: the first %.3g of the rows of each of the "
                                      "first %d layers, row ranges over %d host threads, fp64"
                                      % (frac, blk, threads)},
           "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_ours(args, world, rank, local):
    from sparse_spmv_memory_02_b300 import build as nmbuild
    nmbuild.build()
    wl = nm_synth.WORKLOADS[args.workload]
    N, M = map(int, (args.pattern or "%d:%d" % wl.patterns[0]).split(":"))
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    copies = max(1, args.copies)
    if workload_bytes(wl, N, M, args.batch) > 3 * l2:
        copies = 1  # one step already streams more than 3x L2
    layers = build_workload(wl, N, M, args.batch, copies, keep_dense=not args.no_dense)
    bytes_per_call = step_bytes(layers, args.batch)
    variants = {"fused": capture_step_graphs(layers, copies, fused=True),
                "unfused": capture_step_graphs(layers, copies, fused=False)}
    variant_bytes = {"fused": sum(bytes_per_call), "unfused": sum(bytes_per_call)}
    if silu_pairs(layers):
        variants["fused_silu"] = capture_step_graphs(layers, copies, fused=True, silu=True)
        variant_bytes["fused_silu"] = sum(step_bytes(layers, args.batch, silu=True))
    if args.launch not in variants:
        raise SystemExit("--launch %s: this workload has no gate/up layers" % args.launch)
    streams = variants[args.launch]
    step_b = variant_bytes[args.launch]
    others = [k for k in variants if k != args.launch]

    G = max(1, args.graph_steps)
    sampler = ClockSampler(local).start().wait_first() if rank == 0 else None
    dt, step_samples, t_wall0, t_wall1 = time_graph_steps(streams, copies, G, args.steps,
                                                          args.warmup, world)
    dt = max_over_ranks(dt, world)
    launches = streams[0].launches * args.steps
    # the same steps with one CUDA graph a step (a graph boundary every block)
    sdt, _, _, _ = time_steps(streams, copies, args.steps, args.warmup, world)
    sdt = max_over_ranks(sdt, world)
    one_graph_per_step = {"us_per_step": sdt / args.steps * 1e6,
                          "value": world * step_b * args.steps / sdt / 1e9}
    # the other launch structures of the same step, same protocol
    other_launch = {}
    for k in others:
        odt, _, _, _ = time_graph_steps(variants[k], copies, G, args.steps, args.warmup, world)
        odt = max_over_ranks(odt, world)
        other_launch[k] = {"launches_per_step": variants[k][0].launches,
                           "us_per_step": odt / args.steps * 1e6,
                           "value": variant_bytes[k] * args.steps / odt / 1e9}

    # end to end right after the device-timed steps, before the other legs
    e2e = None
    if not args.no_e2e:
        e_steps = max(20, min(args.steps, 640))
        et, eper, h2d, d2h = e2e_pass(layers, copies, e_steps, args.warmup,
                                      fused=args.launch != "unfused",
                                      silu=args.launch == "fused_silu", per_graph=G)
        ep10, emed, ep90 = percentiles(eper)
        e2e = {"value": step_b / et / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "us_per_step": et * 1e6,
               "us_per_step_p10": ep10 * 1e6, "us_per_step_p50": emed * 1e6,
               "us_per_step_p90": ep90 * 1e6,
               "path": "one CUDA graph per forward of %d steps (blocks), each block its own "
                       "input and output buffers: the blocks' x copied from a pinned host "
                       "buffer (the first two blocks' inline, the rest on a side stream that "
                       "the third block waits for), the blocks' libnm launches (%s), each "
                       "block's y copied to a pinned host buffer on another side stream once "
                       "the block is done; the host waits for the outputs once per forward "
                       "(wall clock)" % (G, args.launch)}
        bt, bper, _, _ = e2e_pass(layers, copies, max(20, min(args.steps, 500)), args.warmup,
                                  fused=args.launch != "unfused",
                                  silu=args.launch == "fused_silu", per_graph=1)
        bp10, bmed, bp90 = percentiles(bper)
        e2e["host_wait_every_step"] = {
            "value": step_b / bt / 1e9, "us_per_step": bt * 1e6, "us_per_step_p10": bp10 * 1e6,
            "us_per_step_p50": bmed * 1e6, "us_per_step_p90": bp90 * 1e6,
            "path": "one CUDA graph per step with its copies; the host waits every step"}

    # each layer alone, L2-cold, for the per-layer figures
    l2_bytes = l2
    first_block = layers[:len(wl.layers)]
    layer_t = layer_pass(first_block, args.batch, args.profile_steps, l2_bytes)
    gate_up = None
    fp = silu_pairs(first_block)
    if fp:
        gi, ui = fp[0]
        pp = pair_pass(first_block[gi], first_block[ui], args.batch, args.profile_steps, l2_bytes)
        gate_up = {k: {"us": t * 1e6, "bytes": b, "gbs": b / t / 1e9, "frac_of_peak": None}
                   for k, (t, b) in pp.items()}
        gate_up["note"] = ("the block's gate and up projections alone: one nm_spmv_group "
                           "launch writing both outputs, or one nm_spmv_gate_up_silu launch "
                           "writing silu(gate x) * (up x)")

    prune = None
    if not args.no_prune:
        pp = prune_pass(wl, N, M, args.profile_steps, l2_bytes)
        name, prow, pk = pp.pop("shape")
        prune = {k: {"us": t * 1e6, "bytes": b, "gbs": b / t / 1e9} for k, (t, b) in pp.items()}
        prune["layer"] = {"name": name, "rows": prow, "K": pk}
        prune["note"] = ("N:M selection from scores |w| * ||x_k|| (column norms of 64 synthetic "
                         "tokens) on the block's largest layer: the u8 mask, or selection and "
                         "pack in one pass; bytes = W read + scale + output written")

    crossover = None
    if not args.no_crossover:
        crossover = crossover_pass()

    calib = None
    if not args.no_calib:
        cp = calib_pass(wl, args.calib_tokens, args.profile_steps)
        calib = {"tokens": args.calib_tokens,
                 "note": "nm_calib_accumulate: H += X^T X over decode-step layer inputs "
                         "(fp16 X, fp32 H) on tcgen05 tensor cores, per distinct input width K; "
                         "flops T K (K+1) (symmetric update: tiles on and above the diagonal, "
                         "mirrored), bytes H read+write + X"}
        for K, (t, fl, by) in cp.items():
            calib["K%d" % K] = {"us": t * 1e6, "tflops": fl / t / 1e12, "gbs": by / t / 1e9}

    probe = read_probe() if rank == 0 else None
    peak0, _ = measured_peaks()
    configs = None
    if not args.no_configs and rank == 0:
        configs = configs_pass(l2, peak0, probe["gbs"] if probe else None,
                               dense=not args.no_dense)

    t_run1 = time.time()
    if sampler is not None:
        sampler.stop()
        time.sleep(0.5)  # nvidia-smi's shutdown has been seen to stall the GPU briefly
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    if clocks is not None:
        clocks["whole_run"] = sampler.summary(t_wall0, t_run1, window="from the headline "
                                              "timing to the end of the configs leg")

    dense = None
    if not args.no_dense:
        ddt, dbytes, _ = dense_pass(layers, copies, max(10, min(args.steps, 500)), args.warmup)
        dense = {"us_per_step": ddt * 1e6, "dense_bytes_per_step": dbytes,
                 "achieved_gbs": dbytes / ddt / 1e9,
                 "speedup_sparse_vs_dense": ddt / (dt / args.steps),
                 "kernel": "cuBLAS fp16 GEMV (torch.mv) on W with dropped weights zeroed"}
        for L in layers:
            L["dense"] = None
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = min(host_cores(), 64)
        # a bounded sample: about 300 MB of packed weights (the whole step
        # when it is smaller), the first rows of every layer of the first block
        blk = len(wl.layers)
        blk_bytes = sum(bytes_per_call[:blk])
        frac = min(1.0, 3e8 / blk_bytes)
        sample = oracle_sample(wl, N, M, args.batch, frac, "cuda", max_layers=blk)
        odt, ob = run_oracle(sample, N, M, threads)
        cpu = {"value": ob / odt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": "%s of the rows of the first %d layers of the step, row ranges over "
                         "%d host threads, fp64" % ("all" if frac >= 1 else "%.3g" % frac, blk,
                                                    threads),
               "seconds": odt}

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    if gate_up:
        for k in ("group", "silu"):
            gate_up[k]["frac_of_peak"] = gate_up[k]["gbs"] / peak
    if prune:
        for k in ("select_mask", "prune_pack"):
            prune[k]["frac_of_peak"] = prune[k]["gbs"] / peak
    if calib:
        tc_peak, tc_kind = measured_tc_peak()
        for k, v in calib.items():
            if k.startswith("K"):
                v["frac_of_tensor_peak"] = v["tflops"] / tc_peak
                v["frac_of_hbm_peak"] = v["gbs"] / peak
        calib["tensor_peak_tflops"] = tc_peak
        calib["tensor_peak_kind"] = tc_kind
    value = world * step_b * args.steps / dt / 1e9
    achieved = step_b * args.steps / dt / 1e9  # this rank's step: all launches are the SpMV kernel
    sp10, smed, sp90 = percentiles(step_samples)
    timing = {"samples": len(step_samples), "steps_per_sample": args.steps / len(step_samples),
              "us_per_step_p10": sp10 * 1e6, "us_per_step_p50": smed * 1e6,
              "us_per_step_p90": sp90 * 1e6, "gbs_p10": step_b / sp90 / 1e9,
              "gbs_p50": step_b / smed / 1e9, "gbs_p90": step_b / sp10 / 1e9}
    peaks = {"measured_copy_gbs": peak, "measured_kind": peak_kind,
             "nominal_gbs": NOMINAL_HBM_GBS, "read_probe": probe,
             "frac_of_measured_copy": achieved / peak,
             "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
             "frac_of_read_probe": achieved / probe["gbs"] if probe else None}
    per_layer = {}
    for L, b, lt in zip(first_block, bytes_per_call, layer_t):
        per_layer[L["name"]] = {"rows": L["rows"], "K": L["K"], "bytes": b, "us": lt * 1e6,
                                "gbs": b / lt / 1e9, "frac_of_peak": b / lt / 1e9 / peak}
    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "storage_dtype": "f16 values, 1-bit masks", "data": "synthetic",
        "config": config_block(args, wl, N, M, copies,
                               [{"name": L["name"], "rows": L["rows"], "K": L["K"]} for L in layers]),
        "us_per_call": {k: v["us"] for k, v in per_layer.items()},
        "us_per_call_note": "each layer alone, a CUDA graph of calls rotating over > 3x L2 of "
                            "packed copies",
        "per_layer": per_layer,
        "gate_up": gate_up,
        "prune": prune,
        "calib": calib,
        "crossover": crossover,
        "step_algorithmic_bytes": step_b,
        "timing": timing,
        "peaks": peaks,
        "configs": configs,
        "frac_of_peak": value / world / peak,
        "peak_gbs": peak, "peak_kind": peak_kind,
        "one_graph_per_step": one_graph_per_step,
        "launch": dict({"structure": args.launch, "launches_per_step": streams[0].launches,
                        "groups": [[layers[i]["name"] for i in g] for g in streams[0].groups]},
                       **other_launch),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": TRAFFIC_PER_LAUNCH.get(
                         (wl.key, "%d:%d" % (N, M), args.batch, args.launch)),
                     "kernel": "nm_spmv_rows_kernel (every one of the %d launches of a step)"
                               % streams[0].launches,
                     "note": "achieved = algorithmic bytes per launch / average launch time over "
                             "the timed steps (CUDA events on the replay stream, %d steps a "
                             "CUDA graph; the step's launches are all this kernel, so this "
                             "equals the step's GB/s); " % G +
                             "peak = %s copy bandwidth (read+write); a read-only stream can "
                             "exceed it" % peak_kind},
        "dense_gemv": dense,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": launches,
        "clocks": clocks,
        "gpu": torch.cuda.get_device_name(),
    }
    print(json.dumps(out), flush=True)


def percentiles(xs):
    """(p10, median, p90) of a list of samples (nearest rank)."""
    s = sorted(xs)
    pick = lambda q: s[min(len(s) - 1, max(0, int(round(q * (len(s) - 1)))))]  # noqa: E731
    return pick(0.1), statistics.median(s), pick(0.9)


def time_samples(run, samples, eager=False):
    """Seconds of each of `samples` timed runs of `run` (CUDA events on the
    current stream), replayed from one CUDA graph unless `eager`."""
    run()
    torch.cuda.synchronize()
    g = None
    if not eager:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                run()
        torch.cuda.current_stream().wait_stream(side)
    go = run if eager else g.replay
    for _ in range(3):
        go()
    torch.cuda.synchronize()
    out = []
    for _ in range(samples):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        go()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) * 1e-3)
    del g
    return out


def run_layer(args):
    """Products of the shapes in --layer (comma-separated ROWSxK), each
    pattern in --pattern (comma-separated, default 2:4) and each batch in
    --batches (default --batch), alone: one JSON line each."""
    from sparse_spmv_memory_02_b300 import build as nmbuild
    nmbuild.build()
    batches = [int(b) for b in args.batches.split(",")] if args.batches else [args.batch]
    for shape in args.layer.split(","):
        rows, K = (int(v) for v in shape.lower().split("x"))
        for pat in (args.pattern or "2:4").split(","):
            N, M = map(int, pat.split(":"))
            for B in batches:
                layer_one(args, rows, K, N, M, B)


def layer_one(args, rows, K, N, M, B):
    """One product shape alone: --calls calls a sample rotating over enough
    packed copies (> 3x L2) that every call streams its weights from HBM."""
    from sparse_spmv_memory_02_b300 import nm
    from sparse_spmv_memory_02_b300.stream import algorithmic_bytes
    W = nm_synth.weights(rows, K, args.seed, "cuda")
    mask = nm_synth.topn_mask(W, N, M)
    x = nm_synth.activations(K, B, args.seed + 500, True, "cuda")
    A = nm.nm_pack(W, mask, N, M)
    del W, mask
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    ncopy = max(2, -(-3 * l2 // A.nbytes))
    mats = [A] + [nm.PackedMatrix(A.values.clone(), A.masks.clone(), rows, K, N, M)
                  for _ in range(ncopy - 1)]
    y = torch.empty(B, rows, dtype=torch.float16, device="cuda")
    n = max(args.calls, ncopy)

    def run():
        for i in range(n):
            if B == 1:
                nm.nm_spmv(mats[i % ncopy], x[0], y[0])
            else:
                nm.nm_spmv_batched(mats[i % ncopy], x, y)
    ts = [t / n for t in time_samples(run, args.samples, eager=args.eager)]
    assert nm.nm_device_errors() == 0
    p10, med, p90 = percentiles(ts)
    nbytes = algorithmic_bytes(A, B, 2)
    peak, peak_kind = measured_peaks()
    out = {"mode": "layer", "rows": rows, "K": K, "pattern": "%d:%d" % (N, M), "batch": B,
           "calls_per_sample": n, "samples": len(ts), "copies": ncopy,
           "launch": "eager" if args.eager else "cuda graph",
           "us": med * 1e6, "us_p10": p10 * 1e6, "us_p90": p90 * 1e6,
           "algorithmic_bytes": nbytes, "gbs": nbytes / med / 1e9,
           "frac_of_peak": nbytes / med / 1e9 / peak, "peak_gbs": peak, "peak_kind": peak_kind,
           "kernel": _libnm_kernel(rows, B, K) if (N, M) == (2, 4) and K % 128 == 0 else None}
    print(json.dumps(out), flush=True)
    del mats, A, x, y
    torch.cuda.empty_cache()


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_init()
    try:
        if args.layer and args.impl == "ours":
            if not torch.cuda.is_available():
                raise SystemExit("bench.py --layer needs a CUDA GPU")
            if rank == 0:
                run_layer(args)
        elif args.impl == "reference":
            run_reference(args, world, rank)
        else:
            if not torch.cuda.is_available():
                raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
