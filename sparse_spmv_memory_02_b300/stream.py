"""A decode step's linear-layer stream as one CUDA graph.

Every generated token runs the same fixed sequence of N:M SpMV calls over all
linear layers of the model (decoding is dominated by SpMV: "SparseDecoding:
Decoding-Aware Pruning for Accurate and Efficient LLM Inference", Abstract).
``LayerStream`` holds the packed matrices with their input and output
buffers, records the whole sequence once into a CUDA graph and replays it per
token, so one graph launch replaces hundreds of host-side launches.  Layers
that read the same input vector (the query, key and value projections; gate
and up) can be fused into one ``nm_spmv_group`` launch, and a gate/up pair
into one ``nm_spmv_gate_up_silu`` launch that writes the gated MLP input
silu(gate x) * (up x) in place of the two outputs.  Every launch is a libnm
kernel; nothing else runs.
"""
from __future__ import annotations

import torch

from .nm import PackedMatrix, nm_spmv, nm_spmv_batched, nm_spmv_gate_up_silu, nm_spmv_group


def shared_input_groups(xs, mats):
    """Consecutive layers reading the same x tensor with the same pattern and
    K, as lists of indices (singletons for the others)."""
    groups = []
    for i, (x, A) in enumerate(zip(xs, mats)):
        if groups:
            j = groups[-1][0]
            if (xs[j] is x and mats[j].K == A.K and mats[j].N == A.N and mats[j].M == A.M
                    and len(groups[-1]) < 8):
                groups[-1].append(i)
                continue
        groups.append([i])
    return groups


class LayerStream:
    def __init__(self, mats, xs, ys, fuse_shared_input: bool = False, silu_pairs=()):
        """mats: PackedMatrix list; xs[i]: fp16 [batch][K_i] (or [K_i]);
        ys[i]: fp16/fp32 [batch][rows_i] (or [rows_i]), preallocated.  With
        fuse_shared_input, consecutive layers passed the same x tensor are
        computed by one grouped launch.  silu_pairs: (gate, up) index pairs of
        consecutive layers with the same x and shape; each becomes one launch
        writing silu(gate x) * (up x) into ys[gate] (ys[up] is not written)."""
        assert len(mats) == len(xs) == len(ys)
        self.mats = list(mats)
        self.xs = list(xs)
        self.ys = list(ys)
        self.silu_pairs = {tuple(p) for p in silu_pairs}
        for gi, ui in self.silu_pairs:
            assert ui == gi + 1 and self.xs[gi] is self.xs[ui]
        groups = (shared_input_groups(self.xs, self.mats) if fuse_shared_input
                  else [[i] for i in range(len(self.mats))])
        # a pair always takes its own launch
        merged = []
        for g in groups:  # unfused: join the pair's two single-layer groups
            if (merged and len(g) == 1 and len(merged[-1]) == 1
                    and (merged[-1][0], g[0]) in self.silu_pairs):
                merged[-1] = [merged[-1][0], g[0]]
            else:
                merged.append(list(g))
        self.groups = []
        for g in merged:
            rest = list(g)
            while rest:
                pair = next(((rest[k], rest[k + 1]) for k in range(len(rest) - 1)
                             if (rest[k], rest[k + 1]) in self.silu_pairs), None)
                if pair is None:
                    self.groups.append(rest)
                    break
                k = rest.index(pair[0])
                if rest[:k]:
                    self.groups.append(rest[:k])
                self.groups.append(list(pair))
                rest = rest[k + 2:]
        self.graph = None

    def __len__(self):
        return len(self.mats)

    @property
    def launches(self) -> int:
        return len(self.groups)

    def run_eager(self, stream=None):
        for g in self.groups:
            if len(g) == 2 and tuple(g) in self.silu_pairs:
                nm_spmv_gate_up_silu(self.mats[g[0]], self.mats[g[1]], self.xs[g[0]],
                                     self.ys[g[0]], stream=stream)
                continue
            if len(g) > 1:
                nm_spmv_group([self.mats[i] for i in g], [self.xs[i] for i in g],
                              [self.ys[i] for i in g], stream=stream)
                continue
            A, x, y = self.mats[g[0]], self.xs[g[0]], self.ys[g[0]]
            if x.dim() == 1:
                nm_spmv(A, x, y, stream=stream)
            else:
                nm_spmv_batched(A, x, y, stream=stream)

    def capture(self, warmup: bool = True):
        """Record the sequence into a CUDA graph (one eager pass first so
        that every kernel is loaded before capture)."""
        if warmup:
            self.run_eager()
            torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                self.run_eager()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = g
        return g

    def replay(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()

    def compressed_bytes(self) -> int:
        return sum(A.nbytes for A in self.mats)


def algorithmic_bytes(A: PackedMatrix, batch: int = 1, y_bytes: int = 2) -> int:
    """Bytes one call must move at minimum: kept values, mask bits, x and y."""
    return (A.rows * (A.K // A.M) * A.N * 2 + A.rows * A.K // 8
            + batch * A.K * 2 + batch * A.rows * y_bytes)
