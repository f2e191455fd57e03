"""A decode step's linear-layer stream as one CUDA graph.

Every generated token runs the same fixed sequence of N:M SpMV calls over all
linear layers of the model (decoding is dominated by SpMV: "SparseDecoding:
Decoding-Aware Pruning for Accurate and Efficient LLM Inference", Abstract).
``LayerStream`` holds the packed matrices with their input and output
buffers, records the whole sequence once into a CUDA graph and replays it per
token, so one graph launch replaces hundreds of host-side launches.  Layers
that read the same input vector (the query, key and value projections; gate
and up) can be fused into one ``nm_spmv_group`` launch.  Every launch is a
libnm kernel; nothing else runs.
"""
from __future__ import annotations

import torch

from .nm import PackedMatrix, nm_spmv, nm_spmv_batched, nm_spmv_group


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
    def __init__(self, mats, xs, ys, fuse_shared_input: bool = False):
        """mats: PackedMatrix list; xs[i]: fp16 [batch][K_i] (or [K_i]);
        ys[i]: fp16/fp32 [batch][rows_i] (or [rows_i]), preallocated.  With
        fuse_shared_input, consecutive layers passed the same x tensor are
        computed by one grouped launch."""
        assert len(mats) == len(xs) == len(ys)
        self.mats = list(mats)
        self.xs = list(xs)
        self.ys = list(ys)
        self.groups = (shared_input_groups(self.xs, self.mats) if fuse_shared_input
                       else [[i] for i in range(len(self.mats))])
        self.graph = None

    def __len__(self):
        return len(self.mats)

    @property
    def launches(self) -> int:
        return len(self.groups)

    def run_eager(self, stream=None):
        for g in self.groups:
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
