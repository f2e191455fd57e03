"""A decode step's linear-layer stream as one CUDA graph.

Every generated token runs the same fixed sequence of N:M SpMV calls over all
linear layers of the model (decoding is dominated by SpMV: "SparseDecoding:
Decoding-Aware Pruning for Accurate and Efficient LLM Inference", Abstract).
``LayerStream`` holds the packed matrices with their input and output
buffers, records the whole sequence once into a CUDA graph and replays it per
token, so one graph launch replaces hundreds of host-side launches.  Each
call is an ``nm_spmv_batched`` launch of libnm; nothing else runs.
"""
from __future__ import annotations

import torch

from .nm import PackedMatrix, nm_spmv, nm_spmv_batched


class LayerStream:
    def __init__(self, mats, xs, ys):
        """mats: PackedMatrix list; xs[i]: fp16 [batch][K_i] (or [K_i]);
        ys[i]: fp16/fp32 [batch][rows_i] (or [rows_i]), preallocated."""
        assert len(mats) == len(xs) == len(ys)
        self.mats = list(mats)
        self.xs = list(xs)
        self.ys = list(ys)
        self.graph = None

    def __len__(self):
        return len(self.mats)

    def run_eager(self, stream=None):
        for A, x, y in zip(self.mats, self.xs, self.ys):
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
