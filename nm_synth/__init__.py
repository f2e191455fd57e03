"""Seeded synthetic inputs for the N:M SpMV workloads.

This module only draws inputs: dense fp16 weights, their magnitude-pruning
keep-mask and fp16 activation vectors.  It holds none of the packing or
product arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it without sharing any of the method's code.

Within a decoder block the query, key and value projections share one
input vector (the attention input) and gate and up share another (the MLP
input), as in the models' forward pass.

Shapes are the decoder linear layers of the models named by the pages
("SparseDecoding Makes LLM Pruning Aware of Generation", Introduction:
Llama-3.1-8B, Llama-3.3-70B, Qwen3-14B, Qwen3-32B).  No trained weights are
used: weights are N(0, 0.02) and the mask keeps the N largest |w| of every
group of M along K (ties go to the lower k); activations are N(0, 1) with
1% of the channels (a fixed seeded set, drawn without replacement) scaled
by 20 to mimic the heavy-tailed outlier channels of decode activations.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

W_STD = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_SCALE = 20.0


@dataclass(frozen=True)
class Layer:
    name: str
    rows: int  # output features
    K: int     # input features


@dataclass(frozen=True)
class Workload:
    key: str
    title: str
    layers: tuple
    patterns: tuple = ((2, 4),)
    batches: tuple = (1,)
    blocks: int = 1            # how many times the layer list repeats (weights differ)
    outliers: bool = True
    config_index: int = 0      # used for seeds: 1000 * index + layer

    def all_layers(self):
        """(global layer index, Layer) over all blocks."""
        n = len(self.layers)
        for b in range(self.blocks):
            for j, layer in enumerate(self.layers):
                yield b * n + j, layer


def _block(q, kv, o_rows, o_k, ff, hidden):
    return (Layer("q", q, hidden), Layer("k", kv, hidden), Layer("v", kv, hidden),
            Layer("o", o_rows, o_k), Layer("gate", ff, hidden), Layer("up", ff, hidden),
            Layer("down", hidden, ff))


WORKLOADS = {
    "single_1024": Workload(
        "single_1024", "single 2:4 SpMV 1024x1024, batch 1",
        (Layer("w", 1024, 1024),), outliers=False, config_index=1),
    "llama31_8b_block": Workload(
        "llama31_8b_block", "Llama-3.1-8B-shaped decoder block, 2:4, batch 1",
        _block(4096, 1024, 4096, 4096, 14336, 4096), config_index=2),
    "qwen3_14b_mlp": Workload(
        "qwen3_14b_mlp", "Qwen3-14B-shaped MLP, pattern sweep, batch 1",
        (Layer("gate", 17408, 5120), Layer("up", 17408, 5120), Layer("down", 5120, 17408)),
        patterns=((2, 4), (4, 8), (1, 4), (2, 8)), config_index=3),
    "llama33_70b_block": Workload(
        "llama33_70b_block", "Llama-3.3-70B-shaped decoder block, 2:4, batch 1/2/4/8",
        _block(8192, 1024, 8192, 8192, 28672, 8192), batches=(1, 2, 4, 8), config_index=4),
    "qwen3_32b_stream": Workload(
        "qwen3_32b_stream", "Qwen3-32B-shaped per-token weight stream, 64 blocks x 7, 2:4",
        (Layer("q", 8192, 5120), Layer("k", 1024, 5120), Layer("v", 1024, 5120),
         Layer("o", 5120, 8192), Layer("gate", 25600, 5120), Layer("up", 25600, 5120),
         Layer("down", 5120, 25600)), blocks=64, config_index=5),
}


def weight_seed(workload: Workload, layer_index: int) -> int:
    return 1000 * workload.config_index + layer_index if workload.config_index != 1 else 0


# Layers of a decoder block that read the same input vector: the query, key
# and value projections read the attention input, gate and up the MLP input.
SHARED_INPUT = {"k": "q", "v": "q", "up": "gate"}


def x_source(workload: Workload, layer_index: int) -> int:
    """Index of the layer whose input vector this layer reads (itself unless
    it shares the block's attention or MLP input with an earlier layer)."""
    n = len(workload.layers)
    block, j = divmod(layer_index, n)
    src = SHARED_INPUT.get(workload.layers[j].name)
    if src is None:
        return layer_index
    for jj, layer in enumerate(workload.layers):
        if layer.name == src:
            return block * n + jj
    return layer_index


def x_seed(workload: Workload, layer_index: int) -> int:
    return weight_seed(workload, x_source(workload, layer_index)) + 500


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weights(rows: int, K: int, seed: int, device="cpu", std: float = W_STD) -> torch.Tensor:
    """Dense fp16 [rows][K], N(0, std) drawn in fp32 and rounded to fp16."""
    g = _gen(seed, device)
    w = torch.randn(rows, K, generator=g, device=device, dtype=torch.float32)
    return (w * std).to(torch.float16)


def topn_mask(W: torch.Tensor, N: int, M: int) -> torch.Tensor:
    """uint8 keep-mask: the N largest |w| of each group of M consecutive
    weights along K; a tie goes to the lower k (|-0| equals |+0|).
    Position q is kept iff fewer than N positions of its group beat it."""
    rows, K = W.shape
    assert K % M == 0
    a = W.abs().to(torch.float32).reshape(rows, K // M, M)
    q = torch.arange(M, device=W.device)
    beaten = torch.zeros_like(a, dtype=torch.int8)
    for q2 in range(M):
        a2 = a[..., q2:q2 + 1]
        beats = (a2 > a) | ((a2 == a) & (q2 < q))
        beaten += beats.to(torch.int8)
    return (beaten < N).to(torch.uint8).reshape(rows, K)


def outlier_channels(K: int, seed: int, device="cpu") -> torch.Tensor:
    n = int(round(OUTLIER_FRACTION * K))
    g = _gen(seed + 77, "cpu")
    return torch.randperm(K, generator=g)[:n].to(device)


def activations(K: int, batch: int, seed: int, outliers: bool = True,
                device="cpu", ld: int | None = None) -> torch.Tensor:
    """fp16 [batch][ld] (ld >= K, padding columns zero): N(0, 1) per entry,
    with 1% shared outlier channels scaled by 20 when ``outliers``."""
    ld = K if ld is None else ld
    g = _gen(seed, device)
    x = torch.randn(batch, K, generator=g, device=device, dtype=torch.float32)
    if outliers:
        ch = outlier_channels(K, seed, device)
        x[:, ch] *= OUTLIER_SCALE
    out = torch.zeros(batch, ld, dtype=torch.float16, device=device)
    out[:, :K] = x.to(torch.float16)
    return out


def layer_inputs(workload: Workload, layer_index: int, layer: Layer, N: int, M: int,
                 batch: int = 1, device="cpu"):
    """(W fp16 [rows][K], mask u8 [rows][K], x fp16 [batch][K]) for one layer."""
    W = weights(layer.rows, layer.K, weight_seed(workload, layer_index), device)
    mask = topn_mask(W, N, M)
    x = activations(layer.K, batch, x_seed(workload, layer_index), workload.outliers, device)
    return W, mask, x


def random_mask(rows: int, K: int, N: int, M: int, seed: int, device="cpu") -> torch.Tensor:
    """A uniformly random valid N:M keep-mask (exactly N per group)."""
    g = _gen(seed, device)
    r = torch.rand(rows, K // M, M, generator=g, device=device)
    idx = r.argsort(dim=-1)[..., :N]
    m = torch.zeros(rows, K // M, M, dtype=torch.uint8, device=device)
    m.scatter_(-1, idx, 1)
    return m.reshape(rows, K)


def small_int_weights(rows: int, K: int, seed: int, lo: int = -8, hi: int = 8,
                      device="cpu") -> torch.Tensor:
    """Integer-valued fp16 weights (exact in fp16 and fp32 products)."""
    g = _gen(seed, device)
    return torch.randint(lo, hi + 1, (rows, K), generator=g, device=device).to(torch.float16)
