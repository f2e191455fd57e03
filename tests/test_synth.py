"""The seeded input generator: reproducible, the stated distributions, and a
mask that follows the magnitude rule (checked against the oracle's rule)."""
import numpy as np
import torch

import nm_synth
import oracle


def test_weights_are_seeded_and_fp16():
    a = nm_synth.weights(64, 128, seed=5)
    b = nm_synth.weights(64, 128, seed=5)
    c = nm_synth.weights(64, 128, seed=6)
    assert a.dtype == torch.float16 and a.shape == (64, 128)
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert abs(a.float().std().item() - 0.02) < 0.002


def test_topn_mask_matches_oracle_rule_with_ties():
    W = nm_synth.small_int_weights(40, 256, seed=1, lo=-2, hi=2)  # many ties
    W[0, :8] = torch.tensor([-0.0, 0.0, -0.0, 0.0, 1, -1, 1, -1], dtype=torch.float16)
    for N, M in [(2, 4), (4, 8), (1, 4), (2, 8), (3, 4)]:
        m = nm_synth.topn_mask(W, N, M).numpy()
        ref = oracle.topn_mask(W.numpy(), N, M)
        assert np.array_equal(m, ref)
        assert np.all(m.reshape(40, -1, M).sum(-1) == N)


def test_activations_outliers():
    K = 4096
    x = nm_synth.activations(K, 3, seed=9)
    ch = nm_synth.outlier_channels(K, 9)
    assert x.shape == (3, K) and x.dtype == torch.float16
    assert len(ch) == round(0.01 * K) == len(set(ch.tolist()))
    big = x[:, ch].float().abs().mean().item()
    rest = torch.ones(K, dtype=torch.bool)
    rest[ch] = False
    small = x[:, rest].float().abs().mean().item()
    assert 10 < big / small < 30
    xp = nm_synth.activations(K, 2, seed=9, ld=K + 8)
    assert xp.shape == (2, K + 8) and torch.all(xp[:, K:] == 0)
    assert torch.equal(xp[:, :K], x[:2])


def test_random_mask_exactly_n_per_group():
    m = nm_synth.random_mask(33, 96, 3, 8, seed=2) if 96 % 8 == 0 else None
    assert m.reshape(33, 12, 8).sum(-1).eq(3).all()


def test_workload_table_shapes():
    w = nm_synth.WORKLOADS
    assert [(l.rows, l.K) for l in w["llama31_8b_block"].layers] == [
        (4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),
        (14336, 4096), (14336, 4096), (4096, 14336)]
    assert len(list(w["qwen3_32b_stream"].all_layers())) == 448
    assert w["llama33_70b_block"].batches == (1, 2, 4, 8)
    assert w["qwen3_14b_mlp"].patterns == ((2, 4), (4, 8), (1, 4), (2, 8))
    assert nm_synth.weight_seed(w["single_1024"], 0) == 0
    assert nm_synth.weight_seed(w["llama31_8b_block"], 3) == 2003
