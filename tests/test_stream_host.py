"""Host logic of the decode-step layer stream (no GPU): which layers share a
launch and which call each launch makes.  Matrices are stand-ins with the
shape fields the grouping reads; the library calls are replaced by recorders
so only the dispatch is exercised."""
from types import SimpleNamespace

import pytest
import torch

from sparse_spmv_memory_02_b300 import stream as st


def _mat(K, N=2, M=4, rows=64):
    return SimpleNamespace(K=K, N=N, M=M, rows=rows)


def _block(batch=1):
    """q, k, v, o, gate, up, down of a decoder block: q/k/v share the
    attention input, gate/up the MLP input."""
    K, F = 64, 128
    xa = torch.zeros(batch, K)
    xo = torch.zeros(batch, K)
    xm = torch.zeros(batch, K)
    xd = torch.zeros(batch, F)
    mats = [_mat(K), _mat(K), _mat(K), _mat(K), _mat(K, rows=F), _mat(K, rows=F), _mat(F)]
    xs = [xa, xa, xa, xo, xm, xm, xd]
    ys = [torch.zeros(batch, m.rows) for m in mats]
    return mats, xs, ys


def test_shared_input_groups_follow_the_block():
    mats, xs, _ = _block()
    assert st.shared_input_groups(xs, mats) == [[0, 1, 2], [3], [4, 5], [6]]


def test_groups_split_on_pattern_k_and_size():
    x = torch.zeros(1, 64)
    mats = [_mat(64), _mat(64, 4, 8), _mat(64, 4, 8), _mat(128), _mat(128)]
    xs = [x, x, x, x, x]
    # another pattern, then another K, start new groups
    assert st.shared_input_groups(xs, mats) == [[0], [1, 2], [3, 4]]
    many = [_mat(64) for _ in range(11)]
    assert st.shared_input_groups([x] * 11, many) == [list(range(8)), [8, 9, 10]]


@pytest.mark.parametrize("fuse,pairs,groups", [
    (True, (), [[0, 1, 2], [3], [4, 5], [6]]),
    (False, (), [[0], [1], [2], [3], [4], [5], [6]]),
    (True, [(4, 5)], [[0, 1, 2], [3], [4, 5], [6]]),
    (False, [(4, 5)], [[0], [1], [2], [3], [4, 5], [6]]),
])
def test_layer_stream_launch_structure(fuse, pairs, groups):
    mats, xs, ys = _block()
    s = st.LayerStream(mats, xs, ys, fuse_shared_input=fuse, silu_pairs=pairs)
    assert s.groups == groups
    assert s.launches == len(groups)
    assert len(s) == 7


def test_pair_inside_a_shared_input_group_takes_its_own_launch():
    x = torch.zeros(1, 64)
    mats = [_mat(64) for _ in range(5)]
    s = st.LayerStream(mats, [x] * 5, [torch.zeros(1, 64) for _ in range(5)],
                       fuse_shared_input=True, silu_pairs=[(1, 2)])
    assert s.groups == [[0], [1, 2], [3, 4]]


def test_pair_must_be_consecutive_and_share_x():
    mats, xs, ys = _block()
    with pytest.raises(AssertionError):
        st.LayerStream(mats, xs, ys, silu_pairs=[(3, 4)])  # o and gate read different x
    with pytest.raises(AssertionError):
        st.LayerStream(mats, xs, ys, silu_pairs=[(4, 6)])


def test_run_eager_dispatches_each_launch_once(monkeypatch):
    calls = []

    def idx(m):  # by identity: the stand-ins of equal shape compare equal
        return next(i for i, mm in enumerate(mats) if mm is m)
    monkeypatch.setattr(st, "nm_spmv_group", lambda ms, x, y, stream=None: calls.append(
        ("group", [idx(m) for m in ms])))
    monkeypatch.setattr(st, "nm_spmv_gate_up_silu", lambda g, u, x, h, stream=None: calls.append(
        ("silu", [idx(g), idx(u)])))
    monkeypatch.setattr(st, "nm_spmv_batched", lambda A, x, y, stream=None: calls.append(
        ("batched", [idx(A)])))
    monkeypatch.setattr(st, "nm_spmv", lambda A, x, y, stream=None: calls.append(
        ("single", [idx(A)])))
    mats, xs, ys = _block(batch=2)
    st.LayerStream(mats, xs, ys, fuse_shared_input=True, silu_pairs=[(4, 5)]).run_eager()
    assert calls == [("group", [0, 1, 2]), ("batched", [3]), ("silu", [4, 5]), ("batched", [6])]
    calls.clear()
    mats1 = [_mat(64)]
    mats[:] = mats1
    st.LayerStream(mats1, [torch.zeros(64)], [torch.zeros(64)]).run_eager()
    assert calls == [("single", [0])]


def test_algorithmic_bytes_counts_each_operand_once():
    A = _mat(4096, 2, 4, rows=1024)
    # values rows*K/2*2 bytes, masks rows*K/8, x and y of fp16 for 3 vectors
    assert st.algorithmic_bytes(A, batch=3) == (1024 * 4096 + 1024 * 4096 // 8
                                                + 3 * 4096 * 2 + 3 * 1024 * 2)
    assert st.algorithmic_bytes(A, batch=1, y_bytes=4) == (1024 * 4096 + 1024 * 4096 // 8
                                                           + 4096 * 2 + 1024 * 4)
