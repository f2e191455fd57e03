"""nm_pack_noalloc, the pack entry point for callers that cannot allocate
device memory (an engine that pre-reserves the GPU's memory for its own
pools, a fixed memory budget, or code that must avoid the synchronisation an
allocation can cause).  It keeps its bad-group counter in a static array
inside the library instead of allocating one per call.

Called through the C ABI with raw device pointers, it must produce exactly
what the CPU oracle's pack produces, and report the same number of bad
groups, on two calls in a row (the shared counter keeps the previous call's
contents and has to be cleared by each call); its output must also equal
nm_pack's.  Like nm_pack it synchronises its stream, so it must refuse a
capturing stream and leave the capture usable.  This file is collected last
so that a stop-at-first-failure run has run everything else before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import nm_synth
import oracle
from sparse_spmv_memory_02_b300 import build as nmbuild
from sparse_spmv_memory_02_b300 import nm


def _noalloc():
    nmbuild.build()
    f = nm.lib().nm_pack_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def test_noalloc_rejects_arguments_on_the_host():
    f = _noalloc()
    A, B, C, D = 0x10000, 0x20000, 0x30000, 0x40000  # never dereferenced
    assert f(A, B, 4, 16, 2, 3, C, D, None) == nm.NM_ERR_UNSUPPORTED
    assert f(A, B, 4, 18, 2, 4, C, D, None) == nm.NM_ERR_INVALID_ARG
    assert f(A, B, 4, 16, 2, 4, C + 8, D, None) == nm.NM_ERR_INVALID_ARG
    # beyond what the 32-bit scratch counter can count
    assert f(A, B, 2 ** 31 - 1, 16, 2, 4, C, D, None) == nm.NM_ERR_INVALID_ARG
    assert "NM_PACK_NOALLOC_MAX_GROUPS" in nm.nm_last_error()
    assert f(0, 0, 0, 16, 2, 4, 0, 0, None) == nm.NM_OK


def _oracle_pack(W, mask, N, M):
    return oracle.pack(W.cpu().numpy().view(np.uint16), mask.cpu().numpy(), N, M)


@pytest.mark.gpu
def test_noalloc_pack_matches_oracle_twice():
    f = _noalloc()
    stream = torch.cuda.current_stream().cuda_stream
    for call, (rows, K, N, M) in enumerate([(300, 4096, 2, 4), (129, 1000, 4, 8)]):
        W = nm_synth.weights(rows, K, 40 + call, "cuda")
        mask = nm_synth.topn_mask(W, N, M)
        ev, em, bad = _oracle_pack(W, mask, N, M)
        assert bad == 0
        vals = torch.full((rows, K // M * N), 7.0, dtype=torch.float16, device="cuda")
        masks = torch.full((rows, (K + 31) // 32), -1, dtype=torch.int32, device="cuda")
        st = f(W.data_ptr(), mask.data_ptr(), rows, K, N, M, vals.data_ptr(), masks.data_ptr(),
               stream)
        assert st == nm.NM_OK, nm.nm_last_error()
        torch.cuda.synchronize()
        assert np.array_equal(vals.cpu().numpy().view(np.uint16), ev)
        assert np.array_equal(masks.cpu().numpy().view(np.uint32), em)
        ref = nm.nm_pack(W, mask, N, M)  # the allocating entry point agrees
        assert torch.equal(vals.view(torch.int16), ref.values.view(torch.int16))
        assert torch.equal(masks, ref.masks)


@pytest.mark.gpu
def test_noalloc_counter_is_cleared_between_calls():
    f = _noalloc()
    stream = torch.cuda.current_stream().cuda_stream
    rows, K, N, M = 64, 256, 2, 4
    W = nm_synth.weights(rows, K, 3, "cuda")
    good = nm_synth.topn_mask(W, N, M)
    bad = good.clone()
    bad[5, 0:4] = 1
    bad[9, 8:12] = 0
    _, _, n_bad = _oracle_pack(W, bad, N, M)
    assert n_bad == 2
    vals = torch.empty(rows, K // M * N, dtype=torch.float16, device="cuda")
    masks = torch.empty(rows, (K + 31) // 32, dtype=torch.int32, device="cuda")
    args = (rows, K, N, M, vals.data_ptr(), masks.data_ptr(), stream)
    assert f(W.data_ptr(), bad.data_ptr(), *args) == nm.NM_ERR_BAD_MASK
    assert nm.nm_last_error().startswith("%d group" % n_bad)
    assert f(W.data_ptr(), good.data_ptr(), *args) == nm.NM_OK
    ev, em, _ = _oracle_pack(W, good, N, M)
    assert np.array_equal(vals.cpu().numpy().view(np.uint16), ev)
    assert np.array_equal(masks.cpu().numpy().view(np.uint32), em)


@pytest.mark.gpu
def test_noalloc_refuses_a_capturing_stream():
    f = _noalloc()
    rows, K, N, M = 64, 256, 2, 4
    W = nm_synth.weights(rows, K, 5, "cuda")
    mask = nm_synth.topn_mask(W, N, M)
    vals = torch.zeros(rows, K // M * N, dtype=torch.float16, device="cuda")
    masks = torch.zeros(rows, (K + 31) // 32, dtype=torch.int32, device="cuda")
    out = torch.zeros(1, device="cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            st = f(W.data_ptr(), mask.data_ptr(), rows, K, N, M, vals.data_ptr(),
                   masks.data_ptr(), side.cuda_stream)
            out.add_(1.0)  # the capture goes on after the refusal
    assert st == nm.NM_ERR_INVALID_ARG
    assert "captured" in nm.nm_last_error()
    g.replay()
    torch.cuda.synchronize()
    assert out.item() == 1.0
    assert not torch.any(masks)  # nothing was queued
