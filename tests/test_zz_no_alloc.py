"""nm_pack_noalloc, the pack entry point for callers that cannot allocate
device memory (an engine that pre-reserves the GPU's memory for its own
pools, a fixed memory budget, or code that must avoid the synchronisation an
allocation can cause).  It keeps its bad-group counter in a static array
inside the library instead of allocating one per call.

Called through the C ABI with raw device pointers, it must produce exactly
what nm_pack produces, on two calls in a row (the shared counter keeps the
previous call's contents and has to be cleared by each call).  This file is
collected last so that a stop-at-first-failure run has run everything else
before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import nm_synth
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


@pytest.mark.gpu
def test_noalloc_pack_matches_nm_pack_twice():
    f = _noalloc()
    stream = torch.cuda.current_stream().cuda_stream
    for call, (rows, K, N, M) in enumerate([(300, 4096, 2, 4), (129, 1000, 4, 8)]):
        W = nm_synth.weights(rows, K, 40 + call, "cuda")
        mask = nm_synth.topn_mask(W, N, M)
        ref = nm.nm_pack(W, mask, N, M)
        vals = torch.full_like(ref.values, 7.0)
        masks = torch.full_like(ref.masks, -1)
        st = f(W.data_ptr(), mask.data_ptr(), rows, K, N, M, vals.data_ptr(), masks.data_ptr(),
               stream)
        assert st == nm.NM_OK, nm.nm_last_error()
        torch.cuda.synchronize()
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
    vals = torch.empty(rows, K // M * N, dtype=torch.float16, device="cuda")
    masks = torch.empty(rows, (K + 31) // 32, dtype=torch.int32, device="cuda")
    args = (rows, K, N, M, vals.data_ptr(), masks.data_ptr(), stream)
    assert f(W.data_ptr(), bad.data_ptr(), *args) == nm.NM_ERR_BAD_MASK
    assert nm.nm_last_error().startswith("2 group")
    assert f(W.data_ptr(), good.data_ptr(), *args) == nm.NM_OK
    ref = nm.nm_pack(W, good, N, M)
    assert np.array_equal(vals.cpu().numpy().view(np.uint16), ref.values.cpu().numpy().view(np.uint16))
