"""The C ABI without a GPU: the library loads, exports every function that
include/nm.h declares, and rejects bad arguments on the host before any CUDA
call is made (so these checks need no device)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from sparse_spmv_memory_02_b300 import build as nmbuild
from sparse_spmv_memory_02_b300 import nm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nm.h")
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module", autouse=True)
def built():
    nmbuild.build()


def declared_functions():
    """Every function any include/*.h declares."""
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(nm_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_interface():
    assert {"nm_packed_sizes", "nm_pack", "nm_unpack", "nm_spmv", "nm_spmv_batched",
            "nm_spmv_group", "nm_spmv_gate_up_silu", "nm_select_mask", "nm_prune_pack",
            "nm_calib_accumulate",
            "nm_device_errors", "nm_status_str",
            "nm_last_error", "nm_version", "nm_pack_noalloc",
            "nm_probe_read_stream"} <= set(declared_functions())


def test_probe_checks_arguments_on_the_host():
    L = nm.lib()
    assert L.nm_probe_read_stream(None, 64, 0x1000, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_probe_read_stream(0x1008, 64, 0x1000, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_probe_read_stream(0x1000, 72, 0x1000, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_probe_read_stream(0x1000, 0, 0x1000, None) == nm.NM_OK


def test_spmv_group_checks_arguments_on_the_host():
    L = nm.lib()
    A = nm.nm_matrix(16, 64, 2, 4, A16, B16)
    B = nm.nm_matrix(16, 128, 2, 4, A16, B16)
    xp = (ctypes.c_void_p * 2)(C16, C16)
    yp = (ctypes.c_void_p * 2)(D16, D16 + 4096)
    mixed = (nm.nm_matrix * 2)(A, B)
    assert L.nm_spmv_group(mixed, 2, xp, 128, yp, None, 1, nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    assert "matrix 1" in nm.nm_last_error()
    assert L.nm_spmv_group(mixed, nm.NM_MAX_GROUP + 1, xp, 128, yp, None, 1, nm.NM_F16,
                           None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_spmv_group(mixed, -1, xp, 128, yp, None, 1, nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_spmv_group(mixed, 0, xp, 128, yp, None, 1, nm.NM_F16, None) == nm.NM_OK
    assert L.nm_spmv_group(None, 1, xp, 128, yp, None, 1, nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    same = (nm.nm_matrix * 2)(A, A)
    # per-matrix checks name the matrix: batch out of range
    assert L.nm_spmv_group(same, 2, xp, 64, yp, None, nm.NM_MAX_BATCH_TC + 1, nm.NM_F16,
                           None) == nm.NM_ERR_INVALID_ARG
    assert nm.nm_last_error().startswith("matrix 0")
    # misaligned x of the second matrix
    xbad = (ctypes.c_void_p * 2)(C16, C16 + 2)
    st = L.nm_spmv_group(same, 2, xbad, 64, yp, None, 1, nm.NM_F16, None)
    assert st in (nm.NM_ERR_INVALID_ARG, nm.NM_ERR_CUDA)


def test_gate_up_silu_checks_arguments_on_the_host():
    L = nm.lib()
    G = nm.nm_matrix(16, 128, 2, 4, A16, B16)
    U_rows = nm.nm_matrix(8, 128, 2, 4, A16, B16)
    U_pat = nm.nm_matrix(16, 128, 1, 4, A16, B16)
    assert L.nm_spmv_gate_up_silu(ctypes.byref(G), ctypes.byref(U_rows), C16, 128, D16, 16, 1,
                                  nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    assert "same rows" in nm.nm_last_error()
    assert L.nm_spmv_gate_up_silu(ctypes.byref(G), ctypes.byref(U_pat), C16, 128, D16, 16, 1,
                                  nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_spmv_gate_up_silu(None, ctypes.byref(G), C16, 128, D16, 16, 1, nm.NM_F16,
                                  None) == nm.NM_ERR_INVALID_ARG
    # per-matrix checks name the matrix: ldh < rows, batch out of range
    assert L.nm_spmv_gate_up_silu(ctypes.byref(G), ctypes.byref(G), C16, 128, D16, 8, 1,
                                  nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    assert nm.nm_last_error().startswith("gate")
    assert L.nm_spmv_gate_up_silu(ctypes.byref(G), ctypes.byref(G), C16, 128, D16, 16, 0,
                                  nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    # K not a multiple of 128: no streaming kernel, unsupported (before any launch)
    G64 = nm.nm_matrix(16, 64, 2, 4, A16, B16)
    assert L.nm_spmv_gate_up_silu(ctypes.byref(G64), ctypes.byref(G64), C16, 64, D16, 16, 1,
                                  nm.NM_F16, None) == nm.NM_ERR_UNSUPPORTED


def test_select_and_prune_pack_check_arguments_on_the_host():
    L = nm.lib()
    for f, extra in ((L.nm_select_mask, (D16,)), (L.nm_prune_pack, (D16, D16 + 4096))):
        assert f(None, None, 16, 64, 2, 4, *extra, None) == nm.NM_ERR_INVALID_ARG
        assert f(A16 + 2, None, 16, 64, 2, 4, *extra, None) == nm.NM_ERR_INVALID_ARG
        assert f(A16, B16 + 4, 16, 64, 2, 4, *extra, None) == nm.NM_ERR_INVALID_ARG
        assert f(A16, None, 16, 64, 2, 3, *extra, None) == nm.NM_ERR_UNSUPPORTED
        assert f(A16, None, 16, 62, 2, 4, *extra, None) == nm.NM_ERR_INVALID_ARG
        assert f(None, None, 0, 64, 2, 4, *extra, None) == nm.NM_OK  # nothing to do


def test_calib_accumulate_checks_arguments_on_the_host():
    L = nm.lib()
    assert L.nm_calib_accumulate(A16, 0, 64, 64, B16, 64, None) == nm.NM_OK  # no tokens
    assert L.nm_calib_accumulate(A16, 4, 0, 64, B16, 64, None) == nm.NM_OK
    assert L.nm_calib_accumulate(A16, -1, 64, 64, B16, 64, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_calib_accumulate(A16, 4, 60, 64, B16, 64, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_calib_accumulate(A16, 4, 64, 60, B16, 64, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_calib_accumulate(A16, 4, 64, 68, B16, 64, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_calib_accumulate(A16, 4, 64, 64, B16, 62, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_calib_accumulate(None, 4, 64, 64, B16, 64, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_calib_accumulate(A16 + 8, 4, 64, 64, B16, 64, None) == nm.NM_ERR_INVALID_ARG


def test_device_errors_rejects_null_on_the_host():
    assert nm.lib().nm_device_errors(None, 0, None) == nm.NM_ERR_INVALID_ARG
    assert "NULL" in nm.nm_last_error()


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", nm.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(nm_\w+)$", out, flags=re.M))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    L = nm.lib()
    for f in declared_functions():
        assert hasattr(L, f)


def test_version_and_status_strings():
    assert nm.nm_version() == int(re.search(r"#define NM_VERSION (\d+)", open(HEADER).read()).group(1))
    names = [nm.nm_status_str(s) for s in range(5)]
    assert names == ["NM_OK", "NM_ERR_INVALID_ARG", "NM_ERR_UNSUPPORTED", "NM_ERR_BAD_MASK",
                     "NM_ERR_CUDA"]
    assert nm.nm_status_str(99) == "NM_ERR_UNKNOWN"


@pytest.mark.parametrize("rows,K,N,M", [(4096, 4096, 2, 4), (3, 12, 2, 4), (5, 40, 4, 8),
                                        (1, 8, 1, 8), (0, 64, 2, 4), (7, 0, 2, 4)])
def test_packed_sizes(rows, K, N, M):
    vb, mb = nm.nm_packed_sizes(rows, K, N, M)
    assert vb == rows * (K // M) * N * 2
    assert mb == rows * ((K + 31) // 32) * 4


@pytest.mark.parametrize("rows,K,N,M,status", [
    (4, 16, 2, 16, nm.NM_ERR_UNSUPPORTED),
    (4, 16, 0, 4, nm.NM_ERR_UNSUPPORTED),
    (4, 16, 5, 4, nm.NM_ERR_UNSUPPORTED),
    (4, 18, 2, 4, nm.NM_ERR_INVALID_ARG),
    (-1, 16, 2, 4, nm.NM_ERR_INVALID_ARG),
    (4, -8, 2, 4, nm.NM_ERR_INVALID_ARG),
    (2 ** 31, 16, 2, 4, nm.NM_ERR_INVALID_ARG),
])
def test_packed_sizes_errors(rows, K, N, M, status):
    with pytest.raises(nm.NMError) as e:
        nm.nm_packed_sizes(rows, K, N, M)
    assert e.value.status == status
    assert nm.nm_last_error()


# Fake device addresses: the checks below fail before anything touches them.
A16, B16, C16, D16 = 0x10000, 0x20000, 0x30000, 0x40000


def _mat(rows=64, K=256, N=2, M=4, values=A16, masks=B16):
    return nm.nm_matrix(rows, K, N, M, values, masks)


def _spmv_b(mat, x=C16, ldx=None, y=D16, ldy=None, batch=1, yt=nm.NM_F16):
    ldx = mat.K if ldx is None else ldx
    ldy = mat.rows if ldy is None else ldy
    return nm.lib().nm_spmv_batched(ctypes.byref(mat), x, ldx, y, ldy, batch, yt, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(batch=0), nm.NM_ERR_INVALID_ARG),
    (dict(batch=nm.NM_MAX_BATCH_TC + 1), nm.NM_ERR_INVALID_ARG),
    (dict(yt=7), nm.NM_ERR_INVALID_ARG),
    (dict(ldx=255), nm.NM_ERR_INVALID_ARG),
    (dict(ldy=63), nm.NM_ERR_INVALID_ARG),
    (dict(batch=2, ldx=260), nm.NM_ERR_INVALID_ARG),      # ldx not a multiple of 8
    (dict(x=0), nm.NM_ERR_INVALID_ARG),
    (dict(y=0), nm.NM_ERR_INVALID_ARG),
    (dict(x=C16 + 8), nm.NM_ERR_INVALID_ARG),             # x not 16-byte aligned
    (dict(y=D16 + 1), nm.NM_ERR_INVALID_ARG),             # y not 2-byte aligned
    (dict(y=D16 + 2, yt=nm.NM_F32), nm.NM_ERR_INVALID_ARG),
])
def test_spmv_batched_rejects_bad_arguments(kwargs, status):
    assert _spmv_b(_mat(), **kwargs) == status
    assert nm.nm_last_error() != ""


@pytest.mark.parametrize("N,M,K", [(4, 8, 256), (1, 4, 256), (2, 8, 256), (2, 4, 192)])
def test_batch_above_8_needs_the_tensor_core_path(N, M, K):
    """Above NM_MAX_BATCH only 2:4 products with K a multiple of 128 run (on
    the tensor cores): any other pattern or K is refused on the host."""
    st = _spmv_b(_mat(K=K, N=N, M=M), ldx=K + (-K) % 8, batch=nm.NM_MAX_BATCH + 1)
    assert st == nm.NM_ERR_UNSUPPORTED
    assert "tensor-core" in nm.nm_last_error()


@pytest.mark.parametrize("mat,status", [
    (_mat(M=16), nm.NM_ERR_UNSUPPORTED),
    (_mat(N=0), nm.NM_ERR_UNSUPPORTED),
    (_mat(N=9, M=8), nm.NM_ERR_UNSUPPORTED),
    (_mat(K=258), nm.NM_ERR_INVALID_ARG),
    (_mat(rows=-1), nm.NM_ERR_INVALID_ARG),
    (_mat(values=0), nm.NM_ERR_INVALID_ARG),
    (_mat(masks=0), nm.NM_ERR_INVALID_ARG),
    (_mat(values=A16 + 2), nm.NM_ERR_INVALID_ARG),
    (_mat(masks=B16 + 4), nm.NM_ERR_INVALID_ARG),
])
def test_spmv_rejects_bad_matrix(mat, status):
    assert nm.lib().nm_spmv(ctypes.byref(mat), C16, D16, nm.NM_F16, None) == status
    assert nm.lib().nm_unpack(ctypes.byref(mat), D16, None) == status


def test_null_descriptor():
    L = nm.lib()
    assert L.nm_spmv(None, C16, D16, nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_spmv_batched(None, C16, 256, D16, 64, 1, nm.NM_F16, None) == nm.NM_ERR_INVALID_ARG
    assert L.nm_unpack(None, D16, None) == nm.NM_ERR_INVALID_ARG


def test_empty_problem_is_a_no_op_without_touching_memory():
    # rows == 0: nothing is launched, so even NULL arrays are accepted
    m = nm.nm_matrix(0, 256, 2, 4, 0, 0)
    assert nm.lib().nm_spmv(ctypes.byref(m), 0, 0, nm.NM_F16, None) == nm.NM_OK
    assert nm.lib().nm_pack(0, 0, 0, 256, 2, 4, 0, 0, None) == nm.NM_OK
    assert nm.lib().nm_pack(0, 0, 5, 0, 2, 4, 0, 0, None) == nm.NM_OK


@pytest.mark.parametrize("args,status", [
    ((A16, B16, 4, 16, 2, 3, C16, D16), nm.NM_ERR_UNSUPPORTED),
    ((A16, B16, 4, 18, 2, 4, C16, D16), nm.NM_ERR_INVALID_ARG),
    ((0, B16, 4, 16, 2, 4, C16, D16), nm.NM_ERR_INVALID_ARG),
    ((A16, 0, 4, 16, 2, 4, C16, D16), nm.NM_ERR_INVALID_ARG),
    ((A16, B16, 4, 16, 2, 4, 0, D16), nm.NM_ERR_INVALID_ARG),
    ((A16 + 1, B16, 4, 16, 2, 4, C16, D16), nm.NM_ERR_INVALID_ARG),
    ((A16, B16, 4, 16, 2, 4, C16 + 2, D16), nm.NM_ERR_INVALID_ARG),
    ((A16, B16, 4, 16, 2, 4, C16, D16 + 4), nm.NM_ERR_INVALID_ARG),
])
def test_pack_rejects_bad_arguments(args, status):
    assert nm.lib().nm_pack(*args, None) == status


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(nm, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(nm, "_lib", None)
    with pytest.raises(ImportError):
        nm.lib()


def test_binding_constants_match_the_header():
    """Every integer #define of include/nm.h that the Python binding mirrors
    (batch and group limits, device error bits, ...) has the same value, and
    the enums' values are those of the binding's names."""
    text = open(HEADER).read()
    defines = {k: int(v.rstrip("uUlL"), 0)
               for k, v in re.findall(r"#define (NM_\w+) (0x[0-9a-fA-F]+|\d+)[uUlL]*", text)}
    mirrored = [k for k in defines if hasattr(nm, k)]
    assert {"NM_MAX_BATCH", "NM_MAX_BATCH_TC", "NM_MAX_GROUP", "NM_DEVERR_PIPE_TIMEOUT",
            "NM_DEVERR_SMEM_ALIGN"} <= set(mirrored), mirrored
    for k in mirrored:
        assert getattr(nm, k) == defines[k], k
    enums = dict(re.findall(r"\b(NM_(?:OK|ERR_\w+|F16|F32))\s*=\s*(\d+)", text))
    assert len(enums) == 7, enums
    for k, v in enums.items():
        assert getattr(nm, k) == int(v), k
