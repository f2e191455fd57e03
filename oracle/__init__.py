"""CPU oracle for the N:M sparse matrix-vector product (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``nm_oracle.c`` (plain C, fp64
accumulation) through ctypes and shares no code with the CUDA library.

The C source states the method and every reading taken where the pages are
silent.  Sources: "SparseDecoding: Decoding-Aware Pruning for Accurate and
Efficient LLM Inference", Abstract (N:M sparse matrix-vector kernel with
bitmask indexing and fixed-step traversal); "SparseDecoding Makes LLM Pruning
Aware of Generation", Key points (same).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile nm_oracle.c into liboracle.so next to it (gcc, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load(path: str | None = None):
    global _lib
    with _lock:
        if _lib is None or path is not None:
            lib = ctypes.CDLL(path or build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_pack.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp]
            lib.oracle_pack.restype = i64
            lib.oracle_unpack.argtypes = [i64, i64, i32, i32, vp, vp, vp]
            lib.oracle_unpack.restype = None
            lib.oracle_spmv_dense_f64.argtypes = [i64, i64, vp, vp, i32, vp, i64,
                                                  vp, vp, i64, i64, i64]
            lib.oracle_spmv_dense_f64.restype = None
            lib.oracle_spmv_packed_f64.argtypes = [i64, i64, i32, i32, vp, vp, i32,
                                                   vp, i64, vp, vp, i64, i64, i64]
            lib.oracle_spmv_packed_f64.restype = None
            lib.oracle_topn_mask.argtypes = [i64, i64, i32, i32, vp, vp]
            lib.oracle_select_mask.argtypes = [i64, i64, i32, i32, vp, vp, vp]
            lib.oracle_select_mask.restype = None
            lib.oracle_calib_f64.argtypes = [i64, i64, vp, i64, vp, vp]
            lib.oracle_calib_f64.restype = None
            lib.oracle_topn_mask.restype = None
            _lib = lib
    return _lib


def use_library(path: str | None):
    """Point the wrappers at another build of nm_oracle.c (tests plant
    mistakes in a temporary copy to check that the pins catch them);
    ``None`` restores the normal build."""
    global _lib
    with _lock:
        _lib = None
    if path is not None:
        _load(path)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    """fp16 (or raw uint16) array -> contiguous uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("expected float16 or uint16 bit patterns, got %s" % a.dtype)
    return a


def values_per_row(K: int, N: int, M: int) -> int:
    return (K // M) * N


def mask_words_per_row(K: int) -> int:
    return (K + 31) // 32


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits))


def pack(W, mask, N: int, M: int):
    """Dense fp16 W[rows][K] + keep-mask -> (values u16 [rows][K/M*N],
    masks u32 [rows][ceil(K/32)], number of invalid groups)."""
    W = _u16(W)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    rows, K = W.shape
    assert mask.shape == (rows, K) and K % M == 0
    values = np.empty((rows, values_per_row(K, N, M)), dtype=np.uint16)
    masks = np.empty((rows, mask_words_per_row(K)), dtype=np.uint32)
    bad = _load().oracle_pack(rows, K, N, M, _ptr(W), _ptr(mask), _ptr(values), _ptr(masks))
    return values, masks, int(bad)


def unpack(values, masks, K: int, N: int, M: int) -> np.ndarray:
    """Packed layout -> dense uint16 bit patterns [rows][K] (dropped = +0.0)."""
    values = _u16(values)
    masks = np.ascontiguousarray(masks, dtype=np.uint32)
    rows = values.shape[0]
    out = np.empty((rows, K), dtype=np.uint16)
    _load().oracle_unpack(rows, K, N, M, _ptr(values), _ptr(masks), _ptr(out))
    return out


def _as_batch(x, K):
    x = _u16(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    assert x.shape[1] >= K
    return x


def spmv_dense(W, mask, x, row_begin: int = 0, row_end: int | None = None):
    """fp64 reference y[b][i] and s[b][i] = sum |w x| from dense W and mask.
    x is fp16 [B][K] (or [K]).  Rows outside [row_begin, row_end) are NaN."""
    W = _u16(W)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    rows, K = W.shape
    x = _as_batch(x, K)
    B, ldx = x.shape
    row_end = rows if row_end is None else row_end
    y = np.full((B, rows), np.nan)
    s = np.full((B, rows), np.nan)
    _load().oracle_spmv_dense_f64(rows, K, _ptr(W), _ptr(mask), B, _ptr(x), ldx,
                                  _ptr(y), _ptr(s), rows, row_begin, row_end)
    return y, s


def spmv_packed(values, masks, K: int, N: int, M: int, x,
                row_begin: int = 0, row_end: int | None = None):
    """fp64 reference from the packed layout (bitmask walk, fixed step)."""
    values = _u16(values)
    masks = np.ascontiguousarray(masks, dtype=np.uint32)
    rows = values.shape[0]
    x = _as_batch(x, K)
    B, ldx = x.shape
    row_end = rows if row_end is None else row_end
    y = np.full((B, rows), np.nan)
    s = np.full((B, rows), np.nan)
    _load().oracle_spmv_packed_f64(rows, K, N, M, _ptr(values), _ptr(masks), B,
                                   _ptr(x), ldx, _ptr(y), _ptr(s), rows,
                                   row_begin, row_end)
    return y, s


def spmv_packed_rows_into(values, masks, K, N, M, x, y, s, row_begin, row_end):
    """Row-range call writing into caller arrays (used to split rows over
    host threads when the oracle is timed; the arithmetic is unchanged)."""
    B, ldx = x.shape
    _load().oracle_spmv_packed_f64(values.shape[0], K, N, M, _ptr(values), _ptr(masks),
                                   B, _ptr(x), ldx, _ptr(y), _ptr(s), y.shape[1],
                                   row_begin, row_end)


def topn_mask(W, N: int, M: int) -> np.ndarray:
    """Keep the N largest |w| of every group of M along K (ties -> lower k)."""
    W = _u16(W)
    rows, K = W.shape
    mask = np.empty((rows, K), dtype=np.uint8)
    _load().oracle_topn_mask(rows, K, N, M, _ptr(W), _ptr(mask))
    return mask


def select_mask(W, N: int, M: int, scale=None) -> np.ndarray:
    """Keep the N largest scores of every group of M along K, score |w| or
    |w| * scale[k] in fp32 (ties -> lower k)."""
    W = _u16(W)
    rows, K = W.shape
    mask = np.empty((rows, K), dtype=np.uint8)
    sp = None
    if scale is not None:
        scale = np.ascontiguousarray(scale, dtype=np.float32)
        assert scale.shape == (K,)
        sp = _ptr(scale)
    _load().oracle_select_mask(rows, K, N, M, _ptr(W), sp, _ptr(mask))
    return mask


def calib_accumulate(X, H0=None):
    """fp64 reference of H0 + X^T X (X fp16 [T][K]) and S = sum_t |x_ti x_tj|.
    Returns (H, S), both [K][K] float64."""
    X = _u16(X)
    T, K = X.shape
    H = np.zeros((K, K)) if H0 is None else np.array(H0, dtype=np.float64, copy=True)
    S = np.empty((K, K))
    _load().oracle_calib_f64(T, K, _ptr(X), K, _ptr(H), _ptr(S))
    return H, S


def calib_within_tolerance(H_gpu, H_ref, S, rel: float = 1e-3):
    """|H - H_ref| <= rel * S + 2**-22 |H_ref| + 1e-6: the products are exact
    in fp32, the sums over tokens carry fp32 rounding (bounded by rel * S),
    and adding to an existing H rounds once more."""
    H_gpu = np.asarray(H_gpu, dtype=np.float64)
    return np.abs(H_gpu - H_ref) <= rel * S + 2.0 ** -22 * np.abs(H_ref) + 1e-6


def silu(g):
    """silu(g) = g / (1 + exp(-g)) in fp64, elementwise (exp overflow for
    g < -709 gives -0.0, the limit)."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


# Largest slope of silu: silu'(g) = s(g) (1 + g (1 - s(g))), s the logistic
# function; its maximum, about 1.0998 near g = 2.3994, rounded up.
SILU_LIPSCHITZ = 1.1


def gate_up_silu(Wg, mg, Wu, mu, x, rel: float = 1e-3, abs_: float = 1e-6):
    """Reference h[b][i] = silu(g) * u with g = (Wg (.) mg) x_b and
    u = (Wu (.) mu) x_b computed by spmv_dense in fp64, and a per-element
    bound on |h - h_ref| for a kernel whose g and u each meet the SpMV
    tolerance |d| <= rel * s + abs_:
        L e_g (|u| + e_u) + |silu(g)| e_u + 2**-10 |h| + 1e-6
    (silu is L-Lipschitz; the last terms cover evaluating silu and the
    product in fp32 and rounding h to fp16).  Returns (h_ref, bound)."""
    g, sg = spmv_dense(Wg, mg, x)
    u, su = spmv_dense(Wu, mu, x)
    eg = rel * sg + abs_
    eu = rel * su + abs_
    h = silu(g) * u
    bound = (SILU_LIPSCHITZ * eg * (np.abs(u) + eu) + np.abs(silu(g)) * eu
             + 2.0 ** -10 * np.abs(h) + 1e-6)
    return h, bound


def within_tolerance(y_gpu, y_ref, s_ref, rel: float = 1e-3, abs_: float = 1e-6):
    """Per-element acceptance rule |y - y_ref| <= rel * s + abs."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    return np.abs(y_gpu - y_ref) <= rel * s_ref + abs_
