"""Thin ctypes binding of libnm (include/nm.h) for PyTorch tensors.

Argument marshalling only: every step of the product runs in libnm's CUDA
kernels.  Tensors supply device memory (``data_ptr()``) and the calls are
ordered on ``torch.cuda.current_stream()`` unless a stream is given.  If the
shared library is missing the import of this module's functions fails
loudly; there is no CPU fallback.

The names mirror the C interface: nm_packed_sizes, nm_pack, nm_unpack,
nm_spmv, nm_spmv_batched, nm_device_errors, nm_status_str, nm_last_error,
nm_version.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnm.so")

NM_OK, NM_ERR_INVALID_ARG, NM_ERR_UNSUPPORTED, NM_ERR_BAD_MASK, NM_ERR_CUDA = 0, 1, 2, 3, 4
NM_F16, NM_F32 = 0, 1
NM_MAX_BATCH = 8
NM_MAX_BATCH_TC = 32
NM_MAX_GROUP = 8


class NMError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_status_name(status), message))
        self.status = status


class nm_matrix(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("K", ctypes.c_int64), ("N", ctypes.c_int32),
                ("M", ctypes.c_int32), ("values", ctypes.c_void_p), ("masks", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libnm.so with argument types declared (raises if absent)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    "libnm.so not found at %s; build it with "
                    "`python -m sparse_spmv_memory_02_b300.build`" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
            mp = ctypes.POINTER(nm_matrix)
            L.nm_packed_sizes.argtypes = [i64, i64, i32, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
            L.nm_pack.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp, vp]
            L.nm_unpack.argtypes = [mp, vp, vp]
            L.nm_spmv.argtypes = [mp, vp, vp, i32, vp]
            L.nm_spmv_batched.argtypes = [mp, vp, i64, vp, i64, i32, i32, vp]
            for f in (L.nm_packed_sizes, L.nm_pack, L.nm_unpack, L.nm_spmv, L.nm_spmv_batched):
                f.restype = ctypes.c_int
            L.nm_status_str.argtypes = [ctypes.c_int]
            L.nm_status_str.restype = ctypes.c_char_p
            L.nm_last_error.argtypes = []
            L.nm_last_error.restype = ctypes.c_char_p
            L.nm_version.argtypes = []
            L.nm_version.restype = ctypes.c_int
            L.nm_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32, vp]
            L.nm_device_errors.restype = ctypes.c_int
            L.nm_spmv_group.argtypes = [mp, i32, ctypes.POINTER(vp), i64, ctypes.POINTER(vp),
                                        ctypes.POINTER(i64), i32, i32, vp]
            L.nm_spmv_group.restype = ctypes.c_int
            L.nm_spmv_gate_up_silu.argtypes = [mp, mp, vp, i64, vp, i64, i32, i32, vp]
            L.nm_spmv_gate_up_silu.restype = ctypes.c_int
            L.nm_calib_accumulate.argtypes = [vp, i64, i64, i64, vp, i64, vp]
            L.nm_calib_accumulate.restype = ctypes.c_int
            L.nm_select_mask.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp]
            L.nm_select_mask.restype = ctypes.c_int
            L.nm_prune_pack.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp, vp]
            L.nm_prune_pack.restype = ctypes.c_int
            L.nm_probe_read_stream.argtypes = [vp, sz, vp, vp]
            L.nm_probe_read_stream.restype = ctypes.c_int
            _lib = L
    return _lib


def _status_name(status: int) -> str:
    try:
        return lib().nm_status_str(status).decode()
    except Exception:
        return "NM_STATUS_%d" % status


def nm_status_str(status: int) -> str:
    return lib().nm_status_str(status).decode()


def nm_last_error() -> str:
    return lib().nm_last_error().decode()


def nm_version() -> int:
    return lib().nm_version()


NM_DEVERR_PIPE_TIMEOUT = 1
NM_DEVERR_SMEM_ALIGN = 2


def nm_device_errors(clear: bool = True, stream=None) -> int:
    """The device error word of the current device (0 after a correct run);
    synchronises the stream, then clears the word if ``clear``."""
    flags = ctypes.c_uint32(0)
    _check(lib().nm_device_errors(ctypes.byref(flags), 1 if clear else 0, _stream(stream)))
    return flags.value


def _check(status: int):
    if status != NM_OK:
        raise NMError(status, nm_last_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check_vec(t, name):
    if t.dtype != torch.float16:
        raise TypeError("%s must be float16, got %s" % (name, t.dtype))
    if t.dim() > 0 and t.stride(-1) != 1:
        raise ValueError("%s must have unit stride along K" % name)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


@dataclass
class PackedMatrix:
    """A packed N:M matrix on the GPU: values fp16 [rows][K/M*N] and masks
    uint32 [rows][ceil(K/32)] (the layout of include/nm.h)."""
    values: torch.Tensor
    masks: torch.Tensor
    rows: int
    K: int
    N: int
    M: int

    def __post_init__(self):
        self._desc = nm_matrix(self.rows, self.K, self.N, self.M,
                               _ptr(self.values), _ptr(self.masks))

    @property
    def desc(self) -> nm_matrix:
        return self._desc

    @property
    def nbytes(self) -> int:
        return self.values.numel() * 2 + self.masks.numel() * 4


def nm_packed_sizes(rows: int, K: int, N: int, M: int):
    vb, mb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().nm_packed_sizes(rows, K, N, M, ctypes.byref(vb), ctypes.byref(mb)))
    return vb.value, mb.value


def nm_pack(W: torch.Tensor, mask: torch.Tensor, N: int, M: int,
            values: torch.Tensor | None = None, masks: torch.Tensor | None = None,
            stream=None) -> PackedMatrix:
    """Pack dense fp16 W [rows][K] with its uint8 keep-mask (synchronises)."""
    rows, K = W.shape
    vb, mb = nm_packed_sizes(rows, K, N, M)
    if values is None:
        values = torch.empty(vb // 2, dtype=torch.float16, device=W.device).view(rows, -1) \
            if rows else torch.empty(0, (K // M) * N, dtype=torch.float16, device=W.device)
    if masks is None:
        masks = torch.empty(mb // 4, dtype=torch.int32, device=W.device).view(rows, -1) \
            if rows else torch.empty(0, (K + 31) // 32, dtype=torch.int32, device=W.device)
    _check(lib().nm_pack(_ptr(W), _ptr(mask), rows, K, N, M, _ptr(values), _ptr(masks),
                         _stream(stream)))
    return PackedMatrix(values, masks, rows, K, N, M)


def nm_unpack(A: PackedMatrix, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(A.rows, A.K, dtype=torch.float16, device=A.values.device)
    _check(lib().nm_unpack(ctypes.byref(A.desc), _ptr(out), _stream(stream)))
    return out


def nm_spmv(A: PackedMatrix, x: torch.Tensor, y: torch.Tensor | None = None,
            y_dtype=torch.float16, stream=None) -> torch.Tensor:
    """y = A x for one fp16 vector x [K]."""
    _check_vec(x, "x")
    if x.shape[-1] < A.K:
        raise ValueError("x has %d entries, the matrix needs K=%d" % (x.shape[-1], A.K))
    if y is None:
        y = torch.empty(A.rows, dtype=y_dtype, device=x.device)
    yt = NM_F32 if y.dtype == torch.float32 else NM_F16
    _check(lib().nm_spmv(ctypes.byref(A.desc), _ptr(x), _ptr(y), yt, _stream(stream)))
    return y


def nm_spmv_batched(A: PackedMatrix, x: torch.Tensor, y: torch.Tensor | None = None,
                    y_dtype=torch.float16, stream=None) -> torch.Tensor:
    """y[b] = A x[b] for x [batch][ldx] (row stride = x.stride(0))."""
    _check_vec(x, "x")
    batch = x.shape[0]
    ldx = x.stride(0) if batch > 1 else x.shape[1]
    if y is None:
        y = torch.empty(batch, A.rows, dtype=y_dtype, device=x.device)
    ldy = y.stride(0) if batch > 1 else y.shape[-1]
    yt = NM_F32 if y.dtype == torch.float32 else NM_F16
    _check(lib().nm_spmv_batched(ctypes.byref(A.desc), _ptr(x), ldx, _ptr(y), ldy, batch, yt,
                                 _stream(stream)))
    return y


def nm_spmv_group(mats, xs, ys=None, y_dtype=torch.float16, stream=None):
    """y_i = A_i x_i for several matrices with the same N, M and K in one
    launch.  xs: one fp16 tensor per matrix, [K] or [batch][ldx] (the same
    tensor may be passed several times, e.g. q/k/v sharing the attention
    input); all share batch and ldx.  Returns the list of y tensors."""
    mats, xs = list(mats), list(xs)
    if len(mats) != len(xs):
        raise ValueError("need one x per matrix")
    count = len(mats)
    if count == 0:
        return []
    for i, x in enumerate(xs):
        _check_vec(x, "x[%d]" % i)
    vec = xs[0].dim() == 1
    batch = 1 if vec else xs[0].shape[0]
    ldx = xs[0].shape[-1] if (vec or batch == 1) else xs[0].stride(0)
    if ys is None:
        ys = [torch.empty(A.rows, dtype=y_dtype, device=xs[0].device) if vec else
              torch.empty(batch, A.rows, dtype=y_dtype, device=xs[0].device) for A in mats]
    ys = list(ys)
    yt = NM_F32 if ys[0].dtype == torch.float32 else NM_F16
    descs = (nm_matrix * count)(*[A.desc for A in mats])
    xp = (ctypes.c_void_p * count)(*[_ptr(x) for x in xs])
    yp = (ctypes.c_void_p * count)(*[_ptr(y) for y in ys])
    ldy = (ctypes.c_int64 * count)(*[(y.stride(0) if (y.dim() > 1 and batch > 1) else y.shape[-1])
                                     for y in ys])
    _check(lib().nm_spmv_group(descs, count, xp, ldx, yp, ldy, batch, yt, _stream(stream)))
    return ys


def nm_spmv_gate_up_silu(gate: PackedMatrix, up: PackedMatrix, x: torch.Tensor,
                         h: torch.Tensor | None = None, h_dtype=torch.float16,
                         stream=None) -> torch.Tensor:
    """h[b] = silu(gate x[b]) * (up x[b]) in one pass over both matrices;
    x [K] or [batch][ldx] fp16, h [rows] or [batch][ldh]."""
    _check_vec(x, "x")
    vec = x.dim() == 1
    batch = 1 if vec else x.shape[0]
    ldx = x.shape[-1] if (vec or batch == 1) else x.stride(0)
    if h is None:
        h = torch.empty(gate.rows, dtype=h_dtype, device=x.device) if vec else \
            torch.empty(batch, gate.rows, dtype=h_dtype, device=x.device)
    ldh = h.stride(0) if (h.dim() > 1 and batch > 1) else h.shape[-1]
    ht = NM_F32 if h.dtype == torch.float32 else NM_F16
    _check(lib().nm_spmv_gate_up_silu(ctypes.byref(gate.desc), ctypes.byref(up.desc), _ptr(x),
                                      ldx, _ptr(h), ldh, batch, ht, _stream(stream)))
    return h


def nm_select_mask(W: torch.Tensor, N: int, M: int, col_scale: torch.Tensor | None = None,
                   mask: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """u8 keep-mask [rows][K] keeping the N largest scores of every group of
    M along K: |w|, or |w| * col_scale[k] (fp32 [K]) when given."""
    if W.dtype != torch.float16 or not W.is_contiguous():
        raise ValueError("W must be a contiguous fp16 tensor")
    rows, K = W.shape
    if mask is None:
        mask = torch.empty(rows, K, dtype=torch.uint8, device=W.device)
    sp = None
    if col_scale is not None:
        if col_scale.dtype != torch.float32 or not col_scale.is_contiguous():
            raise ValueError("col_scale must be a contiguous fp32 tensor")
        sp = _ptr(col_scale)
    _check(lib().nm_select_mask(_ptr(W), sp, rows, K, N, M, _ptr(mask), _stream(stream)))
    return mask


def nm_prune_pack(W: torch.Tensor, N: int, M: int, col_scale: torch.Tensor | None = None,
                  values: torch.Tensor | None = None, masks: torch.Tensor | None = None,
                  stream=None) -> PackedMatrix:
    """nm_select_mask and nm_pack in one pass: the packed matrix of W pruned
    to N:M by score |w| or |w| * col_scale[k]."""
    if W.dtype != torch.float16 or not W.is_contiguous():
        raise ValueError("W must be a contiguous fp16 tensor")
    rows, K = W.shape
    vb, mb = nm_packed_sizes(rows, K, N, M)
    if values is None:
        values = torch.empty(vb // 2, dtype=torch.float16, device=W.device).view(rows, -1) \
            if rows else torch.empty(0, (K // M) * N, dtype=torch.float16, device=W.device)
    if masks is None:
        masks = torch.empty(mb // 4, dtype=torch.int32, device=W.device).view(rows, -1) \
            if rows else torch.empty(0, (K + 31) // 32, dtype=torch.int32, device=W.device)
    sp = None
    if col_scale is not None:
        if col_scale.dtype != torch.float32 or not col_scale.is_contiguous():
            raise ValueError("col_scale must be a contiguous fp32 tensor")
        sp = _ptr(col_scale)
    _check(lib().nm_prune_pack(_ptr(W), sp, rows, K, N, M, _ptr(values), _ptr(masks),
                               _stream(stream)))
    return PackedMatrix(values, masks, rows, K, N, M)


def nm_calib_accumulate(X: torch.Tensor, H: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """H += X^T X for fp16 X [T][K] (decode-step layer inputs) into fp32 H
    [K][K] (created zeroed if not given), on the tensor cores."""
    if X.dtype != torch.float16 or X.dim() != 2 or X.stride(1) != 1:
        raise ValueError("X must be fp16 [T][K] with unit column stride")
    T, K = X.shape
    if H is None:
        H = torch.zeros(K, K, dtype=torch.float32, device=X.device)
    if H.dtype != torch.float32 or H.dim() != 2 or H.stride(1) != 1:
        raise ValueError("H must be fp32 [K][ldh] with unit column stride")
    ldx = X.stride(0) if T > 1 else K
    _check(lib().nm_calib_accumulate(_ptr(X), T, K, ldx, _ptr(H), H.stride(0), _stream(stream)))
    return H


def nm_probe_read_stream(buf: torch.Tensor, sink: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """Read every byte of the contiguous device tensor ``buf`` once (the
    library's read-only HBM stream, include/nm_probe.h); returns the int32
    sink holding the XOR of all 32-bit words read."""
    if not buf.is_contiguous():
        raise ValueError("buf must be contiguous")
    if sink is None:
        sink = torch.empty(1, dtype=torch.int32, device=buf.device)
    _check(lib().nm_probe_read_stream(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                                      _stream(stream)))
    return sink
