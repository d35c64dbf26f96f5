"""Python binding of libcoli.so (include/coli.h): argument marshalling only.

Every computation runs in the CUDA library.  There is no other
implementation: if libcoli.so is missing this module raises ImportError
(build it with ``python bit_weight_gemv_fmt1_gb300/build.py`` or
``__graft_entry__.build()``), and every library error is raised as
ColiError with the library's message.

Tensors are passed as torch CUDA tensors (their data pointers) and numpy
arrays (host uploads); ``stream`` defaults to torch's current stream.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcoli.so")

COLI_OK, COLI_EINVAL, COLI_EFMT, COLI_ENOMEM, COLI_ECUDA, COLI_ETIMEOUT, COLI_EINJECTED, COLI_EDEVICE = \
    0, -1, -2, -3, -4, -5, -6, -7
_NAMES = {-1: "COLI_EINVAL", -2: "COLI_EFMT", -3: "COLI_ENOMEM", -4: "COLI_ECUDA", -5: "COLI_ETIMEOUT",
          -6: "COLI_EINJECTED", -7: "COLI_EDEVICE"}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: the CUDA library has not been built "
                      "(run __graft_entry__.build() or bit_weight_gemv_fmt1_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i64, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int


class _Stats(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("launches", ctypes.c_uint64), ("weight_bytes", ctypes.c_uint64)]


class _Expert(ctypes.Structure):
    _fields_ = [("gate", _vp), ("up", _vp), ("down", _vp)]


_lib.coli_version.restype = ctypes.c_char_p
_lib.coli_last_error.restype = ctypes.c_char_p
_lib.coli_tensor_upload.argtypes = [_int, _int, _i64, _i64, _vp, _vp, _vp, ctypes.POINTER(_vp)]
_lib.coli_tensor_upload_host.argtypes = [_int, _int, _i64, _i64, _vp, _vp, ctypes.POINTER(_vp)]
_lib.coli_tensor_free.argtypes = [_vp]
_lib.coli_tensor_free.restype = None
_lib.coli_tensor_info.argtypes = [_vp] + [ctypes.POINTER(_int)] * 2 + [ctypes.POINTER(_i64)] * 4
_lib.coli_matmul.argtypes = [_vp, _vp, _vp, _int, _vp]
_lib.coli_matmul_multi.argtypes = [_int, ctypes.POINTER(_vp), _vp, ctypes.POINTER(_vp), _int, _vp]
_lib.coli_matmul_rows.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp, _int, _vp]
_lib.coli_matmul_rows_t.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _vp, _int, _vp]
_lib.coli_moe_route.argtypes = [_vp, _int, _int, _int, _vp, _vp, _vp]
_lib.coli_moe_block.argtypes = [_vp, _int, ctypes.POINTER(_Expert), _int, _vp, _vp, _int, _vp, _vp]
_lib.coli_moe_block_noalloc.argtypes = [_vp, _int, ctypes.POINTER(_Expert), _int, _vp, _vp, _int, _vp, _vp, _vp]
_lib.coli_expert_table_create.argtypes = [ctypes.POINTER(_Expert), _int, ctypes.POINTER(_vp)]
_lib.coli_expert_table_free.argtypes = [_vp]
_lib.coli_expert_table_free.restype = None
_lib.coli_moe_block_t.argtypes = [_vp, _int, _vp, _vp, _vp, _int, _vp, _vp]
_lib.coli_moe_topk.argtypes = [_vp, _vp, _int, _int, _int, ctypes.c_float, _int, ctypes.c_float, _vp, _vp, _vp]
_lib.coli_moe_router.argtypes = [_vp, _int, _vp, _vp, _int, ctypes.c_float, _int, ctypes.c_float, _vp, _vp, _vp]
_lib.coli_sync_check.argtypes = [_vp]
_lib.coli_get_stats.argtypes = [ctypes.POINTER(_Stats)]
_lib.coli_get_stats.restype = None
_lib.coli_reset_stats.restype = None
_lib.coli_set_fail_after.argtypes = [_i64]
_lib.coli_set_fail_after.restype = None

EXPORTS = ("coli_tensor_upload", "coli_tensor_upload_host", "coli_tensor_free", "coli_tensor_info", "coli_matmul", "coli_matmul_multi",
           "coli_matmul_rows", "coli_matmul_rows_t",
           "coli_moe_route", "coli_moe_topk", "coli_moe_router", "coli_moe_block", "coli_moe_block_noalloc",
           "coli_expert_table_create", "coli_expert_table_free", "coli_moe_block_t",
           "coli_sync_check", "coli_last_error", "coli_get_stats", "coli_reset_stats", "coli_set_fail_after",
           "coli_version")


class ColiError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


def _check(rc: int):
    if rc != COLI_OK:
        raise ColiError(rc, _lib.coli_last_error().decode())


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def version() -> str:
    return _lib.coli_version().decode()


class Tensor:
    """An uploaded weight matrix (owns its device memory)."""

    def __init__(self, handle: int, fmt: int, gs: int, O: int, I: int):
        self._h = handle
        self.fmt, self.gs, self.O, self.I = fmt, gs, O, I

    @property
    def handle(self) -> int:
        return self._h

    def info(self) -> dict:
        f, g = _int(), _int()
        O, I, db, ab = _i64(), _i64(), _i64(), _i64()
        _check(_lib.coli_tensor_info(self._h, f, g, O, I, db, ab))
        return dict(fmt=f.value, gs=g.value, O=O.value, I=I.value, device_bytes=db.value, alg_bytes=ab.value)

    def free(self):
        if self._h:
            _lib.coli_tensor_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def tensor_upload(fmt: int, gs: int, O: int, I: int, data: np.ndarray, scales: np.ndarray | None,
                  stream=None) -> Tensor:
    data = np.ascontiguousarray(data)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    out = _vp()
    _check(_lib.coli_tensor_upload(int(fmt), int(gs), int(O), int(I), data.ctypes.data,
                                   None if sc is None else sc.ctypes.data, _stream(stream), ctypes.byref(out)))
    return Tensor(out.value, int(fmt), int(gs), int(O), int(I))


def tensor_upload_host(fmt: int, gs: int, O: int, I: int, data: np.ndarray, scales: np.ndarray | None) -> Tensor:
    """As tensor_upload, but the weights stay in pinned host memory and the
    kernels read them zero-copy over the CPU-GPU link."""
    data = np.ascontiguousarray(data)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    out = _vp()
    _check(_lib.coli_tensor_upload_host(int(fmt), int(gs), int(O), int(I), data.ctypes.data,
                                        None if sc is None else sc.ctypes.data, ctypes.byref(out)))
    return Tensor(out.value, int(fmt), int(gs), int(O), int(I))


def matmul(W: Tensor, x, y, S: int | None = None, stream=None):
    """y[S, O] = x[S, I] @ W^T (x, y: contiguous float32 CUDA tensors)."""
    S = x.shape[0] if S is None else S
    _check(_lib.coli_matmul(W.handle, _ptr(x), _ptr(y), int(S), _stream(stream)))
    return y


def matmul_rows(W: Tensor, o0: int, stride: int, n_rows: int, n_heads: int, x, y, S: int | None = None,
                stream=None):
    """Per-head row-range matvec of the kv_b absorption path:
    y[s, h, j] = sum_i W[o0 + h*stride + j, i] * x[s, h, i]  (x [S, n_heads, I], y [S, n_heads, n_rows])."""
    S = x.shape[0] if S is None else S
    _check(_lib.coli_matmul_rows(W.handle, int(o0), int(stride), int(n_rows), int(n_heads), _ptr(x), _ptr(y), int(S),
                                 _stream(stream)))
    return y


def matmul_rows_t(W: Tensor, o0: int, stride: int, n_rows: int, n_heads: int, x, y, S: int | None = None,
                  stream=None):
    """Transposed per-head product: y[s, h, i] = sum_j x[s, h, j] * W[o0 + h*stride + j, i]
    (x [S, n_heads, n_rows], y [S, n_heads, I])."""
    S = x.shape[0] if S is None else S
    _check(_lib.coli_matmul_rows_t(W.handle, int(o0), int(stride), int(n_rows), int(n_heads), _ptr(x), _ptr(y),
                                   int(S), _stream(stream)))
    return y


def matmul_multi(Ws, x, ys, S: int | None = None, stream=None):
    n = len(Ws)
    S = x.shape[0] if S is None else S
    Wa = (_vp * n)(*[w.handle for w in Ws])
    Ya = (_vp * n)(*[_ptr(y) for y in ys])
    _check(_lib.coli_matmul_multi(n, Wa, _ptr(x), Ya, int(S), _stream(stream)))
    return ys


def moe_route(ids, n_experts: int, offsets, order, stream=None):
    S, K = ids.shape
    _check(_lib.coli_moe_route(_ptr(ids), int(S), int(K), int(n_experts), _ptr(offsets), _ptr(order),
                               _stream(stream)))
    return offsets, order


def moe_topk(logits, K: int, ids, w, bias=None, top_p: float = 0.0, norm_topk: bool = False,
             routed_scale: float = 1.0, stream=None):
    """Router top-K of device f32 logits [S, E] into ids [S, K] int32 and w [S, K] f32 (see coli.h)."""
    S, E = logits.shape
    _check(_lib.coli_moe_topk(_ptr(logits), _ptr(bias), int(S), int(E), int(K), float(top_p), int(bool(norm_topk)),
                              float(routed_scale), _ptr(ids), _ptr(w), _stream(stream)))
    return ids, w


def moe_router(x, router: Tensor, K: int, ids, w, bias=None, top_p: float = 0.0, norm_topk: bool = False,
               routed_scale: float = 1.0, stream=None):
    """logits = x @ router^T, then moe_topk (one call, see coli.h)."""
    S = x.shape[0]
    _check(_lib.coli_moe_router(_ptr(x), int(S), router.handle, _ptr(bias), int(K), float(top_p),
                                int(bool(norm_topk)), float(routed_scale), _ptr(ids), _ptr(w), _stream(stream)))
    return ids, w


class ExpertTable:
    """An expert table: the host array of coli_expert descriptors (keeps the
    tensors alive) and, from the first block call on, the library's checked
    device copy (coli_expert_table_create), freed with the object."""

    def __init__(self, experts):
        self.experts = list(experts)
        self.arr = (_Expert * len(self.experts))(*[_Expert(g.handle, u.handle, d.handle)
                                                   for (g, u, d) in self.experts])
        self._t = None

    def __len__(self):
        return len(self.experts)

    def handle(self) -> int:
        if self._t is None:
            h = _vp()
            _check(_lib.coli_expert_table_create(self.arr, len(self.experts), ctypes.byref(h)))
            self._t = h.value
        return self._t

    def __del__(self):
        if getattr(self, "_t", None):
            _lib.coli_expert_table_free(self._t)
            self._t = None


def moe_block(x, table: ExpertTable, ids, w, y, stream=None):
    """coli_moe_block_t on the table's device copy."""
    S, K = ids.shape
    _check(_lib.coli_moe_block_t(_ptr(x), int(S), table.handle(), _ptr(ids), _ptr(w), int(K), _ptr(y),
                                 _stream(stream)))
    return y


def moe_block_array(x, table: ExpertTable, ids, w, y, stream=None):
    """coli_moe_block on the host array (the table is checked on every call)."""
    S, K = ids.shape
    _check(_lib.coli_moe_block(_ptr(x), int(S), table.arr, len(table), _ptr(ids), _ptr(w), int(K), _ptr(y),
                               _stream(stream)))
    return y


def moe_block_noalloc(x, table: ExpertTable, ids, w, y, dev_error, stream=None):
    """The decode expert block without any device allocation (see coli.h);
    dev_error is a 1-element int32 CUDA tensor that receives the kernel's
    error code (0 = none)."""
    S, K = ids.shape
    _check(_lib.coli_moe_block_noalloc(_ptr(x), int(S), table.arr, len(table), _ptr(ids), _ptr(w), int(K), _ptr(y),
                                       _ptr(dev_error), _stream(stream)))
    return y


def sync_check(stream=None):
    _check(_lib.coli_sync_check(_stream(stream)))


def stats() -> dict:
    s = _Stats()
    _lib.coli_get_stats(ctypes.byref(s))
    return dict(calls=s.calls, launches=s.launches, weight_bytes=s.weight_bytes)


def reset_stats():
    _lib.coli_reset_stats()


def set_fail_after(n: int):
    _lib.coli_set_fail_after(int(n))


def last_error() -> str:
    return _lib.coli_last_error().decode()
