"""Python face of the plain-C oracle in ``coli_oracle.c``.

TEST INFRASTRUCTURE ONLY.  Nothing in the library package imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It compiles ``coli_oracle.c`` with gcc (OpenMP over
independent outputs) into ``oracle/_build/`` and calls it through ctypes with
numpy arrays.  All arithmetic lives in the C file; this module only marshals.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against facts the colibri pages fix (nibble extremes, fmt=4 with gs >= I equal
to fmt=2, the two evaluation orders, brute force on tiny shapes, closed forms,
library routines for the special cases) and ``tests/test_oracle_mutations.py``
shows that each planted mistake fails a pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "coli_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


class OracleMat(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("gs", ctypes.c_int), ("O", _i64), ("I", _i64),
                ("data", _ptr), ("scales", _ptr)]


def build(mutation: int = 0, openmp: bool = True) -> str:
    """Compile the oracle (optionally with one planted mistake) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    name = f"liboracle_m{mutation}.so" if mutation else "liboracle.so"
    out = os.path.join(_BUILD, name)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm",
           f"-DORACLE_MUTATION={mutation}"]
    if openmp:
        cmd.insert(1, "-fopenmp")
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def lib(mutation: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutation not in _LIBS:
            L = ctypes.CDLL(build(mutation))
            L.oracle_row_bytes.restype = _i64
            L.oracle_row_bytes.argtypes = [ctypes.c_int, _i64]
            L.oracle_scale_count.restype = _i64
            L.oracle_scale_count.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64]
            L.oracle_dequant_row.restype = ctypes.c_int
            L.oracle_dequant_row.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _ptr, _ptr, _i64, _ptr]
            L.oracle_matmul.restype = ctypes.c_int
            L.oracle_matmul.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _ptr, _ptr, _i64, _ptr,
                                        _ptr, _ptr, _ptr]
            L.oracle_matmul_inline.restype = ctypes.c_int
            L.oracle_matmul_inline.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _ptr, _ptr, _i64,
                                               _ptr, _ptr]
            L.oracle_silu.restype = ctypes.c_double
            L.oracle_silu.argtypes = [ctypes.c_double]
            L.oracle_route.restype = _i64
            L.oracle_route.argtypes = [_ptr, _i64, _i64, _i64, _ptr, _ptr]
            for fn in (L.oracle_matmul_rows, L.oracle_matmul_rows_t):
                fn.restype = ctypes.c_int
                fn.argtypes = [ctypes.c_int, ctypes.c_int, _i64, _i64, _ptr, _ptr, _i64, _i64, _i64, _i64, _i64,
                               _ptr, _ptr]
            L.oracle_moe_block.restype = ctypes.c_int
            L.oracle_moe_topk.argtypes = [_ptr, _ptr, _i64, _i64, _i64, ctypes.c_float, ctypes.c_int,
                                          ctypes.c_float, _ptr, _ptr]
            L.oracle_moe_block.argtypes = [_i64, _i64, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr, _ptr,
                                           _ptr, _ptr, _ptr]
            L.oracle_threads.restype = ctypes.c_int
            L.oracle_set_threads.restype = ctypes.c_int
            L.oracle_set_threads.argtypes = [ctypes.c_int]
            L.oracle_mutation.restype = ctypes.c_int
            _LIBS[mutation] = L
        return _LIBS[mutation]


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _data(fmt: int, data: np.ndarray) -> np.ndarray:
    if fmt == 0:
        return np.ascontiguousarray(data, dtype=np.float32)
    return np.ascontiguousarray(data).view(np.uint8)


def _scales(scales):
    return None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)


def threads(mutation: int = 0) -> int:
    return int(lib(mutation).oracle_threads())


def set_threads(n: int, mutation: int = 0) -> int:
    """Thread count of the oracle's parallel loops (for timing); returns the previous one."""
    return int(lib(mutation).oracle_set_threads(int(n)))


def row_bytes(fmt: int, I: int, mutation: int = 0) -> int:
    return int(lib(mutation).oracle_row_bytes(fmt, I))


def scale_count(fmt: int, gs: int, O: int, I: int, mutation: int = 0) -> int:
    return int(lib(mutation).oracle_scale_count(fmt, gs, O, I))


def dequant(fmt: int, gs: int, O: int, I: int, data, scales, mutation: int = 0) -> np.ndarray:
    """Whole dequantized matrix [O, I] in float64 (row by row through the oracle)."""
    d, s = _data(fmt, data), _scales(scales)
    out = np.empty((O, I), dtype=np.float64)
    L = lib(mutation)
    for o in range(O):
        rc = L.oracle_dequant_row(fmt, gs, O, I, _p(d), _p(s), o, _p(out[o]))
        if rc:
            raise ValueError("oracle_dequant_row rejected its arguments")
    return out


def matmul(fmt: int, gs: int, O: int, I: int, data, scales, x, mutation: int = 0, want=("y",)):
    """y[S, O] (f32), and on request y64 (double) and yabs (sum of |terms|)."""
    d, s = _data(fmt, data), _scales(scales)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, I)
    S = x.shape[0]
    y = np.empty((S, O), dtype=np.float32)
    y64 = np.empty((S, O), dtype=np.float64) if "y64" in want else None
    yabs = np.empty((S, O), dtype=np.float64) if "yabs" in want else None
    rc = lib(mutation).oracle_matmul(fmt, gs, O, I, _p(d), _p(s), S, _p(x), _p(y), _p(y64), _p(yabs))
    if rc:
        raise ValueError("oracle_matmul rejected its arguments")
    res = {"y": y, "y64": y64, "yabs": yabs}
    return res["y"] if want == ("y",) else tuple(res[k] for k in want)


def matmul_inline(fmt: int, gs: int, O: int, I: int, data, scales, x, mutation: int = 0) -> np.ndarray:
    d, s = _data(fmt, data), _scales(scales)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, I)
    y64 = np.empty((x.shape[0], O), dtype=np.float64)
    rc = lib(mutation).oracle_matmul_inline(fmt, gs, O, I, _p(d), _p(s), x.shape[0], _p(x), _p(y64))
    if rc:
        raise ValueError("oracle_matmul_inline rejected its arguments")
    return y64


def silu(g: float, mutation: int = 0) -> float:
    return float(lib(mutation).oracle_silu(float(g)))


def route(ids, n_experts: int, mutation: int = 0):
    """(offsets[E+1], order[n_valid]) of the stable counting sort of slots by expert."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    S, K = ids.shape
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    order = np.zeros(max(S * K, 1), dtype=np.int64)
    n = lib(mutation).oracle_route(_p(ids), S, K, n_experts, _p(offsets), _p(order))
    if n < 0:
        raise ValueError("oracle_route rejected its arguments")
    return offsets, order[:n].copy()


class Mat:
    """One quantized matrix in host layout: fmt, gs, O, I, packed data, f32 scales."""

    def __init__(self, fmt, gs, O, I, data, scales):
        self.fmt, self.gs, self.O, self.I = int(fmt), int(gs), int(O), int(I)
        self.data = _data(fmt, data)
        self.scales = _scales(scales) if fmt != 0 else None

    def c(self) -> OracleMat:
        return OracleMat(self.fmt, self.gs, self.O, self.I,
                         self.data.ctypes.data, 0 if self.scales is None else self.scales.ctypes.data)


def moe_block(H: int, F: int, experts, x, ids, w, mutation: int = 0, want=("y",)):
    """experts: list of (gate Mat, up Mat, down Mat).  Returns y [S, H] f32 (and y64)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, H)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    S, K = ids.shape
    assert x.shape[0] == S and w.shape == ids.shape
    E = len(experts)
    G = (OracleMat * E)(*[e[0].c() for e in experts])
    U = (OracleMat * E)(*[e[1].c() for e in experts])
    D = (OracleMat * E)(*[e[2].c() for e in experts])
    y = np.empty((S, H), dtype=np.float32)
    y64 = np.empty((S, H), dtype=np.float64) if "y64" in want else None
    rc = lib(mutation).oracle_moe_block(H, F, S, K, E, ctypes.cast(G, _ptr), ctypes.cast(U, _ptr),
                                        ctypes.cast(D, _ptr), _p(x), _p(ids), _p(w), _p(y), _p(y64))
    if rc:
        raise ValueError("oracle_moe_block rejected its arguments")
    return y if want == ("y",) else tuple({"y": y, "y64": y64}[k] for k in want)


def moe_topk(logits, K: int, bias=None, top_p: float = 0.0, norm_topk: bool = False, routed_scale: float = 1.0,
             mutation: int = 0):
    """Router top-K of f32 logits [S, E]: (ids [S, K] int32, w [S, K] f32)."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    S, E = logits.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ids = np.empty((S, K), dtype=np.int32)
    w = np.empty((S, K), dtype=np.float32)
    rc = lib(mutation).oracle_moe_topk(_p(logits), _p(b), S, E, K, float(top_p), int(bool(norm_topk)),
                                       float(routed_scale), _p(ids), _p(w))
    if rc:
        raise ValueError("oracle_moe_topk rejected its arguments")
    return ids, w


def matmul_rows(fmt: int, gs: int, O: int, I: int, data, scales, o0: int, stride: int, n_rows: int, n_heads: int,
                x, mutation: int = 0) -> np.ndarray:
    """Per-head row-range matvec of the absorption path: x [S][n_heads][I] -> y [S][n_heads][n_rows]."""
    d, s = _data(fmt, data), _scales(scales)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, n_heads, I)
    y = np.empty((x.shape[0], n_heads, n_rows), dtype=np.float32)
    rc = lib(mutation).oracle_matmul_rows(fmt, gs, O, I, _p(d), _p(s), o0, stride, n_rows, n_heads, x.shape[0],
                                          _p(x), _p(y))
    if rc:
        raise ValueError("oracle_matmul_rows rejected its arguments")
    return y


def matmul_rows_t(fmt: int, gs: int, O: int, I: int, data, scales, o0: int, stride: int, n_rows: int, n_heads: int,
                  x, mutation: int = 0) -> np.ndarray:
    """Transposed per-head row-range product: x [S][n_heads][n_rows] -> y [S][n_heads][I]."""
    d, s = _data(fmt, data), _scales(scales)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, n_heads, n_rows)
    y = np.empty((x.shape[0], n_heads, I), dtype=np.float32)
    rc = lib(mutation).oracle_matmul_rows_t(fmt, gs, O, I, _p(d), _p(s), o0, stride, n_rows, n_heads, x.shape[0],
                                            _p(x), _p(y))
    if rc:
        raise ValueError("oracle_matmul_rows_t rejected its arguments")
    return y
