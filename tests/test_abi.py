"""The C ABI on the CPU: the library loads, exports every entry point that
include/coli.h declares, and refuses bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coli.h")


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(coli_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._load_build_module().build()
    return ctypes.CDLL(path)


def test_header_declares_entry_points():
    names = declared()
    for n in ("coli_tensor_upload", "coli_matmul", "coli_moe_block", "coli_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared() if not hasattr(lib, n)]
    assert not missing, f"declared in coli.h but not exported: {missing}"


def test_binding_exports_match_header():
    import bit_weight_gemv_fmt1_gb300 as coli
    assert sorted(coli.EXPORTS) == declared()


def test_version(lib):
    lib.coli_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.coli_version()


@pytest.mark.parametrize("fmt,gs,code", [(5, 0, -2), (5, 4, -2), (5, 12, -2), (6, 0, -2), (8, 0, -2), (-1, 0, -2),
                                         (4, 0, -2), (4, 63, -2), (4, 1, -2)])
def test_upload_refuses_bad_format(lib, fmt, gs, code):
    lib.coli_last_error.restype = ctypes.c_char_p
    out = ctypes.c_void_p(123)
    buf = (ctypes.c_uint8 * 64)()
    sc = (ctypes.c_float * 64)()
    rc = lib.coli_tensor_upload(fmt, gs, ctypes.c_int64(4), ctypes.c_int64(8), buf, sc, None, ctypes.byref(out))
    assert rc == code
    assert out.value is None
    assert lib.coli_last_error()
    out = ctypes.c_void_p(123)
    rc = lib.coli_tensor_upload_host(fmt, gs, ctypes.c_int64(4), ctypes.c_int64(8), buf, sc, ctypes.byref(out))
    assert rc == code
    assert out.value is None


def test_upload_refuses_bad_sizes(lib):
    out = ctypes.c_void_p()
    buf = (ctypes.c_uint8 * 64)()
    sc = (ctypes.c_float * 64)()
    assert lib.coli_tensor_upload(2, 0, ctypes.c_int64(0), ctypes.c_int64(8), buf, sc, None, ctypes.byref(out)) == -1
    assert lib.coli_tensor_upload(2, 0, ctypes.c_int64(4), ctypes.c_int64(8), None, sc, None, ctypes.byref(out)) == -1
    assert lib.coli_tensor_upload(2, 0, ctypes.c_int64(4), ctypes.c_int64(8), buf, None, None, ctypes.byref(out)) == -1
    assert lib.coli_tensor_upload(2, 0, ctypes.c_int64(4), ctypes.c_int64(8), buf, sc, None, None) == -1
    assert lib.coli_tensor_upload_host(2, 0, ctypes.c_int64(0), ctypes.c_int64(8), buf, sc, ctypes.byref(out)) == -1
    assert lib.coli_tensor_upload_host(2, 0, ctypes.c_int64(4), ctypes.c_int64(8), None, sc, ctypes.byref(out)) == -1
    assert lib.coli_tensor_upload_host(2, 0, ctypes.c_int64(4), ctypes.c_int64(8), buf, None, ctypes.byref(out)) == -1


def test_compute_calls_refuse_null(lib):
    assert lib.coli_matmul(None, None, None, 1, None) == -1
    assert lib.coli_moe_route(None, 1, 8, 256, None, None, None) == -1
    assert lib.coli_moe_block(None, 1, None, 1, None, None, 8, None, None) == -1
    out = ctypes.c_void_p(1)
    assert lib.coli_expert_table_create(None, 1, ctypes.byref(out)) == -1
    assert out.value is None          # cleared before the arguments are refused
    assert lib.coli_moe_block_t(None, 1, None, None, None, 8, None, None) == -1
    lib.coli_expert_table_free(None)  # a NULL table is a no-op
    i64 = ctypes.c_int64
    assert lib.coli_matmul_rows(None, i64(0), i64(0), i64(1), 1, None, None, 1, None) == -1
    assert lib.coli_matmul_rows_t(None, i64(0), i64(0), i64(1), 1, None, None, 1, None) == -1
    assert lib.coli_moe_topk(None, None, 1, 8, 2, ctypes.c_float(0.0), 0, ctypes.c_float(1.0), None, None,
                             None) == -1


def test_fail_after_is_host_side(lib):
    # a refused call (bad arguments) is checked before the injection gate
    lib.coli_set_fail_after(ctypes.c_int64(0))
    try:
        assert lib.coli_matmul(None, None, None, 1, None) == -1
    finally:
        lib.coli_set_fail_after(ctypes.c_int64(-1))
