"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every function
include/fp8gb.h declares. No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8gb.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libpath():
    import __graft_entry__
    try:
        return __graft_entry__._build_module().build()
    except RuntimeError as e:
        pytest.skip(f"no CUDA toolkit to build with: {e}")


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("fp8_quantize", "fp8_scaled_mm", "fp8_requantize_weights", "fp8_linear_fwd", "fp8_linear_bwd",
                 "fp8_history_commit", "fp8_get_last_error_detail", "fp8_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_validation_without_gpu(libpath):
    lib = ctypes.CDLL(libpath)
    lib.fp8_status_string.restype = ctypes.c_char_p
    assert lib.fp8_status_string(0) == b"FP8_OK"
    assert lib.fp8_status_string(5) == b"FP8_ERR_TIMEOUT"
    # argument validation happens before any CUDA call: a negative size is rejected here
    lib.fp8_scaled_mm.restype = ctypes.c_int
    st = lib.fp8_scaled_mm(None, 0, None, 0, ctypes.c_int64(-1), ctypes.c_int64(1), ctypes.c_int64(1),
                           ctypes.c_int64(16), ctypes.c_int64(16), 0, None, None, None, ctypes.c_int64(8), None)
    assert st == 1
    buf = ctypes.create_string_buffer(256)
    lib.fp8_get_last_error_detail(buf, ctypes.c_size_t(256))
    assert b"negative" in buf.value
    # misaligned pointers are rejected with FP8_ERR_ALIGNMENT before any launch
    st = lib.fp8_scaled_mm(ctypes.c_void_p(0x1001), 0, ctypes.c_void_p(0x2000), 0, ctypes.c_int64(16),
                           ctypes.c_int64(16), ctypes.c_int64(16), ctypes.c_int64(16), ctypes.c_int64(16), 0,
                           ctypes.c_void_p(0x3000), ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000),
                           ctypes.c_int64(16), None)
    assert st == 3


def test_binding_names_match_the_header(libpath):
    import fp8_mixed_precision_saturating_gb300 as fp8gb
    for n in declared_functions():
        assert hasattr(fp8gb, n), n
