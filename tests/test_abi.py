"""The C ABI without a GPU: libnvfp4.so loads, exports every function that
include/nvfp4.h declares, and its host-only calls (status strings, size
queries, argument checks that fail before any CUDA call) behave."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_scaled_03_gb300 import build
    return C.CDLL(build.build())


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(nvfp4_\w+)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("nvfp4_quantize", "nvfp4_gemm", "nvfp4_mlp_fwd", "nvfp4_mlp_bwd"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_status_strings(lib):
    lib.nvfp4_status_string.restype = C.c_char_p
    for s in range(8):
        assert lib.nvfp4_status_string(s)
    assert lib.nvfp4_status_string(6) == b"CUDA error"


def test_quantize_sizes_match_the_layout_rule(lib):
    sz = C.c_size_t
    c, s, st, w = sz(), sz(), sz(), sz()
    # ROW_1X16 [200, 80]: codes 200*40, scales pad128(200)*pad4(5) = 256*8
    assert lib.nvfp4_quantize_sizes(C.c_int64(200), C.c_int64(80), 0, 0, C.byref(c), C.byref(s),
                                    C.byref(st), C.byref(w)) == 0
    assert (c.value, s.value, st.value) == (8000, 2048, 0) and w.value > 0
    # COL_1X16 of [208, 80] -> operand [80, 208]: scales pad128(80)*pad4(13) = 128*16
    assert lib.nvfp4_quantize_sizes(C.c_int64(208), C.c_int64(80), 1, 0, C.byref(c), C.byref(s),
                                    C.byref(st), C.byref(w)) == 0
    assert (c.value, s.value) == (80 * 104, 2048)
    # BLOCK_16X16 + EMIT_T [512, 256]: transposed scales pad128(256)*pad4(32)
    assert lib.nvfp4_quantize_sizes(C.c_int64(512), C.c_int64(256), 2, 4, C.byref(c), C.byref(s),
                                    C.byref(st), C.byref(w)) == 0
    assert (c.value, s.value, st.value) == (512 * 128, 512 * 16, 256 * 32)
    # amax given: no workspace
    assert lib.nvfp4_quantize_sizes(C.c_int64(128), C.c_int64(64), 0, 8, None, None, None,
                                    C.byref(w)) == 0 and w.value == 0
    assert lib.nvfp4_quantize_sizes(C.c_int64(128), C.c_int64(40), 0, 0, None, None, None,
                                    None) == 2


def test_argument_errors_return_before_any_launch(lib):
    lib.nvfp4_quantize.argtypes = [C.c_void_p, C.c_int32, C.c_int64, C.c_int64, C.c_int64,
                                   C.c_int32, C.c_uint32, C.c_uint64, C.c_uint64, C.c_void_p,
                                   C.c_void_p, C.c_size_t, C.c_void_p]
    # null input / output
    assert lib.nvfp4_quantize(None, 0, 16, 16, 16, 0, 0, 0, 0, None, None, 0, None) == 1
    lib.nvfp4_gemm.argtypes = [C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                               C.c_int32, C.c_void_p, C.c_int64, C.c_int64, C.c_int64,
                               C.c_void_p, C.c_size_t, C.c_void_p]
    assert lib.nvfp4_gemm(None, 0, None, 0, None, 0, None, 128, 128, 128, None, 0, None) == 1


def test_mlp_sizes(lib):
    sz = C.c_size_t
    s, w = sz(), sz()
    assert lib.nvfp4_mlp_sizes(C.c_int64(256), C.c_int64(256), C.c_int64(512), C.byref(s),
                               C.byref(w)) == 0
    # saved holds G and U (bf16 [M, F] each) plus the quantised operands
    assert s.value > 2 * 256 * 512 * 2 and w.value > 4 * 256 * 512 * 2
    assert lib.nvfp4_mlp_sizes(C.c_int64(100), C.c_int64(256), C.c_int64(512), C.byref(s),
                               C.byref(w)) == 2
