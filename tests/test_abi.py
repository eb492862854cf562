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


def test_mx_sizes_follow_the_header_rule(lib):
    """nvfp4_mx_sizes against the layout rule the header states: codes of
    out_rows x out_cols at 4 or 8 bits, one scale byte per 32 outputs, and the
    MMA layout padded to 128 rows x 4 scale columns per 512-byte atom."""
    sz = C.c_size_t

    def sizes(rows, cols, mode, fmt):
        c, s, w = sz(), sz(), sz()
        st = lib.nvfp4_mx_sizes(C.c_int64(rows), C.c_int64(cols), C.c_int32(mode),
                                C.c_int32(fmt), C.byref(c), C.byref(s), C.byref(w))
        return st, c.value, s.value, w.value

    def atoms(orows, ocols):
        return -(-orows // 128) * -(-(ocols // 32) // 4) * 512

    for rows, cols in ((64, 96), (333, 1056), (1, 32)):
        for fmt, bits in ((0, 4), (1, 8)):
            assert sizes(rows, cols, 0, fmt) == (0, rows * cols * bits // 8, rows * cols // 32,
                                                 atoms(rows, cols))
    for rows, cols in ((64, 136), (320, 1000)):
        for fmt, bits in ((0, 4), (1, 8)):
            assert sizes(rows, cols, 1, fmt) == (0, rows * cols * bits // 8, rows * cols // 32,
                                                 atoms(cols, rows))
    assert sizes(64, 48, 0, 0)[0] == 2      # 48 columns: not whole 32-element blocks
    assert sizes(40, 64, 1, 1)[0] == 2      # 40 rows along the column blocks
    assert lib.nvfp4_mx_sizes(C.c_int64(64), C.c_int64(64), 0, 0, None, None, None) == 0


def test_swiglu_argument_errors_return_before_any_launch(lib):
    """The SwiGLU entry points check their arguments on the host: unknown
    flags and NULL pointers (invalid argument), rows not a multiple of 16
    (shape), a short workspace, and misaligned tensors -- all before touching
    a device, so the fake addresses below are never dereferenced."""
    vp, i64, u32, u64, sz = C.c_void_p, C.c_int64, C.c_uint32, C.c_uint64, C.c_size_t
    lib.nvfp4_swiglu_workspace_bytes.restype = sz
    lib.nvfp4_swiglu_fwd.argtypes = [vp, vp, vp, i64, i64, u32, u64, vp, vp, vp, sz, vp]
    lib.nvfp4_swiglu_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, u32, u64, vp, vp, vp, vp,
                                     vp, sz, vp]
    wsb = lib.nvfp4_swiglu_workspace_bytes()
    assert wsb >= 16 and wsb % 16 == 0
    t, a, ws = 0x10000, 0x20000, 0x30000        # 16-byte aligned fake addresses
    fwd, bwd = lib.nvfp4_swiglu_fwd, lib.nvfp4_swiglu_bwd
    assert fwd(t, t, t, 32, 64, 0x80, 0, a, a, ws, wsb, None) == 1    # unknown flag
    assert fwd(t, t, None, 32, 64, 0, 0, a, a, ws, wsb, None) == 1    # NULL output
    assert fwd(t, t, t, 32, 64, 0, 0, a, None, ws, wsb, None) == 1    # NULL amax
    assert fwd(t, t, t, 40, 64, 1, 0, a, a, ws, wsb, None) == 2       # rows % 16
    assert fwd(t, t, t, 32, 60, 1, 0, a, a, ws, wsb, None) == 2       # cols % 8
    assert fwd(t, t, t, 32, 64, 1, 0, a, a, ws, wsb - 16, None) == 5  # workspace
    assert fwd(t + 8, t, t, 32, 64, 1, 0, a, a, ws, wsb, None) == 3   # misaligned G
    assert bwd(t, t, t, t, t, 32, 64, 2, 0, a, a, a, a, ws, wsb, None) == 1   # SR: not a flag here
    assert bwd(t, t, t, t, None, 32, 64, 0, 0, a, a, a, a, ws, wsb, None) == 1
    assert bwd(t, t, t, t, t, 24, 64, 0, 0, a, a, a, a, ws, wsb, None) == 2
    assert bwd(t, t, t, t, t, 32, 64, 0, 0, a, a, a, a, None, wsb, None) == 5
    assert bwd(t, t, t, t, t + 4, 32, 64, 0, 0, a, a, a, a, ws, wsb, None) == 3
    assert bwd(t, t, t, t, t, 32, 64, 0, 0, a, a, a + 2, a, ws, wsb, None) == 3  # amax not 4-aligned


class _Desc(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("codes_t", C.c_void_p),
                ("scales_t", C.c_void_p), ("amax", C.c_void_p), ("s_dec", C.c_void_p),
                ("rows", C.c_int64), ("cols", C.c_int64), ("mode", C.c_int32),
                ("flags", C.c_uint32)]


def test_mlp_intermediates_lie_inside_their_buffers(lib):
    """nvfp4_mlp_tensor / nvfp4_mlp_operand are host-side address arithmetic:
    with stand-in buffer addresses, every intermediate lies inside the buffer
    the header names for it, 256-byte aligned, with the stated shape, and no
    two intermediates overlap."""
    M, D, F = 384, 256, 640
    sb, wb = C.c_size_t(), C.c_size_t()
    assert lib.nvfp4_mlp_sizes(C.c_int64(M), C.c_int64(D), C.c_int64(F), C.byref(sb),
                               C.byref(wb)) == 0
    saved, ws = 1 << 40, 1 << 44            # stand-ins; nothing is dereferenced
    lib.nvfp4_mlp_tensor.argtypes = [C.c_int64] * 3 + [C.c_void_p, C.c_void_p, C.c_int32,
                                                       C.POINTER(C.c_void_p),
                                                       C.POINTER(C.c_int64), C.POINTER(C.c_int64)]
    lib.nvfp4_mlp_operand.argtypes = [C.c_int64] * 3 + [C.c_void_p, C.c_void_p, C.c_int32,
                                                        C.POINTER(_Desc)]
    spans = []

    def inside(ptr, n, in_saved):
        base, size = (saved, sb.value) if in_saved else (ws, wb.value)
        assert base <= ptr and ptr + n <= base + size
        assert ptr % 256 == 0
        spans.append((ptr, ptr + n))

    shapes = {0: (M, F), 1: (M, F), 2: (M, F), 3: (M, F), 4: (M, F), 5: (M, F), 6: (M, D)}
    for which, shape in shapes.items():
        p, r, c = C.c_void_p(), C.c_int64(), C.c_int64()
        assert lib.nvfp4_mlp_tensor(M, D, F, saved, ws, which, C.byref(p), C.byref(r),
                                    C.byref(c)) == 0
        assert (r.value, c.value) == shape
        inside(p.value, r.value * c.value * 2, which in (0, 1))
    ops = {16: (F, D, 1), 17: (F, D, 1), 18: (D, F, 1), 19: (M, D, 0), 20: (D, M, 1),
           21: (M, F, 0), 22: (F, M, 1), 23: (M, D, 0), 24: (D, M, 0), 25: (M, F, 0),
           26: (F, M, 0), 27: (M, F, 0), 28: (F, M, 0)}
    for which, (rows, cols, in_saved) in ops.items():
        d = _Desc()
        assert lib.nvfp4_mlp_operand(M, D, F, saved, ws, which, C.byref(d)) == 0
        assert (d.rows, d.cols) == (rows, cols)
        pr, pc = (rows + 127) // 128 * 128, (cols // 16 + 3) // 4 * 4
        inside(d.codes, rows * cols // 2, in_saved)
        inside(d.scales, pr * pc, in_saved)
        inside(d.amax, 4, in_saved)
        inside(d.s_dec, 4, in_saved)
        if which in (16, 17, 18):
            inside(d.codes_t, rows * cols // 2, in_saved)
            inside(d.scales_t, (cols + 127) // 128 * 128 * ((rows // 16 + 3) // 4 * 4), in_saved)
        else:
            assert not d.codes_t and not d.scales_t
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:])), "intermediates overlap"
    d = _Desc()
    p, r, c = C.c_void_p(), C.c_int64(), C.c_int64()
    assert lib.nvfp4_mlp_operand(M, D, F, saved, ws, 99, C.byref(d)) == 1      # unknown
    assert lib.nvfp4_mlp_operand(M, D, F, None, ws, 16, C.byref(d)) == 1       # holder NULL
    assert lib.nvfp4_mlp_operand(M, D, F, saved, None, 16, C.byref(d)) == 0    # other NULL ok
    assert lib.nvfp4_mlp_tensor(M, D, F, saved, None, 2, C.byref(p), C.byref(r), C.byref(c)) == 1
    assert lib.nvfp4_mlp_tensor(100, D, F, saved, ws, 2, C.byref(p), C.byref(r), C.byref(c)) == 2


def test_quantize_rowcol_argument_errors_before_any_launch(lib):
    """nvfp4_quantize_rowcol rejects bad arguments on the host, before any CUDA
    call: stand-in addresses suffice (nothing is dereferenced)."""
    f = lib.nvfp4_quantize_rowcol
    f.argtypes = [C.c_void_p, C.c_int32, C.c_int64, C.c_int64, C.c_int64, C.c_uint32,
                  C.c_uint32, C.c_uint64, C.c_uint64, C.c_uint64, C.POINTER(_Desc),
                  C.POINTER(_Desc), C.c_void_p]
    base = 1 << 40

    def desc(k):
        d = _Desc()
        d.codes, d.scales, d.amax, d.s_dec = base + k * 4096, base + k * 4096 + 1024, \
            base + k * 4096 + 2048, base + k * 4096 + 2052
        return d

    x, G = base + (1 << 20), 8  # AMAX_GIVEN
    r, c = desc(1), desc(2)

    def call(x=x, dt=0, rows=64, cols=64, ld=64, rf=G, cf=G | 1, r=r, c=c):
        return f(x, dt, rows, cols, ld, rf, cf, 0, 0, 0, C.byref(r) if r else None,
                 C.byref(c) if c else None, None)

    assert call(x=None) == 1                      # NULL input
    assert call(c=None) == 1                      # NULL output descriptor
    assert call(dt=1) == 1                        # fp32 input
    assert call(rf=0) == 1                        # amax not given
    assert call(rf=G | 1) == 1                    # RHT on the row operand
    assert call(cf=G | 4) == 1                    # EMIT_T
    assert call(rows=40) == 2 and call(cols=72, ld=72) == 2 and call(ld=32) == 2
    assert call(x=x + 8) == 3 and call(ld=68) == 3
    bad = desc(3)
    bad.codes += 4
    assert call(r=bad) == 3                       # codes not 16-byte aligned


def test_debug_inject_rejects_unknown_bits_without_a_device(lib):
    """nvfp4_debug_inject refuses stall bits it does not know before touching
    the device."""
    lib.nvfp4_debug_inject.argtypes = [C.c_uint32, C.c_uint64]
    assert lib.nvfp4_debug_inject(4, 0) == 1
    assert lib.nvfp4_debug_inject(0xFFFFFFFC, 1000) == 1


def test_sgd_step_argument_errors_before_any_launch(lib):
    """nvfp4_sgd_step refuses bad arguments before touching the device:
    NULL pointers, unknown flags, a non-finite rate, overlapping W and G
    (INVALID_ARG), n <= 0 or not a multiple of 4 (SHAPE), misalignment
    (ALIGN), a missing workspace when the amax is asked for (WORKSPACE)."""
    f = lib.nvfp4_sgd_step
    f.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_float, C.c_uint32, C.c_void_p,
                  C.c_void_p, C.c_size_t, C.c_void_p]
    INVALID, SHAPE, ALIGN, WORKSPACE = 1, 2, 3, 5
    W, G, A, WS = 0x10000, 0x20000, 0x30000, 0x40000   # never dereferenced on these paths
    assert f(None, G, 64, 0.1, 0, None, None, 0, None) == INVALID
    assert f(W, None, 64, 0.1, 0, None, None, 0, None) == INVALID
    assert f(W, G, 64, 0.1, 1, None, None, 0, None) == INVALID
    assert f(W, G, 64, float("inf"), 0, None, None, 0, None) == INVALID
    assert f(W, G, 64, float("nan"), 0, None, None, 0, None) == INVALID
    assert f(W, W + 64, 64, 0.1, 0, None, None, 0, None) == INVALID    # overlapping
    assert f(W, G, 0, 0.1, 0, None, None, 0, None) == SHAPE
    assert f(W, G, 66, 0.1, 0, None, None, 0, None) == SHAPE
    assert f(W + 4, G, 64, 0.1, 0, None, None, 0, None) == ALIGN
    assert f(W, G, 64, 0.1, 0, A + 2, WS, 4096, None) == ALIGN
    assert f(W, G, 64, 0.1, 16, A, None, 0, None) == WORKSPACE
    assert f(W, G, 64, 0.1, 16, A, WS, 16, None) == WORKSPACE


@pytest.mark.parametrize("std,cc", [("c11", "gcc"), ("c++17", "g++")])
def test_header_compiles_as_plain_c_and_cpp(tmp_path, std, cc):
    """The boundary header stands alone: no CUDA or torch types, valid C11 and
    C++17, warning-free, and every entry point has C linkage when included
    from C++ (its names are not mangled)."""
    import subprocess
    ext = "c" if std == "c11" else "cpp"
    src = tmp_path / f"use.{ext}"
    init = "= {0}" if std == "c11" else "{}"
    src.write_text('#include "nvfp4.h"\n'
                   f"int probe(void) {{ nvfp4_tensor t {init}; (void)t;\n"
                   "  return (int)nvfp4_quantize_sizes(128, 256, NVFP4_ROW_1X16, 0, 0, 0, 0, 0); }\n")
    obj = tmp_path / "use.o"
    subprocess.check_call([cc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-c",
                           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(obj)])
    syms = subprocess.check_output(["nm", str(obj)], text=True)
    assert re.search(r"\bU nvfp4_quantize_sizes\b", syms), syms
