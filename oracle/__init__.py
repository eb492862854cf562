"""CPU oracle for the NVFP4 linear-layer hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  It shares no code with the CUDA
library (``nvfp4_block_scaled_03_gb300``) and never consumes its outputs.

The arithmetic lives in ``nvfp4_oracle.c`` (plain single-threaded C, IEEE
binary32 without FMA contraction, FP64 for the GEMM); this module compiles it
with the host C compiler and marshals numpy arrays through ctypes.  The MLP
composition is in :mod:`oracle.mlp`.

Source of the method: the "NVFP4 pretraining recipe" page (re-post of NVIDIA's
NVFP4 pretraining blog), sections "NVFP4 format and advantages" and "NVFP4
pretraining recipe" (five bullets, Figure 1 text).  Every function here and
in :mod:`oracle.mlp` is pinned by ``-m "not gpu"`` tests to something other
than itself (brute force, closed forms, exhaustive searches, another
project's Philox4x32-10 run in its interpreter, invariants); none is left
"parity unpinned".
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_HDR = os.path.join(_HERE, "nvfp4_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnvfp4_oracle.so")

ROW_1X16, COL_1X16, BLOCK_16X16 = 0, 1, 2
MXFP4, MXFP8 = 0, 1
MX_ROW, MX_COL = 0, 1
RHT, SR, EMIT_T, AMAX_GIVEN = 1, 2, 4, 8
IN_BF16, IN_FP32 = 0, 1

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (host C compiler, no CUDA)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cc = os.environ.get("CC", "gcc")
        subprocess.check_call([cc, *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _QOut(C.Structure):
    _fields_ = [
        ("codes", C.c_void_p), ("scales", C.c_void_p), ("scales_sw", C.c_void_p),
        ("codes_t", C.c_void_p), ("scales_t", C.c_void_p), ("scales_t_sw", C.c_void_p),
        ("amax", C.c_float), ("s_enc", C.c_float), ("s_dec", C.c_float),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            i64, u64, u32, f32, vp = C.c_int64, C.c_uint64, C.c_uint32, C.c_float, C.c_void_p
            sig = {
                "orc_e2m1_value": ([C.c_uint8], f32), "orc_e2m1_rne": ([f32], C.c_uint8),
                "orc_e2m1_sr": ([f32, u32], C.c_uint8), "orc_e4m3_value": ([C.c_uint8], f32),
                "orc_e4m3_rne_sat": ([f32], C.c_uint8),
                "orc_bf16_from_double": ([C.c_double], C.c_uint16),
                "orc_bf16_value": ([C.c_uint16], f32),
                "orc_bf16_round_array": ([vp, i64, vp], None),
                "orc_philox4x32_10": ([vp, vp, vp], None),
                "orc_sr_word": ([u64, u64, u64], u32),
                "orc_rht_signs": ([u64, vp], None), "orc_rht16": ([vp, vp], None),
                "orc_out_shape": ([C.c_int, i64, i64, vp, vp], None),
                "orc_swizzled_bytes": ([i64, i64], i64),
                "orc_swizzle_offset": ([i64, i64, i64], i64),
                "orc_quantize": ([vp, C.c_int, i64, i64, i64, C.c_int, u32, u64, u64, f32,
                                  C.POINTER(_QOut)], C.c_int),
                "orc_quantize_window": ([vp, C.c_int, i64, i64, i64, C.c_int, u32, u64, u64, f32,
                                         u64, C.POINTER(_QOut)], C.c_int),
                "orc_amax": ([vp, C.c_int, i64, i64, i64, C.c_int, u32, u64], f32),
                "orc_dequant": ([vp, vp, f32, i64, i64, vp], None),
                "orc_gemm_fp64": ([vp, vp, f32, vp, vp, f32, i64, i64, i64, vp], None),
                "orc_gemm_fp64_sampled": ([vp, vp, f32, vp, vp, f32, i64, vp, vp, i64, vp],
                                          None),
                "orc_e8m0_value": ([C.c_uint8], f32),
                "orc_e8m0_scale": ([f32, C.c_int], C.c_uint8),
                "orc_mx_quantize": ([vp, C.c_int, i64, i64, i64, C.c_int, C.c_int, vp, vp],
                                    C.c_int),
                "orc_mx_dequant": ([vp, vp, C.c_int, i64, i64, vp], None),
                "orc_swiglu_fwd": ([vp, vp, i64, vp], None),
                "orc_swiglu_bwd": ([vp, vp, vp, i64, vp, vp], None),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


# ---- scalar formats ---------------------------------------------------------
def e2m1_value(code: int) -> float:
    return float(lib().orc_e2m1_value(code))


def e2m1_rne(y: float) -> int:
    return int(lib().orc_e2m1_rne(y))


def e2m1_sr(y: float, rbits: int) -> int:
    return int(lib().orc_e2m1_sr(y, rbits))


def e4m3_value(code: int) -> float:
    return float(lib().orc_e4m3_value(code))


def e4m3_rne_sat(t: float) -> int:
    return int(lib().orc_e4m3_rne_sat(t))


def bf16_from_double(x: float) -> int:
    return int(lib().orc_bf16_from_double(x))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round_f64(x: np.ndarray) -> np.ndarray:
    """Round FP64 values to bf16 (RNE, no double rounding); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, np.uint16)
    lib().orc_bf16_round_array(_p(x), x.size, _p(out))
    return out


def philox(ctr, key) -> list[int]:
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    o = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(o))
    return [int(v) for v in o]


def sr_word(seed: int, offset: int, idx: int) -> int:
    return int(lib().orc_sr_word(seed, offset, idx))


def rht_signs(seed: int) -> np.ndarray:
    s = np.zeros(16, dtype=np.float32)
    lib().orc_rht_signs(seed, _p(s))
    return s


def rht16(v, signs) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32).copy()
    s = np.ascontiguousarray(signs, dtype=np.float32)
    assert v.shape == (16,) and s.shape == (16,)
    lib().orc_rht16(_p(v), _p(s))
    return v


# ---- quantiser ----------------------------------------------------------------
def out_shape(mode: int, rows: int, cols: int) -> tuple[int, int]:
    return (cols, rows) if mode == COL_1X16 else (rows, cols)


def swizzled_bytes(orows: int, ocols: int) -> int:
    return int(lib().orc_swizzled_bytes(orows, ocols))


def swizzle_offset(r: int, c: int, ocols: int) -> int:
    return int(lib().orc_swizzle_offset(r, c, ocols))


def quantize(x: np.ndarray, mode: int, flags: int = 0, seed: int = 0, offset: int = 0,
             amax_given: float | None = None, sr_index_base: int = 0) -> dict:
    """Quantise a 2-D bf16 (uint16 bit patterns) or float32 array.

    ``sr_index_base`` evaluates a window of output rows of a larger operand:
    each element's stochastic-rounding index is its index in the window plus
    the base (the window's first output row times the output columns).

    Returns a dict with ``codes`` [orows, ocols/2] uint8, ``scales`` [orows,
    ocols/16] uint8 (row-major E4M3), ``scales_sw`` (MMA layout, padded),
    ``amax``, ``s_enc``, ``s_dec``, ``rows``/``cols`` (logical output shape) and,
    for 16x16 with EMIT_T, ``codes_t``/``scales_t``/``scales_t_sw``.
    """
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        dt = IN_BF16
    elif x.dtype == np.float32:
        dt = IN_FP32
    else:
        raise TypeError(f"oracle quantize takes bf16 bits (uint16) or float32, got {x.dtype}")
    rows, cols = x.shape
    orows, ocols = out_shape(mode, rows, cols)
    if (mode == COL_1X16 and rows % 16) or (mode != COL_1X16 and cols % 16):
        raise ValueError("blocked dimension must be a multiple of 16")
    res = {
        "codes": np.zeros((orows, ocols // 2), np.uint8),
        "scales": np.zeros((orows, ocols // 16), np.uint8),
        "scales_sw": np.zeros(max(1, swizzled_bytes(orows, ocols)), np.uint8),
    }
    q = _QOut()
    q.codes, q.scales, q.scales_sw = (res["codes"].ctypes.data, res["scales"].ctypes.data,
                                      res["scales_sw"].ctypes.data)
    if flags & EMIT_T:
        res["codes_t"] = np.zeros((ocols, orows // 2), np.uint8)
        res["scales_t"] = np.zeros((ocols, orows // 16), np.uint8)
        res["scales_t_sw"] = np.zeros(max(1, swizzled_bytes(ocols, orows)), np.uint8)
        q.codes_t, q.scales_t, q.scales_t_sw = (res["codes_t"].ctypes.data,
                                                res["scales_t"].ctypes.data,
                                                res["scales_t_sw"].ctypes.data)
    if amax_given is not None:
        flags |= AMAX_GIVEN
    rc = lib().orc_quantize_window(_p(x), dt, rows, cols, cols, mode, flags, seed, offset,
                                   float(amax_given or 0.0), int(sr_index_base), C.byref(q))
    if rc != 0:
        raise ValueError(f"oracle quantize rejected its arguments (rc={rc})")
    res["scales_sw"] = res["scales_sw"][:swizzled_bytes(orows, ocols)]
    if flags & EMIT_T:
        res["scales_t_sw"] = res["scales_t_sw"][:swizzled_bytes(ocols, orows)]
    res.update(amax=np.float32(q.amax), s_enc=np.float32(q.s_enc), s_dec=np.float32(q.s_dec),
               rows=orows, cols=ocols, mode=mode, flags=flags)
    return res


def amax(x: np.ndarray, mode: int, flags: int = 0, seed: int = 0) -> np.float32:
    x = np.ascontiguousarray(x)
    dt = IN_BF16 if x.dtype == np.uint16 else IN_FP32
    rows, cols = x.shape
    return np.float32(lib().orc_amax(_p(x), dt, rows, cols, cols, mode, flags, seed))


def transposed_view(q: dict) -> dict:
    """The 16x16 operand read through its transpose (EMIT_T outputs)."""
    return {"codes": q["codes_t"], "scales": q["scales_t"], "scales_sw": q["scales_t_sw"],
            "s_dec": q["s_dec"], "amax": q["amax"], "rows": q["cols"], "cols": q["rows"]}


def dequant(q: dict) -> np.ndarray:
    out = np.zeros((q["rows"], q["cols"]), np.float64)
    lib().orc_dequant(_p(q["codes"]), _p(q["scales"]), float(q["s_dec"]), q["rows"], q["cols"],
                      _p(out))
    return out


def gemm_fp64(qa: dict, qb: dict) -> np.ndarray:
    """ref[m, n] = sum_k deqA[m, k] * deqB[n, k] in FP64 (both K-major)."""
    assert qa["cols"] == qb["cols"], "contraction dims differ"
    M, N, K = qa["rows"], qb["rows"], qa["cols"]
    out = np.zeros((M, N), np.float64)
    lib().orc_gemm_fp64(_p(qa["codes"]), _p(qa["scales"]), float(qa["s_dec"]),
                        _p(qb["codes"]), _p(qb["scales"]), float(qb["s_dec"]), M, N, K, _p(out))
    return out


def gemm_fp64_sampled(qa: dict, qb: dict, m_idx, n_idx) -> np.ndarray:
    assert qa["cols"] == qb["cols"], "contraction dims differ"
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int64)
    out = np.zeros(len(m_idx), np.float64)
    lib().orc_gemm_fp64_sampled(_p(qa["codes"]), _p(qa["scales"]), float(qa["s_dec"]),
                                _p(qb["codes"]), _p(qb["scales"]), float(qb["s_dec"]),
                                qa["cols"], _p(m_idx), _p(n_idx), len(m_idx), _p(out))
    return out


# ---- MX comparison formats (OCP Microscaling: 32-element blocks, E8M0) --------
def e8m0_value(b: int) -> float:
    return float(lib().orc_e8m0_value(b))


def e8m0_scale(amax: float, fmt: int) -> int:
    return int(lib().orc_e8m0_scale(amax, fmt))


def mx_quantize(x: np.ndarray, mode: int, fmt: int) -> dict:
    """MXFP4 / MXFP8 quantisation of a 2-D bf16 (uint16 bits) or float32
    array: 32-element blocks along the output's rows (``MX_ROW``: along the
    input's columns; ``MX_COL``: along its rows, output transposed).  Returns
    ``codes`` ([orows, ocols/2] packed E2M1 or [orows, ocols] E4M3),
    ``scales`` ([orows, ocols/32] E8M0), ``rows``/``cols`` (output shape)."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        dt = IN_BF16
    elif x.dtype == np.float32:
        dt = IN_FP32
    else:
        raise TypeError(f"oracle mx_quantize takes bf16 bits (uint16) or float32, got {x.dtype}")
    rows, cols = x.shape
    orows, ocols = (cols, rows) if mode == MX_COL else (rows, cols)
    if ocols % 32:
        raise ValueError("blocked dimension must be a multiple of 32")
    codes = np.zeros((orows, ocols // 2 if fmt == MXFP4 else ocols), np.uint8)
    scales = np.zeros((orows, ocols // 32), np.uint8)
    rc = lib().orc_mx_quantize(_p(x), dt, rows, cols, cols, mode, fmt, _p(codes), _p(scales))
    if rc != 0:
        raise ValueError(f"oracle mx_quantize rejected its arguments (rc={rc})")
    return {"codes": codes, "scales": scales, "rows": orows, "cols": ocols, "fmt": fmt,
            "mode": mode}


def mx_dequant(q: dict) -> np.ndarray:
    out = np.zeros((q["rows"], q["cols"]), np.float64)
    lib().orc_mx_dequant(_p(q["codes"]), _p(q["scales"]), q["fmt"], q["rows"], q["cols"],
                         _p(out))
    return out


def swiglu_fwd(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g, np.uint16)
    u = np.ascontiguousarray(u, np.uint16)
    h = np.zeros_like(g)
    lib().orc_swiglu_fwd(_p(g), _p(u), g.size, _p(h))
    return h


def swiglu_bwd(dh: np.ndarray, g: np.ndarray, u: np.ndarray):
    dh = np.ascontiguousarray(dh, np.uint16)
    g = np.ascontiguousarray(g, np.uint16)
    u = np.ascontiguousarray(u, np.uint16)
    dg = np.zeros_like(g)
    du = np.zeros_like(g)
    lib().orc_swiglu_bwd(_p(dh), _p(g), _p(u), g.size, _p(dg), _p(du))
    return dg, du
