"""ctypes binding of libnvfp4.so with the C ABI's names (include/nvfp4.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  If the library is not
built, importing this module raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass, field

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libnvfp4.so")

# status codes
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGN, ERR_ARCH, ERR_WORKSPACE, ERR_CUDA, \
    ERR_DEVICE_TIMEOUT = range(8)
# enums and flags
IN_BF16, IN_FP32 = 0, 1
ROW_1X16, COL_1X16, BLOCK_16X16 = 0, 1, 2
RHT, SR, EMIT_T, AMAX_GIVEN = 1, 2, 4, 8
D_BF16, D_F32_ACCUM, D_BF16_ADD_C = 0, 1, 2
MXFP4, MXFP8 = 0, 1
MX_ROW, MX_COL = 0, 1
(TILE_AUTO, TILE_128X128, TILE_128X256, TILE_PAIR_256X256, TILE_128X256_K128,
 TILE_PAIR_256X384) = 0, 1, 2, 3, 5, 6


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


class Tensor(C.Structure):
    """Mirror of ``nvfp4_tensor``."""
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("codes_t", C.c_void_p),
                ("scales_t", C.c_void_p), ("amax", C.c_void_p), ("s_dec", C.c_void_p),
                ("rows", C.c_int64), ("cols", C.c_int64), ("mode", C.c_int32),
                ("flags", C.c_uint32)]


class MlpParams(C.Structure):
    """Mirror of ``nvfp4_mlp_params``."""
    _fields_ = [("M", C.c_int64), ("D", C.c_int64), ("F", C.c_int64), ("Wg", C.c_void_p),
                ("Wu", C.c_void_p), ("Wd", C.c_void_p), ("seed", C.c_uint64),
                ("step", C.c_uint64), ("flags", C.c_uint32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = C.CDLL(LIB_PATH)
    i32, i64, u32, u64, vp, sz = C.c_int32, C.c_int64, C.c_uint32, C.c_uint64, C.c_void_p, C.c_size_t
    P = C.POINTER
    sigs = {
        "nvfp4_status_string": ([C.c_int], C.c_char_p),
        "nvfp4_version": ([], C.c_int),
        "nvfp4_device_check": ([C.c_int], C.c_int),
        "nvfp4_check_device_errors": ([vp], C.c_int),
        "nvfp4_debug_inject": ([u32, u64], C.c_int),
        "nvfp4_quantize_sizes": ([i64, i64, i32, u32, P(sz), P(sz), P(sz), P(sz)], C.c_int),
        "nvfp4_quantize": ([vp, i32, i64, i64, i64, i32, u32, u64, u64, P(Tensor), vp, sz, vp],
                           C.c_int),
        "nvfp4_quantize_noalloc": ([vp, i32, i64, i64, i64, i32, u32, u64, u64, P(Tensor), vp],
                                   C.c_int),
        "nvfp4_amax": ([vp, i32, i64, i64, i64, u64, vp, vp, vp, sz, vp], C.c_int),
        "nvfp4_quantize_rowcol": ([vp, i32, i64, i64, i64, u32, u32, u64, u64, u64, P(Tensor),
                                   P(Tensor), vp], C.c_int),
        "nvfp4_gemm": ([P(Tensor), i32, P(Tensor), i32, vp, i32, vp, i64, i64, i64, vp, sz, vp],
                       C.c_int),
        "nvfp4_gemm_ex": ([P(Tensor), i32, P(Tensor), i32, vp, i32, vp, i64, i64, i64, i32, vp],
                          C.c_int),
        "nvfp4_mx_sizes": ([i64, i64, i32, i32, P(sz), P(sz), P(sz)], C.c_int),
        "nvfp4_mx_quantize": ([vp, i32, i64, i64, i64, i32, i32, vp, vp, vp, vp], C.c_int),
        "nvfp4_mx_gemm": ([vp, vp, vp, vp, i32, vp, i64, i64, i64, vp], C.c_int),
        "nvfp4_swiglu_workspace_bytes": ([], sz),
        "nvfp4_swiglu_fwd": ([vp, vp, vp, i64, i64, u32, u64, vp, vp, vp, sz, vp], C.c_int),
        "nvfp4_swiglu_bwd": ([vp, vp, vp, vp, vp, i64, i64, u32, u64, vp, vp, vp, vp, vp, sz, vp],
                             C.c_int),
        "nvfp4_mlp_sizes": ([i64, i64, i64, P(sz), P(sz)], C.c_int),
        "nvfp4_mlp_fwd": ([P(MlpParams), vp, vp, vp, sz, vp, sz, vp], C.c_int),
        "nvfp4_mlp_bwd": ([P(MlpParams), vp, vp, vp, vp, vp, vp, vp, sz, vp], C.c_int),
        "nvfp4_mlp_tensor": ([i64, i64, i64, vp, vp, i32, P(vp), P(i64), P(i64)], C.c_int),
        "nvfp4_mlp_operand": ([i64, i64, i64, vp, vp, i32, P(Tensor)], C.c_int),
        "nvfp4_sgd_step": ([vp, vp, i64, C.c_float, u32, vp, vp, sz, vp], C.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


lib = _load()


def status_string(s: int) -> str:
    return lib.nvfp4_status_string(s).decode()


def _check(status: int, where: str):
    if status != OK:
        raise NVFP4Error(status, where)


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


@dataclass
class QTensor:
    """A quantised operand: the device buffers plus the ABI descriptor."""
    codes: torch.Tensor
    scales: torch.Tensor
    amax: torch.Tensor
    s_dec: torch.Tensor
    codes_t: torch.Tensor | None = None
    scales_t: torch.Tensor | None = None
    desc: Tensor = field(default_factory=Tensor)

    @property
    def rows(self):
        return self.desc.rows

    @property
    def cols(self):
        return self.desc.cols


def quantize_sizes(rows, cols, mode, flags=0):
    c, s, st, w = C.c_size_t(), C.c_size_t(), C.c_size_t(), C.c_size_t()
    _check(lib.nvfp4_quantize_sizes(rows, cols, mode, flags, C.byref(c), C.byref(s), C.byref(st),
                                    C.byref(w)), "nvfp4_quantize_sizes")
    return c.value, s.value, st.value, w.value


def alloc_qtensor(rows, cols, mode, flags=0, device="cuda") -> QTensor:
    """Allocate the output buffers of quantising an input [rows, cols]."""
    cb, sb, stb, _ = quantize_sizes(rows, cols, mode, flags)
    u8 = dict(dtype=torch.uint8, device=device)
    q = QTensor(codes=torch.empty(cb, **u8), scales=torch.empty(sb, **u8),
                amax=torch.zeros(1, dtype=torch.float32, device=device),
                s_dec=torch.zeros(1, dtype=torch.float32, device=device))
    if flags & EMIT_T:
        q.codes_t = torch.empty(cb, **u8)
        q.scales_t = torch.empty(stb, **u8)
    d = q.desc
    d.codes, d.scales = q.codes.data_ptr(), q.scales.data_ptr()
    d.codes_t, d.scales_t = _ptr(q.codes_t), _ptr(q.scales_t)
    d.amax, d.s_dec = q.amax.data_ptr(), q.s_dec.data_ptr()
    return q


_ws_cache: dict = {}


def _workspace(nbytes, device):
    key = (str(device), torch.cuda.current_stream().cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def nvfp4_quantize(x: torch.Tensor, mode: int, flags: int = 0, seed: int = 0, offset: int = 0,
                   out: QTensor | None = None, workspace: torch.Tensor | None = None,
                   amax: float | torch.Tensor | None = None, stream=None) -> QTensor:
    """Quantise a 2-D bf16/fp32 CUDA tensor (see nvfp4_quantize in nvfp4.h)."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    if x.dtype == torch.bfloat16:
        dt = IN_BF16
    elif x.dtype == torch.float32:
        dt = IN_FP32
    else:
        raise TypeError(f"x must be bf16 or fp32, got {x.dtype}")
    rows, cols = x.shape
    if amax is not None:
        flags |= AMAX_GIVEN
    if out is None:
        out = alloc_qtensor(rows, cols, mode, flags, device=x.device)
    if amax is not None:
        out.amax.copy_(torch.as_tensor(amax, dtype=torch.float32).reshape(1))
    _, _, _, wsb = quantize_sizes(rows, cols, mode, flags)
    if workspace is None and wsb:
        workspace = _workspace(wsb, x.device)
    _check(lib.nvfp4_quantize(x.data_ptr(), dt, rows, cols, x.stride(0), mode, flags, seed, offset,
                              C.byref(out.desc), _ptr(workspace),
                              0 if workspace is None else workspace.numel(), _stream(stream)),
           "nvfp4_quantize")
    return out


def nvfp4_amax(x: torch.Tensor, amax_plain: torch.Tensor | None = None,
               amax_rht: torch.Tensor | None = None, seed: int = 0,
               workspace: torch.Tensor | None = None, stream=None):
    """max |x| and/or max |RHT(x)| along columns from one read (see nvfp4_amax
    in nvfp4.h); the outputs are 1-element float32 CUDA tensors, e.g. the
    `amax` of the QTensors then quantised with NVFP4_AMAX_GIVEN."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    dt = {torch.bfloat16: IN_BF16, torch.float32: IN_FP32}.get(x.dtype)
    if dt is None:
        raise TypeError(f"x must be bf16 or fp32, got {x.dtype}")
    for t in (amax_plain, amax_rht):
        if t is not None and (t.dtype != torch.float32 or t.numel() != 1 or not t.is_cuda):
            raise ValueError("amax outputs must be 1-element float32 CUDA tensors")
    rows, cols = x.shape
    if workspace is None:  # the partial-maxima workspace does not depend on the shape
        workspace = _workspace(quantize_sizes(128, 128, ROW_1X16)[3], x.device)
    _check(lib.nvfp4_amax(x.data_ptr(), dt, rows, cols, x.stride(0), seed, _ptr(amax_plain),
                          _ptr(amax_rht), _ptr(workspace), workspace.numel(), _stream(stream)),
           "nvfp4_amax")


def nvfp4_quantize_rowcol(x: torch.Tensor, row_flags: int = 0, col_flags: int = 0, seed: int = 0,
                          row_offset: int = 0, col_offset: int = 0,
                          row_out: QTensor | None = None, col_out: QTensor | None = None,
                          amax_row: torch.Tensor | None = None, amax_col: torch.Tensor | None = None,
                          stream=None):
    """Row-wise and column-wise quantisation of a bf16 x from one read (see
    nvfp4_quantize_rowcol in nvfp4.h).  The two amaxes are given: either
    already in row_out.amax / col_out.amax, or as 1-element float32 CUDA
    tensors amax_row / amax_col (copied there).  Returns (row_out, col_out)."""
    if x.dim() != 2 or x.stride(1) != 1 or x.dtype != torch.bfloat16:
        raise ValueError("x must be a 2-D bf16 tensor with unit column stride")
    rows, cols = x.shape
    row_flags |= AMAX_GIVEN
    col_flags |= AMAX_GIVEN
    if row_out is None:
        row_out = alloc_qtensor(rows, cols, ROW_1X16, device=x.device)
    if col_out is None:
        col_out = alloc_qtensor(rows, cols, COL_1X16, device=x.device)
    if amax_row is not None:
        row_out.amax.copy_(amax_row.reshape(1))
    if amax_col is not None:
        col_out.amax.copy_(amax_col.reshape(1))
    _check(lib.nvfp4_quantize_rowcol(x.data_ptr(), IN_BF16, rows, cols, x.stride(0), row_flags,
                                     col_flags, seed, row_offset, col_offset, C.byref(row_out.desc),
                                     C.byref(col_out.desc), _stream(stream)),
           "nvfp4_quantize_rowcol")
    return row_out, col_out


def nvfp4_quantize_noalloc(x: torch.Tensor, mode: int, flags: int = 0, seed: int = 0,
                           offset: int = 0, out: QTensor | None = None, stream=None) -> QTensor:
    """nvfp4_quantize without a workspace: scratch lives inside the library
    (see nvfp4_quantize_noalloc in nvfp4.h for who needs this and its limits)."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    dt = {torch.bfloat16: IN_BF16, torch.float32: IN_FP32}.get(x.dtype)
    if dt is None:
        raise TypeError(f"x must be bf16 or fp32, got {x.dtype}")
    rows, cols = x.shape
    if out is None:
        out = alloc_qtensor(rows, cols, mode, flags, device=x.device)
    _check(lib.nvfp4_quantize_noalloc(x.data_ptr(), dt, rows, cols, x.stride(0), mode, flags, seed,
                                      offset, C.byref(out.desc), _stream(stream)),
           "nvfp4_quantize_noalloc")
    return out


def mx_sizes(rows, cols, mode, fmt):
    """(codes, scales, scales in the MMA layout) byte sizes."""
    c, s, w = C.c_size_t(), C.c_size_t(), C.c_size_t()
    _check(lib.nvfp4_mx_sizes(rows, cols, mode, fmt, C.byref(c), C.byref(s), C.byref(w)),
           "nvfp4_mx_sizes")
    return c.value, s.value, w.value


def nvfp4_mx_quantize(x: torch.Tensor, mode: int, fmt: int, codes: torch.Tensor | None = None,
                      scales: torch.Tensor | None = None, scales_sw: torch.Tensor | None = None,
                      stream=None):
    """MXFP4 / MXFP8 quantisation of a 2-D bf16/fp32 CUDA tensor (see
    nvfp4_mx_quantize in nvfp4.h); returns (codes, scales) as uint8 tensors
    shaped [out_rows, out_cols/2 or out_cols] and [out_rows, out_cols/32].
    ``scales_sw`` (optional, uint8, mx_sizes()[2] bytes) also receives the
    scales in the MMA layout nvfp4_mx_gemm reads."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    dt = {torch.bfloat16: IN_BF16, torch.float32: IN_FP32}.get(x.dtype)
    if dt is None:
        raise TypeError(f"x must be bf16 or fp32, got {x.dtype}")
    rows, cols = x.shape
    orows, ocols = (cols, rows) if mode == MX_COL else (rows, cols)
    cb, sb, swb = mx_sizes(rows, cols, mode, fmt)
    if codes is None:
        codes = torch.empty(orows, cb // orows, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(orows, sb // orows, dtype=torch.uint8, device=x.device)
    if codes.numel() < cb or scales.numel() < sb or (scales_sw is not None and
                                                     scales_sw.numel() < swb):
        raise ValueError("output buffers are smaller than nvfp4_mx_sizes gives")
    _check(lib.nvfp4_mx_quantize(x.data_ptr(), dt, rows, cols, x.stride(0), mode, fmt,
                                 codes.data_ptr(), scales.data_ptr(), _ptr(scales_sw),
                                 _stream(stream)),
           "nvfp4_mx_quantize")
    return codes, scales


def nvfp4_mx_gemm(a_codes: torch.Tensor, a_scales_sw: torch.Tensor, b_codes: torch.Tensor,
                  b_scales_sw: torch.Tensor, fmt: int, M: int, N: int, K: int,
                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """D bf16 [M, N] = A . B^T for MX operands (see nvfp4_mx_gemm in nvfp4.h)."""
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a_codes.device)
    _check(lib.nvfp4_mx_gemm(a_codes.data_ptr(), a_scales_sw.data_ptr(), b_codes.data_ptr(),
                             b_scales_sw.data_ptr(), fmt, out.data_ptr(), M, N, K,
                             _stream(stream)), "nvfp4_mx_gemm")
    return out


def nvfp4_gemm(A: QTensor, B: QTensor, a_view: int = 0, b_view: int = 0,
               out: torch.Tensor | None = None, d_mode: int = D_BF16,
               C_add: torch.Tensor | None = None, tile: int = TILE_AUTO, stream=None) -> torch.Tensor:
    """D = alpha * A . B^T (see nvfp4_gemm in nvfp4.h); returns D."""
    M = A.desc.cols if a_view else A.desc.rows
    K = A.desc.rows if a_view else A.desc.cols
    N = B.desc.cols if b_view else B.desc.rows
    if out is None:
        dtype = torch.float32 if d_mode == D_F32_ACCUM else torch.bfloat16
        out = (torch.zeros if d_mode == D_F32_ACCUM else torch.empty)(
            (M, N), dtype=dtype, device=A.codes.device)
    if tile:
        st = lib.nvfp4_gemm_ex(C.byref(A.desc), a_view, C.byref(B.desc), b_view, out.data_ptr(),
                               d_mode, _ptr(C_add), M, N, K, tile, _stream(stream))
    else:
        st = lib.nvfp4_gemm(C.byref(A.desc), a_view, C.byref(B.desc), b_view, out.data_ptr(),
                            d_mode, _ptr(C_add), M, N, K, None, 0, _stream(stream))
    _check(st, "nvfp4_gemm")
    return out


def _bf16_2d(*ts):
    for t in ts:
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("SwiGLU tensors must be contiguous 2-D bf16 CUDA tensors")
        if t.shape != ts[0].shape:
            raise ValueError("SwiGLU tensors must have one shape")


def _amax_outs(n, device):
    return [torch.zeros(1, dtype=torch.float32, device=device) for _ in range(n)]


def nvfp4_swiglu_fwd(G, U, rht=True, seed=0, H=None, workspace=None, stream=None):
    """H = silu(G) * U with the amaxes of H's row-wise and column-wise (RHT)
    quantisations (see nvfp4_swiglu_fwd in nvfp4.h); returns
    (H, amax_row, amax_col), the amaxes as 1-element float32 CUDA tensors."""
    H = torch.empty_like(G) if H is None else H
    _bf16_2d(G, U, H)
    rows, cols = G.shape
    if workspace is None:
        workspace = _workspace(lib.nvfp4_swiglu_workspace_bytes(), G.device)
    a_row, a_col = _amax_outs(2, G.device)
    _check(lib.nvfp4_swiglu_fwd(G.data_ptr(), U.data_ptr(), H.data_ptr(), rows, cols,
                                RHT if rht else 0, seed, a_row.data_ptr(), a_col.data_ptr(),
                                workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "nvfp4_swiglu_fwd")
    return H, a_row, a_col


def nvfp4_swiglu_bwd(dH, G, U, rht=True, seed=0, workspace=None, stream=None):
    """dG, dU of the SwiGLU with the amaxes of their row-wise and column-wise
    quantisations; returns (dG, dU, amax_dg_row, amax_dg_col, amax_du_row,
    amax_du_col)."""
    dG, dU = torch.empty_like(G), torch.empty_like(G)
    _bf16_2d(dH, G, U, dG, dU)
    rows, cols = G.shape
    if workspace is None:
        workspace = _workspace(lib.nvfp4_swiglu_workspace_bytes(), G.device)
    a = _amax_outs(4, G.device)
    _check(lib.nvfp4_swiglu_bwd(dH.data_ptr(), G.data_ptr(), U.data_ptr(), dG.data_ptr(),
                                dU.data_ptr(), rows, cols, RHT if rht else 0, seed,
                                *(t.data_ptr() for t in a), workspace.data_ptr(),
                                workspace.numel(), _stream(stream)), "nvfp4_swiglu_bwd")
    return (dG, dU, *a)


def mlp_sizes(M, D, F):
    s, w = C.c_size_t(), C.c_size_t()
    _check(lib.nvfp4_mlp_sizes(M, D, F, C.byref(s), C.byref(w)), "nvfp4_mlp_sizes")
    return s.value, w.value


def mlp_params(M, D, F, Wg, Wu, Wd, seed=0, step=0, rht=True,
               weight_amax_given=False) -> MlpParams:
    return MlpParams(M, D, F, Wg.data_ptr(), Wu.data_ptr(), Wd.data_ptr(), seed, step,
                     (RHT if rht else 0) | (AMAX_GIVEN if weight_amax_given else 0))


def nvfp4_mlp_fwd(p: MlpParams, X, Y, saved, workspace, stream=None):
    _check(lib.nvfp4_mlp_fwd(C.byref(p), X.data_ptr(), Y.data_ptr(), saved.data_ptr(),
                             saved.numel(), workspace.data_ptr(), workspace.numel(),
                             _stream(stream)), "nvfp4_mlp_fwd")
    return Y


def nvfp4_mlp_bwd(p: MlpParams, dY, saved, dX, dWg, dWu, dWd, workspace, stream=None):
    _check(lib.nvfp4_mlp_bwd(C.byref(p), dY.data_ptr(), saved.data_ptr(), dX.data_ptr(),
                             dWg.data_ptr(), dWu.data_ptr(), dWd.data_ptr(), workspace.data_ptr(),
                             workspace.numel(), _stream(stream)), "nvfp4_mlp_bwd")
    return dX


# intermediates of an MLP step inside the saved / workspace buffers
MLP_G, MLP_U, MLP_H, MLP_DH, MLP_DG, MLP_DU, MLP_DX_GATE = range(7)
(MLP_Q_WG, MLP_Q_WU, MLP_Q_WD, MLP_Q_X, MLP_Q_XC, MLP_Q_H, MLP_Q_HC, MLP_Q_DY, MLP_Q_DYC,
 MLP_Q_DG, MLP_Q_DGC, MLP_Q_DU, MLP_Q_DUC) = range(16, 29)


def _slice_of(ptr, nbytes, bufs):
    """The bytes [ptr, ptr + nbytes) as a uint8 view of whichever buffer holds them."""
    for b in bufs:
        if b is not None and b.data_ptr() <= ptr and ptr + nbytes <= b.data_ptr() + b.numel():
            off = ptr - b.data_ptr()
            return b[off:off + nbytes]
    raise ValueError("address outside the given buffers")


def mlp_tensor(M, D, F, saved, workspace, which) -> torch.Tensor:
    """The bf16 intermediate `which` (MLP_G ... MLP_DX_GATE) of the last MLP
    call, as a [rows, cols] view into saved / workspace (nvfp4_mlp_tensor)."""
    p, r, c = C.c_void_p(), C.c_int64(), C.c_int64()
    _check(lib.nvfp4_mlp_tensor(M, D, F, _ptr(saved), _ptr(workspace), which, C.byref(p),
                                C.byref(r), C.byref(c)), "nvfp4_mlp_tensor")
    raw = _slice_of(p.value, r.value * c.value * 2, (saved, workspace))
    return raw.view(torch.bfloat16).view(r.value, c.value)


def mlp_operand(M, D, F, saved, workspace, which) -> QTensor:
    """The quantised operand `which` (MLP_Q_*) of the last MLP call, as a
    QTensor whose tensors are views into saved / workspace (nvfp4_mlp_operand)."""
    d = Tensor()
    _check(lib.nvfp4_mlp_operand(M, D, F, _ptr(saved), _ptr(workspace), which, C.byref(d)),
           "nvfp4_mlp_operand")
    bufs = (saved, workspace)
    rows, cols = d.rows, d.cols
    # the operand's sizes: K-major [rows, cols] (the quantiser's ROW_1X16 form of the same shape)
    cb, sb, _, _ = quantize_sizes(rows, cols, ROW_1X16)
    q = QTensor(codes=_slice_of(d.codes, cb, bufs), scales=_slice_of(d.scales, sb, bufs),
                amax=_slice_of(d.amax, 4, bufs).view(torch.float32),
                s_dec=_slice_of(d.s_dec, 4, bufs).view(torch.float32), desc=d)
    if d.codes_t:
        cbt, sbt, _, _ = quantize_sizes(cols, rows, ROW_1X16)
        q.codes_t = _slice_of(d.codes_t, cbt, bufs)
        q.scales_t = _slice_of(d.scales_t, sbt, bufs)
    return q


ZERO_GRAD = 16


def nvfp4_sgd_step(W: torch.Tensor, G: torch.Tensor, lr: float, zero_grad: bool = False,
                   amax: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                   stream=None):
    """W -= lr * G on FP32 master weight and gradient (G zeroed with
    zero_grad), writing max |W| of the updated weight into the 1-element
    float32 CUDA tensor `amax` when given (see nvfp4_sgd_step in nvfp4.h)."""
    for t in (W, G):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("W and G must be contiguous float32 CUDA tensors")
    if W.numel() != G.numel():
        raise ValueError("W and G must have the same number of elements")
    if amax is not None and (amax.dtype != torch.float32 or amax.numel() != 1 or not amax.is_cuda):
        raise ValueError("amax must be a 1-element float32 CUDA tensor")
    if amax is not None and workspace is None:
        workspace = _workspace(quantize_sizes(128, 128, ROW_1X16)[3], W.device)
    _check(lib.nvfp4_sgd_step(W.data_ptr(), G.data_ptr(), W.numel(), float(lr),
                              ZERO_GRAD if zero_grad else 0, _ptr(amax), _ptr(workspace),
                              workspace.numel() if workspace is not None else 0,
                              _stream(stream)), "nvfp4_sgd_step")
    return W


STALL_QUANTIZE, STALL_GEMM = 1, 2


def debug_inject(stall_mask: int = 0, wait_limit_ns: int = 0):
    """Failure injection for tests of the bounded waits (nvfp4_debug_inject)."""
    _check(lib.nvfp4_debug_inject(stall_mask, wait_limit_ns), "nvfp4_debug_inject")


def check_device_errors(stream=None):
    _check(lib.nvfp4_check_device_errors(_stream(stream)), "nvfp4_check_device_errors")
