"""GPU parity of the MX comparison GEMMs (nvfp4_mx_gemm: MXFP4 and MXFP8
operands on the CTA-pair tensor-core kernel) against the oracle's FP64
product of the dequantised operands, within the NVFP4 GEMM's tolerance."""
import functools

import numpy as np
import pytest

from nvfp4_block_scaled_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_03_gb300 import binding
    return binding


import gpu_helpers as H  # noqa: E402


def _swizzle(orc, scales):
    """Row-major E8M0 scales [rows][K/32] -> the MMA layout (the atom layout
    of the NVFP4 scales: a scale matrix of K/32 columns is the NVFP4 one of an
    operand with K/2 columns)."""
    rows, sc = scales.shape
    out = np.zeros(orc.swizzled_bytes(rows, sc * 16), np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(sc), indexing="ij")
    off = np.vectorize(lambda a, b: orc.swizzle_offset(int(a), int(b), sc * 16))(r, c)
    out[off.ravel()] = scales.ravel()
    return out


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _ref(orc, qa, qb):
    return orc.mx_dequant(qa) @ orc.mx_dequant(qb).T


@pytest.mark.parametrize("fmt", ["MXFP8", "MXFP4"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (256, 256, 512), (200, 136, 384),
                                   (384, 520, 1024)])
def test_mx_gemm_oracle_operands(nv, orc, fmt, M, N, K):
    f = {"MXFP4": nv.MXFP4, "MXFP8": nv.MXFP8}[fmt]
    X = syn.activations((M, K), seed=1)
    W = syn.weights((N, K), seed=2)
    qa, qb = orc.mx_quantize(X, orc.MX_ROW, f), orc.mx_quantize(W, orc.MX_ROW, f)
    D = nv.nvfp4_mx_gemm(_dev(qa["codes"]), _dev(_swizzle(orc, qa["scales"])), _dev(qb["codes"]),
                         _dev(_swizzle(orc, qb["scales"])), f, M, N, K)
    nv.check_device_errors()
    H.assert_gemm_close(H.host_f64(D), _ref(orc, qa, qb), f"{fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", ["MXFP8", "MXFP4"])
def test_mx_gemm_wgrad_form(nv, orc, fmt):
    """dW = dY^T X over the tokens, both operands from the column quantiser
    (blocks of 32 tokens), quantised on the GPU; the reference quantises the
    same inputs with the oracle."""
    import torch
    f = {"MXFP4": nv.MXFP4, "MXFP8": nv.MXFP8}[fmt]
    M, K, N = 384, 256, 264
    X = syn.activations((M, K), seed=1)
    dY = syn.gradients((M, N), seed=3)
    ops = []
    for t in (dY, X):
        cols = t.shape[1]
        swb = nv.mx_sizes(M, cols, nv.MX_COL, f)[2]
        sw = torch.empty(swb, dtype=torch.uint8, device="cuda")
        codes, _ = nv.nvfp4_mx_quantize(H.dev_bf16(t), nv.MX_COL, f, scales_sw=sw)
        ops.append((codes, sw))
    D = nv.nvfp4_mx_gemm(ops[0][0], ops[0][1], ops[1][0], ops[1][1], f, N, K, M)
    nv.check_device_errors()
    qa, qb = orc.mx_quantize(dY, orc.MX_COL, f), orc.mx_quantize(X, orc.MX_COL, f)
    H.assert_gemm_close(H.host_f64(D), _ref(orc, qa, qb), f"{fmt} WGRAD")


@functools.lru_cache(maxsize=1)
def _405b_inputs():
    return syn.activations((8192, 16384), seed=1), syn.weights((53248, 16384), seed=2)


@pytest.mark.parametrize("fmt", ["MXFP8", "MXFP4"])
def test_mx_gemm_405b_up_projection_sampled(nv, orc, fmt):
    """The Llama-3.1-405B up projection FPROP at full size (X [8192, 16384],
    W [53248, 16384]) on GPU-quantised operands, checked on 4096 sampled
    outputs: MX blocks are row-local (no tensor scale), so the oracle
    quantises only the sampled rows."""
    import torch
    f = {"MXFP4": nv.MXFP4, "MXFP8": nv.MXFP8}[fmt]
    X, W = _405b_inputs()
    M, K = X.shape
    N = W.shape[0]
    dev = []
    for t in (X, W):
        swb = nv.mx_sizes(t.shape[0], K, nv.MX_ROW, f)[2]
        sw = torch.empty(swb, dtype=torch.uint8, device="cuda")
        codes, _ = nv.nvfp4_mx_quantize(H.dev_bf16(t), nv.MX_ROW, f, scales_sw=sw)
        dev.append((codes, sw))
    D = nv.nvfp4_mx_gemm(dev[0][0], dev[0][1], dev[1][0], dev[1][1], f, M, N, K)
    nv.check_device_errors()
    rng = np.random.default_rng(9)
    rows_m = np.unique(rng.integers(0, M, 256))
    rows_n = np.unique(rng.integers(0, N, 256))
    m = rng.choice(rows_m, 4096)
    n = rng.choice(rows_n, 4096)
    da = orc.mx_dequant(orc.mx_quantize(np.ascontiguousarray(X[rows_m]), orc.MX_ROW, f))
    db = orc.mx_dequant(orc.mx_quantize(np.ascontiguousarray(W[rows_n]), orc.MX_ROW, f))
    ia, ib = np.searchsorted(rows_m, m), np.searchsorted(rows_n, n)
    ref = np.einsum("ij,ij->i", da[ia], db[ib])
    got = H.host_f64(D[torch.from_numpy(m).cuda(), torch.from_numpy(n).cuda()])
    H.assert_gemm_close(got, ref, f"{fmt} 405B up projection")


def _mx_dev(nv, t, mode, f):
    import torch
    swb = nv.mx_sizes(t.shape[0], t.shape[1], mode, f)[2]
    sw = torch.empty(swb, dtype=torch.uint8, device="cuda")
    codes, _ = nv.nvfp4_mx_quantize(H.dev_bf16(t), mode, f, scales_sw=sw)
    return codes, sw


def _mx_rows(orc, x, mode, f, rows):
    """Dequantised operand rows `rows` of the MX quantisation of x: a row of
    the row form is an input row, of the column form an input column (MX
    blocks are local to it: no tensor scale)."""
    xs = np.ascontiguousarray(x[:, rows] if mode == orc.MX_COL else x[rows])
    return orc.mx_dequant(orc.mx_quantize(xs, mode, f))


@pytest.mark.parametrize("fmt", ["MXFP8", "MXFP4"])
def test_mx_gemm_405b_dgrad_wgrad_sampled(nv, orc, fmt):
    """The Llama-3.1-405B up projection's DGRAD (dX = dY W: dY [8192, 53248]
    row form, W read through its column form, K = 53248) and WGRAD (dW = dY^T X:
    both column forms, K = 8192) at full size on GPU-quantised operands,
    checked on 4096 sampled outputs against the oracle's quantisation of the
    sampled operand rows."""
    import torch
    f = {"MXFP4": nv.MXFP4, "MXFP8": nv.MXFP8}[fmt]
    X, W = _405b_inputs()
    M, K = X.shape
    N = W.shape[0]
    dY = syn.gradients((M, N), seed=3)
    rng = np.random.default_rng(13)
    for name, (a, am, b, bm, gm, gn, gk) in {
            "DGRAD": (dY, orc.MX_ROW, W, orc.MX_COL, M, K, N),
            "WGRAD": (dY, orc.MX_COL, X, orc.MX_COL, N, K, M)}.items():
        (ca, sa), (cb, sb) = _mx_dev(nv, a, am, f), _mx_dev(nv, b, bm, f)
        D = nv.nvfp4_mx_gemm(ca, sa, cb, sb, f, gm, gn, gk)
        nv.check_device_errors()
        del ca, sa, cb, sb
        rows_m = np.unique(rng.integers(0, gm, 256))
        rows_n = np.unique(rng.integers(0, gn, 256))
        m, n = rng.choice(rows_m, 4096), rng.choice(rows_n, 4096)
        da, db = _mx_rows(orc, a, am, f, rows_m), _mx_rows(orc, b, bm, f, rows_n)
        ref = np.einsum("ij,ij->i", da[np.searchsorted(rows_m, m)], db[np.searchsorted(rows_n, n)])
        got = H.host_f64(D[torch.from_numpy(m).cuda(), torch.from_numpy(n).cuda()])
        H.assert_gemm_close(got, ref, f"{fmt} 405B {name}")
        del D


def test_mx_gemm_rejects_bad_arguments(nv):
    import torch
    z = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_mx_gemm(z, z, z, z, nv.MXFP4, 128, 128, 64)  # K not a multiple of 128
    assert e.value.status == nv.ERR_SHAPE
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_mx_gemm(z, z, z, z, 5, 128, 128, 128)
    assert e.value.status == nv.ERR_INVALID_ARG
    nv.check_device_errors()
