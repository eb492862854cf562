"""GPU parity of the block-scaled GEMM against the oracle's FP64 product.

The GEMM's operands are the oracle's quantised operands uploaded to the
device, so these tests isolate the GEMM; the end-to-end test feeds the GPU
quantiser's own outputs.  Tolerance: max|D-ref|/max|ref| <= 1e-2 and
|D-ref| <= 4 ulp_bf16(ref) + 1e-3 rms(ref) per element.
"""
import numpy as np
import pytest

import gpu_helpers as H
from nvfp4_block_scaled_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_03_gb300 import binding
    return binding


def _layer(orc, M, K, N, seed=0):
    """Oracle operands of the three GEMMs of one linear layer."""
    X = syn.activations((M, K), seed=1)
    W = syn.weights((N, K), seed=2)
    dY = syn.gradients((M, N), seed=3)
    return {
        "X": orc.quantize(X, orc.ROW_1X16),
        "W": orc.quantize(W, orc.BLOCK_16X16, orc.EMIT_T),
        "dY": orc.quantize(dY, orc.ROW_1X16, orc.SR, seed=seed, offset=0),
        "dYc": orc.quantize(dY, orc.COL_1X16, orc.RHT | orc.SR, seed=seed, offset=1),
        "Xc": orc.quantize(X, orc.COL_1X16, orc.RHT, seed=seed),
        "raw": (X, W, dY),
    }


def _gemms(orc, L):
    Wt = orc.transposed_view(L["W"])
    return {"FPROP": (L["X"], L["W"]), "DGRAD": (L["dY"], Wt), "WGRAD": (L["dYc"], L["Xc"])}


@pytest.mark.parametrize("tile", [1, 2, 3, 5, 6])
@pytest.mark.parametrize("M,K,N", [(128, 256, 512), (208, 192, 144), (320, 1024, 272),
                                   (128, 64, 16), (320, 576, 1040)])
def test_gemm_small(nv, orc, M, K, N, tile):
    L = _layer(orc, M, K, N)
    for name, (a, b) in _gemms(orc, L).items():
        if a["cols"] % 64 or b["rows"] % 8:
            continue  # WGRAD of a ragged token count: K = M must be a multiple of 64
        A, B = H.upload(nv, a), H.upload(nv, b)
        D = nv.nvfp4_gemm(A, B, tile=tile)
        nv.check_device_errors()
        H.assert_gemm_close(H.host_f64(D), orc.gemm_fp64(a, b), f"{name} {M}x{N}x{a['cols']}")


def test_gemm_rejects_retired_tile(nv, orc):
    """Tile configuration 4 (a retired variant) is refused before any launch."""
    L = _layer(orc, 128, 256, 512)
    A, B = H.upload(nv, L["X"]), H.upload(nv, L["W"])
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_gemm(A, B, tile=4)
    assert e.value.status == nv.ERR_INVALID_ARG


def test_gemm_transposed_view_on_device(nv, orc):
    """DGRAD reads W through codes_t/scales_t of the GPU quantiser (b_view=1)."""
    M, K, N = 256, 384, 512
    X, W, dY = syn.linear_layer(M, K, N)
    qW = nv.nvfp4_quantize(H.dev_bf16(W), nv.BLOCK_16X16, nv.EMIT_T)
    qdY = nv.nvfp4_quantize(H.dev_bf16(dY), nv.ROW_1X16, nv.SR, seed=4, offset=2)
    D = nv.nvfp4_gemm(qdY, qW, b_view=1)
    oW = orc.quantize(W, orc.BLOCK_16X16, orc.EMIT_T)
    odY = orc.quantize(dY, orc.ROW_1X16, orc.SR, seed=4, offset=2)
    H.assert_gemm_close(H.host_f64(D), orc.gemm_fp64(odY, orc.transposed_view(oW)), "DGRAD")


def test_gemm_output_modes(nv, orc):
    """F32_ACCUM adds float(bf16(result)) exactly; ADD_C adds a bf16 C."""
    import torch
    M, K, N = 256, 512, 384
    L = _layer(orc, M, K, N)
    a, b = L["X"], L["W"]
    A, B = H.upload(nv, a), H.upload(nv, b)
    ref = orc.gemm_fp64(a, b)
    D = nv.nvfp4_gemm(A, B)
    rng = np.random.Generator(np.random.PCG64(3))
    W0 = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).cuda()
    acc = W0.clone()
    nv.nvfp4_gemm(A, B, out=acc, d_mode=nv.D_F32_ACCUM)
    exp = W0 + D.float()      # the fold: one fp32 add of the bf16 result per element
    assert torch.equal(acc, exp)
    Cb = H.dev_bf16(syn.gradients((M, N), seed=9) )
    E = nv.nvfp4_gemm(A, B, d_mode=nv.D_BF16_ADD_C, C_add=Cb)
    H.assert_gemm_close(H.host_f64(E), ref + H.host_f64(Cb), "ADD_C")
    nv.check_device_errors()


@pytest.mark.parametrize("tile", [3, 6])
@pytest.mark.parametrize("M,K,N", [(512, 256, 784), (768, 512, 512), (512, 320, 1168)])
def test_gemm_output_modes_pair_kernel(nv, orc, M, K, N, tile):
    """The fold into FP32 and the bf16 add on the CTA-pair kernels (the large-
    shape path: 256- and 384-wide tiles), with a ragged last tile: F32_ACCUM
    equals W0 + float(D) exactly, D the bf16 output of the same kernel; ADD_C
    is within the GEMM tolerance of the FP64 product plus C on the 256-wide
    tile and refused on the 384-wide one."""
    import torch
    L = _layer(orc, M, K, N)
    a, b = L["X"], L["W"]
    A, B = H.upload(nv, a), H.upload(nv, b)
    ref = orc.gemm_fp64(a, b)
    D = nv.nvfp4_gemm(A, B, tile=tile)
    H.assert_gemm_close(H.host_f64(D), ref, f"bf16 tile {tile}")
    rng = np.random.Generator(np.random.PCG64(5))
    W0 = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).cuda()
    acc = W0.clone()
    nv.nvfp4_gemm(A, B, out=acc, d_mode=nv.D_F32_ACCUM, tile=tile)
    assert torch.equal(acc, W0 + D.float())
    Cb = H.dev_bf16(syn.gradients((M, N), seed=9))
    if tile == nv.TILE_PAIR_256X384:
        with pytest.raises(nv.NVFP4Error) as e:
            nv.nvfp4_gemm(A, B, d_mode=nv.D_BF16_ADD_C, C_add=Cb, tile=tile)
        assert e.value.status == nv.ERR_INVALID_ARG
    else:
        E = nv.nvfp4_gemm(A, B, d_mode=nv.D_BF16_ADD_C, C_add=Cb, tile=tile)
        H.assert_gemm_close(H.host_f64(E), ref + H.host_f64(Cb), "ADD_C pair")
    nv.check_device_errors()


def test_gemm_wide_pair_tile_equals_pair_tile_llama8b(nv):
    """The 384-wide pair tile (two MMAs per K step, N = 256 and N = 128, two
    tensor-memory scale slots) against the 256-wide one at the bench's full
    shapes (M=8192, K=4096, N=14336: FPROP, DGRAD through W's transposed
    view, WGRAD of the column operands) on GPU-quantised operands: every
    output element identical (the same MMAs accumulate each element in the
    same K order), in the bf16 and the FP32-fold modes."""
    import torch
    M, K, N = 8192, 4096, 14336
    X, W, dY = syn.linear_layer(M, K, N)
    qX = nv.nvfp4_quantize(H.dev_bf16(X), nv.ROW_1X16)
    qW = nv.nvfp4_quantize(H.dev_bf16(W), nv.BLOCK_16X16, nv.EMIT_T)
    qdY = nv.nvfp4_quantize(H.dev_bf16(dY), nv.ROW_1X16, nv.SR, seed=0, offset=0)
    qdYc = nv.nvfp4_quantize(H.dev_bf16(dY), nv.COL_1X16, nv.RHT | nv.SR, seed=0, offset=1)
    qXc = nv.nvfp4_quantize(H.dev_bf16(X), nv.COL_1X16, nv.RHT, seed=0)
    for name, a, b, bv in (("FPROP", qX, qW, 0), ("DGRAD", qdY, qW, 1), ("WGRAD", qdYc, qXc, 0)):
        d3 = nv.nvfp4_gemm(a, b, b_view=bv, tile=nv.TILE_PAIR_256X256)
        d6 = nv.nvfp4_gemm(a, b, b_view=bv, tile=nv.TILE_PAIR_256X384)
        nv.check_device_errors()
        assert torch.equal(d3, d6), f"{name}: 384-wide tile differs from the 256-wide tile"
        del d3, d6
    acc3 = torch.full((M, N), 0.25, dtype=torch.float32, device="cuda")
    acc6 = acc3.clone()
    nv.nvfp4_gemm(qX, qW, out=acc3, d_mode=nv.D_F32_ACCUM, tile=nv.TILE_PAIR_256X256)
    nv.nvfp4_gemm(qX, qW, out=acc6, d_mode=nv.D_F32_ACCUM, tile=nv.TILE_PAIR_256X384)
    nv.check_device_errors()
    assert torch.equal(acc3, acc6)


def test_gemm_end_to_end_gpu_quantiser(nv, orc):
    """GPU quantiser -> GPU GEMM for FPROP/DGRAD/WGRAD vs the oracle chain."""
    M, K, N = 256, 512, 768
    X, W, dY = syn.linear_layer(M, K, N)
    qX = nv.nvfp4_quantize(H.dev_bf16(X), nv.ROW_1X16)
    qW = nv.nvfp4_quantize(H.dev_bf16(W), nv.BLOCK_16X16, nv.EMIT_T)
    qdY = nv.nvfp4_quantize(H.dev_bf16(dY), nv.ROW_1X16, nv.SR, seed=0, offset=0)
    qdYc = nv.nvfp4_quantize(H.dev_bf16(dY), nv.COL_1X16, nv.RHT | nv.SR, seed=0, offset=1)
    qXc = nv.nvfp4_quantize(H.dev_bf16(X), nv.COL_1X16, nv.RHT, seed=0)
    L = _layer(orc, M, K, N)
    got = {"FPROP": nv.nvfp4_gemm(qX, qW), "DGRAD": nv.nvfp4_gemm(qdY, qW, b_view=1),
           "WGRAD": nv.nvfp4_gemm(qdYc, qXc)}
    for name, (a, b) in _gemms(orc, L).items():
        H.assert_gemm_close(H.host_f64(got[name]), orc.gemm_fp64(a, b), name)


def _sample_positions(M, N, n=4096, seed=11):
    rng = np.random.Generator(np.random.PCG64(seed))
    m = rng.integers(0, M, n)
    k = rng.integers(0, N, n)
    cm, cn = np.meshgrid(np.arange(128), np.arange(128), indexing="ij")   # first tile
    lm, ln = np.meshgrid(np.arange(M - 128, M), np.arange(N - 128, N), indexing="ij")  # last
    return (np.concatenate([m, cm.ravel(), lm.ravel()]),
            np.concatenate([k, cn.ravel(), ln.ravel()]))


def test_gemm_llama8b_full_sampled(nv, orc):
    """The bench workload (M=8192, K=4096, N=14336): FPROP, DGRAD, WGRAD at
    full size in the bench's launch configuration, checked on 4096 random
    outputs plus the first and the last 128x128 tile (FP64 oracle dot
    products); rms(ref) for the tolerance is taken over the sampled outputs."""
    M, K, N = 8192, 4096, 14336
    L = _layer(orc, M, K, N)
    for name, (a, b) in _gemms(orc, L).items():
        A, B = H.upload(nv, a), H.upload(nv, b)
        D = nv.nvfp4_gemm(A, B)
        nv.check_device_errors()
        m, n = _sample_positions(a["rows"], b["rows"])
        ref = orc.gemm_fp64_sampled(a, b, m, n)
        got = H.host_f64(D[m, n])
        H.assert_gemm_close(got, ref, name)
        del A, B, D


def test_gemm_405b_up_projection_full_sampled(nv, orc):
    """The Llama-3.1-405B MLP up projection at full size (X [8192, 16384],
    W [53248, 16384], dY [8192, 53248]): FPROP (K = 16384), DGRAD through W's
    transposed view (K = 53248) and WGRAD (K = 8192), each on oracle-quantised
    operands, checked on 4096 random outputs plus the first and last 128x128
    tiles."""
    import gc
    M, K, N = 8192, 16384, 53248
    X = syn.activations((M, K), seed=1)
    W = syn.weights((N, K), seed=2)
    qW = orc.quantize(W, orc.BLOCK_16X16, orc.EMIT_T)
    del W
    gc.collect()
    qX = orc.quantize(X, orc.ROW_1X16)
    _check_sampled(nv, orc, "FPROP 405B", qX, qW)
    del qX
    gc.collect()
    dY = syn.gradients((M, N), seed=3)
    qdY = orc.quantize(dY, orc.ROW_1X16, orc.SR, seed=0, offset=0)
    _check_sampled(nv, orc, "DGRAD 405B", qdY, orc.transposed_view(qW))
    del qdY, qW
    gc.collect()
    qdYc = orc.quantize(dY, orc.COL_1X16, orc.RHT | orc.SR, seed=0, offset=1)
    del dY
    gc.collect()
    qXc = orc.quantize(X, orc.COL_1X16, orc.RHT, seed=0)
    _check_sampled(nv, orc, "WGRAD 405B", qdYc, qXc)


def _check_sampled(nv, orc, name, a, b):
    A, B = H.upload(nv, a), H.upload(nv, b)
    D = nv.nvfp4_gemm(A, B)
    nv.check_device_errors()
    m, n = _sample_positions(a["rows"], b["rows"])
    ref = orc.gemm_fp64_sampled(a, b, m, n)
    H.assert_gemm_close(H.host_f64(D[m, n]), ref, name)
    del A, B, D


@pytest.mark.parametrize("M,K,N,tile", [(128, 256, 512, 0), (512, 256, 784, 3)])
def test_gemm_zero_operand(nv, orc, M, K, N, tile):
    """An all-zero operand quantises to s_dec = 1, zero scales and zero codes
    (the zero-amax edge of the per-tensor scale); its product with any
    operand is exactly zero, on the single-SM and the CTA-pair kernels."""
    import torch
    X, W, _ = syn.linear_layer(M, K, N)
    Z = np.zeros((M, K), np.uint16)
    qZ = nv.nvfp4_quantize(H.dev_bf16(Z), nv.ROW_1X16)
    qW = nv.nvfp4_quantize(H.dev_bf16(W), nv.BLOCK_16X16, nv.EMIT_T)
    oZ = orc.quantize(Z, orc.ROW_1X16)
    H.assert_quant_equal(qZ, oZ, "zeros")
    assert float(qZ.s_dec.cpu()[0]) == 1.0 and not qZ.scales.cpu().numpy().any()
    for D in (nv.nvfp4_gemm(qZ, qW, tile=tile),
              nv.nvfp4_gemm(qW, qZ, tile=tile if tile == 0 else 2),
              nv.nvfp4_gemm(qZ, qZ, tile=tile)):
        nv.check_device_errors()
        assert not torch.any(D.float() != 0), "a product with a zero operand is not zero"
    ref = orc.gemm_fp64(oZ, orc.quantize(W, orc.BLOCK_16X16, orc.EMIT_T))
    assert not ref.any()


def test_gemm_405b_down_projection_gpu_quantised_sampled(nv, orc):
    """The Llama-3.1-405B MLP down projection at full size: H [8192, 53248]
    (activations), W_down [16384, 53248], dY [8192, 16384]; FPROP Y = H W^T
    (K = 53248), DGRAD dH = dY W through W's transposed view (K = 16384),
    WGRAD dW = dY^T H (K = 8192, both RHT, dY^T with SR).  The GPU quantises
    every operand whole; the oracle takes each tensor's amax itself and
    quantises sampled 128-row slabs of every operand, which must equal the
    GPU's bytes, and the GEMMs are checked on the first and last slab pairs'
    outputs plus 4096 random outputs within the slabs."""
    import gc
    import torch
    M, N, K = 8192, 16384, 53248
    rng = np.random.Generator(np.random.PCG64(21))

    def pick(n):
        k = n // 128
        return sorted({0, k - 1} | set(rng.integers(1, k - 1, 2).tolist()))

    Hh = syn.activations((M, K), seed=1)
    W = syn.weights((N, K), seed=2)
    dY = syn.gradients((M, N), seed=3)
    sM, sN, sK = pick(M), pick(N), pick(K)

    def host_q(q):
        return (q.codes.cpu().numpy().reshape(q.rows, q.cols // 2), q.scales.cpu().numpy(),
                float(q.amax.cpu()[0]), float(q.s_dec.cpu()[0]))

    def oracle_op(x, mode, flags, q, slabs, name, offset=0):
        amax = orc.amax(x, mode, flags & orc.RHT, seed=0)
        codes, scales, a, sd = host_q(q)
        assert np.float32(a) == amax, name
        os_ = H.oracle_slabs(orc, x, mode, flags, amax, slabs, seed=0, offset=offset)
        H.assert_slabs_equal(codes, scales, a, sd, os_, slabs, name)
        return H.compact_operand(os_)

    def check(D, a, b, sa, sb, name):
        nv.check_device_errors()
        lm, ln, gm, gn = H.sampled_positions(sa, sb)
        ref = orc.gemm_fp64_sampled(a, b, lm, ln)
        got = H.host_f64(D[torch.from_numpy(gm).cuda(), torch.from_numpy(gn).cuda()])
        H.assert_gemm_close(got, ref, name)

    qW = nv.nvfp4_quantize(H.dev_bf16(W), nv.BLOCK_16X16, nv.EMIT_T)
    wamax = orc.amax(W, orc.BLOCK_16X16)
    assert np.float32(float(qW.amax.cpu()[0])) == wamax
    codes, scales, a, sd = host_q(qW)
    oW = H.oracle_slabs(orc, W, orc.BLOCK_16X16, orc.EMIT_T, wamax, sN)
    H.assert_slabs_equal(codes, scales, a, sd, oW, sN, "W")
    codes_t = qW.codes_t.cpu().numpy().reshape(K, N // 2)
    oWt = H.oracle_slabs_transposed(orc, W, wamax, sK)
    H.assert_slabs_equal(codes_t, qW.scales_t.cpu().numpy(), a, sd, oWt, sK, "W^T")
    oW, oWt = H.compact_operand(oW), H.compact_operand(oWt)
    del W
    gc.collect()
    qH = nv.nvfp4_quantize(H.dev_bf16(Hh), nv.ROW_1X16)
    check(nv.nvfp4_gemm(qH, qW), oracle_op(Hh, orc.ROW_1X16, 0, qH, sM, "H"), oW, sM, sN,
          "FPROP 405B down")
    del qH
    qdY = nv.nvfp4_quantize(H.dev_bf16(dY), nv.ROW_1X16, nv.SR, seed=0, offset=0)
    check(nv.nvfp4_gemm(qdY, qW, b_view=1),
          oracle_op(dY, orc.ROW_1X16, orc.SR, qdY, sM, "dY"), oWt, sM, sK, "DGRAD 405B down")
    del qdY, qW
    torch.cuda.empty_cache()
    qdYc = nv.nvfp4_quantize(H.dev_bf16(dY), nv.COL_1X16, nv.RHT | nv.SR, seed=0, offset=1)
    qHc = nv.nvfp4_quantize(H.dev_bf16(Hh), nv.COL_1X16, nv.RHT, seed=0)
    a_op = oracle_op(dY, orc.COL_1X16, orc.RHT | orc.SR, qdYc, sN, "dY^T", offset=1)
    b_op = oracle_op(Hh, orc.COL_1X16, orc.RHT, qHc, sK, "H^T")
    check(nv.nvfp4_gemm(qdYc, qHc), a_op, b_op, sN, sK, "WGRAD 405B down")
