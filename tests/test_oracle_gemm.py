"""Pins of the oracle's FP64 GEMM -- CPU only.

Losslessly quantisable inputs reduce the NVFP4 GEMM to a textbook GEMM of the
inputs, which numpy's float64 matmul computes independently ("NVFP4
pretraining recipe", Figure 1 text: NVFP4 inputs, high-precision products).
"""
import numpy as np
import pytest

E4M3_POS = np.array([(m * 2.0 ** -9) if e == 0 else (8 + m) * 2.0 ** (e - 10)
                     for e in range(16) for m in range(8)][:127], np.float64)


def lossless(orc, rng, R, C, p=8):
    """float32 [R, C] that NVFP4 (1x16) represents exactly."""
    codes = rng.integers(0, 16, (R, C))
    Sb = rng.integers(16, 0x70, (R, C // 16))
    Sb[0, 0] = 0x7E
    for r in range(R):
        for b in range(C // 16):
            codes[r, b * 16 + rng.integers(0, 16)] = 7 | (rng.integers(0, 2) << 3)
    vals = np.array([orc.e2m1_value(c) for c in range(16)])[codes]
    return (vals * np.repeat(E4M3_POS[Sb], 16, axis=1) * 2.0 ** -p).astype(np.float32)


@pytest.mark.parametrize("M,N,K", [(8, 12, 16), (16, 8, 32), (32, 24, 128)])
def test_gemm_reduces_to_textbook_gemm(orc, M, N, K):
    rng = np.random.Generator(np.random.PCG64(M * 1000 + N + K))
    A = lossless(orc, rng, M, K)
    B = lossless(orc, rng, N, K, p=9)
    qa, qb = orc.quantize(A, orc.ROW_1X16), orc.quantize(B, orc.ROW_1X16)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    got = orc.gemm_fp64(qa, qb)
    if K <= 32:
        assert np.array_equal(got, ref)       # few terms of few bits: exact
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=0)


def test_gemm_through_transposed_weight_view(orc):
    """DGRAD reads W [N, K] through its transpose: dY [M, N] x W -> [M, K]."""
    from nvfp4_block_scaled_03_gb300 import synthetic as syn
    W = syn.weights((32, 48), seed=31, master_fp32=True)
    dY = syn.gradients((16, 32), seed=32)
    qW = orc.quantize(W, orc.BLOCK_16X16, orc.EMIT_T)
    qd = orc.quantize(dY, orc.ROW_1X16)
    got = orc.gemm_fp64(qd, orc.transposed_view(qW))
    ref = orc.dequant(qd) @ orc.dequant(qW)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-300)


def test_sampled_equals_full(orc):
    from nvfp4_block_scaled_03_gb300 import synthetic as syn
    A = orc.quantize(syn.activations((40, 64), seed=33), orc.ROW_1X16)
    B = orc.quantize(syn.weights((24, 64), seed=34), orc.ROW_1X16)
    full = orc.gemm_fp64(A, B)
    rng = np.random.Generator(np.random.PCG64(35))
    m = rng.integers(0, 40, 100)
    n = rng.integers(0, 24, 100)
    assert np.array_equal(orc.gemm_fp64_sampled(A, B, m, n), full[m, n])
