"""GPU parity of the SwiGLU MLP forward + backward (nine NVFP4 GEMMs), stage
by stage against the oracle.

The composed MLP is compared stage by stage: every stage takes the GPU's own
upstream tensors (read from the caller's saved / workspace buffers through
nvfp4_mlp_tensor / nvfp4_mlp_operand) as its input, so the comparison of
each stage is exact where the stage is exact and within its own tolerance
where it is not, with no drift accumulated from earlier stages:

* each quantised operand the MLP writes -- W_g, W_u, W_d (16x16 + transpose,
  from the FP32 masters), X, H, dY, dG, dU row-wise and X^T, H^T, dY^T, dG^T,
  dU^T column-wise (RHT when enabled), with the recipe's rounding per operand
  and SR offsets 8 step + 0..5 -- byte for byte against the oracle's
  quantisation of the GPU's bf16 tensor (codes, MMA-layout scales, amax,
  s_dec);
* H = silu(G) U and dG, dU against the oracle's SwiGLU of the GPU's G, U,
  dH within one bf16 ulp (the bound test_gpu_swiglu derives);
* each of the nine GEMM outputs against the oracle's FP64 product of the
  (identical) quantised operands, within the GEMM tolerance; dX as the bf16
  DGRAD of dU W_u added to the GPU's bf16 dG W_g;
* the fold into the FP32 master gradients exactly: dW(c) == c + dW(0).

At Llama-3-8B size (32768 tokens) the quantised operands are compared on
sampled 128-row slabs and the GEMMs on the outputs of the first and last slab
pair plus 4096 random outputs within the slabs ("NVFP4 pretraining recipe"
page, Figure 1 text: the MLP's GEMMs in NVFP4).
"""
import gc

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


def _np(t):
    return t.cpu().numpy()


def _bits(t):
    """bf16 device tensor -> uint16 bit patterns on the host."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _ulp_bf16(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.maximum(np.where(a > 0, 2.0 ** (e - 7), 0.0), 2.0 ** -133)


def _within_one_ulp(got_bits, ref_bits, name):
    got = syn.bf16_bits_to_f32(got_bits).astype(np.float64)
    ref = syn.bf16_bits_to_f32(ref_bits).astype(np.float64)
    bad = np.argwhere(np.abs(got - ref) > _ulp_bf16(ref))
    assert bad.size == 0, f"{name}: {len(bad)} values beyond one bf16 ulp, first {bad[:4].tolist()}"


class Run:
    """One GPU forward + backward of the MLP with its buffers kept."""

    def __init__(self, nv, M, D, F, seed, step, rht, X, Wg, Wu, Wd, dY, dw_init=0.0):
        import torch
        self.nv, self.M, self.D, self.F = nv, M, D, F
        self.W = [H.dev_f32(w) for w in (Wg, Wu, Wd)]
        self.p = nv.mlp_params(M, D, F, *self.W, seed=seed, step=step, rht=rht)
        sb, wb = nv.mlp_sizes(M, D, F)
        self.saved = torch.empty(sb, dtype=torch.uint8, device="cuda")
        self.ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
        self.Y = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
        self.dX = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
        self.dW = [torch.full((F, D), dw_init, dtype=torch.float32, device="cuda"),
                   torch.full((F, D), dw_init, dtype=torch.float32, device="cuda"),
                   torch.full((D, F), dw_init, dtype=torch.float32, device="cuda")]
        nv.nvfp4_mlp_fwd(self.p, H.dev_bf16(X), self.Y, self.saved, self.ws)
        self.fwd = {k: _bits(self.t(k)).copy() if k != nv.MLP_H else None
                    for k in (nv.MLP_G, nv.MLP_U)}
        self.H_bits = _bits(self.t(nv.MLP_H))          # the workspace is reused by the backward
        self.qH = self._q_host(nv.MLP_Q_H)
        self.qX = self._q_host(nv.MLP_Q_X)
        nv.nvfp4_mlp_bwd(self.p, H.dev_bf16(dY), self.saved, self.dX, *self.dW, self.ws)
        nv.check_device_errors()

    def t(self, which):
        return self.nv.mlp_tensor(self.M, self.D, self.F, self.saved, self.ws, which)

    def q(self, which):
        return self.nv.mlp_operand(self.M, self.D, self.F, self.saved, self.ws, which)

    def _q_host(self, which):
        q = self.q(which)
        return {"codes": _np(q.codes).reshape(q.rows, q.cols // 2).copy(),
                "scales_sw": _np(q.scales).copy(), "amax": float(_np(q.amax)[0]),
                "s_dec": float(_np(q.s_dec)[0]), "rows": q.rows, "cols": q.cols}

    def q_host(self, which):
        if which == self.nv.MLP_Q_H:
            return self.qH
        if which == self.nv.MLP_Q_X:
            return self.qX
        return self._q_host(which)


def _inputs(M, D, F):
    X = syn.activations((M, D), seed=1)
    Wg = syn.weights((F, D), seed=4, master_fp32=True)
    Wu = syn.weights((F, D), seed=5, master_fp32=True)
    Wd = syn.weights((D, F), seed=6, master_fp32=True)
    dY = syn.gradients((M, D), seed=3)
    return X, Wg, Wu, Wd, dY


def _check_operand(orc, gq, x, mode, flags, seed, offset, slabs, name):
    """The GPU's operand gq (host dict) against the oracle's quantisation of
    x: whole (slabs None) or on 128-row slabs with the oracle's own amax."""
    if slabs is None:
        o = orc.quantize(x, mode, flags, seed=seed, offset=offset)
        assert np.array_equal(gq["codes"], o["codes"]), f"{name}: codes differ"
        assert np.array_equal(gq["scales_sw"], o["scales_sw"]), f"{name}: scales differ"
        assert np.float32(gq["amax"]) == o["amax"] and np.float32(gq["s_dec"]) == o["s_dec"], name
        return o
    amax = orc.amax(x, mode, flags & orc.RHT, seed=seed)
    assert np.float32(gq["amax"]).view(np.uint32) == np.float32(amax).view(np.uint32), \
        f"{name}: amax {gq['amax']!r} != oracle {amax!r}"
    os_ = H.oracle_slabs(orc, x, mode, flags, amax, slabs, seed=seed, offset=offset)
    H.assert_slabs_equal(gq["codes"], gq["scales_sw"], gq["amax"], gq["s_dec"], os_, slabs, name)
    return H.compact_operand(os_)


def _check_weight(orc, gq, w, slabs, slabs_t, name):
    """16x16 weight: K-major operand and its transposed view.  Returns the
    oracle operands (whole, or compact slabs of each view)."""
    if slabs is None:
        o = orc.quantize(w, orc.BLOCK_16X16, orc.EMIT_T)
        H.assert_quant_equal(gq, o, name)
        return o, orc.transposed_view(o)
    amax = orc.amax(w, orc.BLOCK_16X16)
    codes = _np(gq.codes).reshape(gq.rows, gq.cols // 2)
    codes_t = _np(gq.codes_t).reshape(gq.cols, gq.rows // 2)
    a, sd = float(_np(gq.amax)[0]), float(_np(gq.s_dec)[0])
    assert np.float32(a) == amax, name
    o = H.oracle_slabs(orc, w, orc.BLOCK_16X16, orc.EMIT_T, amax, slabs)
    H.assert_slabs_equal(codes, _np(gq.scales), a, sd, o, slabs, name)
    ot = H.oracle_slabs_transposed(orc, w, amax, slabs_t)
    H.assert_slabs_equal(codes_t, _np(gq.scales_t), a, sd, ot, slabs_t, name + "^T")
    return H.compact_operand(o), H.compact_operand(ot)


def _check_gemm(orc, got, a, b, a_slabs, b_slabs, name, add=None):
    """GPU GEMM output `got` (device, bf16 or fp32) against the oracle's FP64
    product of a and b (+ add, an FP64 array over the same outputs)."""
    if a_slabs is None:
        ref = orc.gemm_fp64(a, b)
        if add is not None:
            ref = ref + add
        return H.assert_gemm_close(H.host_f64(got), ref, name)
    lm, ln, gm, gn = H.sampled_positions(a_slabs, b_slabs)
    ref = orc.gemm_fp64_sampled(a, b, lm, ln)
    if add is not None:
        ref = ref + add(gm, gn)
    import torch
    sel = got[torch.from_numpy(gm).cuda(), torch.from_numpy(gn).cuda()]
    return H.assert_gemm_close(H.host_f64(sel), ref, name)


def _staged(nv, orc, M, D, F, rht, seed, step, sampled):
    X, Wg, Wu, Wd, dY = _inputs(M, D, F)
    run = Run(nv, M, D, F, seed, step, rht, X, Wg, Wu, Wd, dY)
    rf = orc.RHT if rht else 0
    off = [8 * step + i for i in range(6)]
    rng = np.random.Generator(np.random.PCG64(7))

    def pick(n):  # 128-row slabs: all, or the first, the last and two random
        if not sampled:
            return None
        k = n // 128
        return sorted({0, k - 1} | set(rng.integers(1, k - 1, 2).tolist()))

    sM, sD, sF = pick(M), pick(D), pick(F)
    # ---- weights (16x16 from the FP32 masters) and the forward -------------
    oWg, oWgT = _check_weight(orc, run.q(nv.MLP_Q_WG), Wg, sF, sD, "Wg")
    oWu, oWuT = _check_weight(orc, run.q(nv.MLP_Q_WU), Wu, sF, sD, "Wu")
    oWd, oWdT = _check_weight(orc, run.q(nv.MLP_Q_WD), Wd, sD, sF, "Wd")
    oX = _check_operand(orc, run.q_host(nv.MLP_Q_X), X, orc.ROW_1X16, 0, seed, 0, sM, "X")
    oXc = _check_operand(orc, run.q_host(nv.MLP_Q_XC), X, orc.COL_1X16, rf, seed, 0, sD, "X^T")
    G, U = run.fwd[nv.MLP_G], run.fwd[nv.MLP_U]
    _check_gemm(orc, run.t(nv.MLP_G), oX, oWg, sM, sF, "G = X Wg^T")
    _check_gemm(orc, run.t(nv.MLP_U), oX, oWu, sM, sF, "U = X Wu^T")
    Hb = run.H_bits
    rows = slice(None) if not sampled else np.concatenate([np.arange(s * 128, s * 128 + 128)
                                                           for s in sM])
    _within_one_ulp(Hb[rows], orc.swiglu_fwd(G[rows], U[rows]), "H = silu(G) U")
    oH = _check_operand(orc, run.q_host(nv.MLP_Q_H), Hb, orc.ROW_1X16, 0, seed, 0, sM, "H")
    oHc = _check_operand(orc, run.q_host(nv.MLP_Q_HC), Hb, orc.COL_1X16, rf, seed, 0, sF, "H^T")
    del Hb
    _check_gemm(orc, run.Y, oH, oWd, sM, sD, "Y = H Wd^T")
    del oH
    gc.collect()
    # ---- backward ------------------------------------------------------------
    odY = _check_operand(orc, run.q_host(nv.MLP_Q_DY), dY, orc.ROW_1X16, orc.SR, seed, off[0],
                         sM, "dY")
    odYc = _check_operand(orc, run.q_host(nv.MLP_Q_DYC), dY, orc.COL_1X16, rf | orc.SR, seed,
                          off[1], sD, "dY^T")
    _check_gemm(orc, run.t(nv.MLP_DH), odY, oWdT, sM, sF, "dH = dY Wd")
    _check_gemm(orc, run.dW[2], odYc, oHc, sD, sF, "dWd = dY^T H")
    del odY, odYc, oHc
    dH = _bits(run.t(nv.MLP_DH))
    dG, dU = _bits(run.t(nv.MLP_DG)), _bits(run.t(nv.MLP_DU))
    rdG, rdU = orc.swiglu_bwd(dH[rows], G[rows], U[rows])
    _within_one_ulp(dG[rows], rdG, "dG")
    _within_one_ulp(dU[rows], rdU, "dU")
    del dH, G, U, rdG, rdU
    gc.collect()
    odG = _check_operand(orc, run.q_host(nv.MLP_Q_DG), dG, orc.ROW_1X16, orc.SR, seed, off[2],
                         sM, "dG")
    odGc = _check_operand(orc, run.q_host(nv.MLP_Q_DGC), dG, orc.COL_1X16, rf | orc.SR, seed,
                          off[3], sF, "dG^T")
    del dG
    odU = _check_operand(orc, run.q_host(nv.MLP_Q_DU), dU, orc.ROW_1X16, orc.SR, seed, off[4],
                         sM, "dU")
    odUc = _check_operand(orc, run.q_host(nv.MLP_Q_DUC), dU, orc.COL_1X16, rf | orc.SR, seed,
                          off[5], sF, "dU^T")
    del dU
    gc.collect()
    dXg = run.t(nv.MLP_DX_GATE)
    _check_gemm(orc, dXg, odG, oWgT, sM, sD, "dX_gate = dG Wg")
    dXg64 = H.host_f64(dXg)
    add = dXg64 if not sampled else (lambda m, n: dXg64[m, n])
    _check_gemm(orc, run.dX, odU, oWuT, sM, sD, "dX = dU Wu + dX_gate", add=add)
    _check_gemm(orc, run.dW[0], odGc, oXc, sF, sD, "dWg = dG^T X")
    _check_gemm(orc, run.dW[1], odUc, oXc, sF, sD, "dWu = dU^T X")
    return run, (X, Wg, Wu, Wd, dY)


@pytest.mark.parametrize("M,D,F", [(256, 256, 512), (384, 384, 640)])
@pytest.mark.parametrize("rht", [True, False])
def test_mlp_staged_matches_oracle(nv, orc, M, D, F, rht):
    """Every stage of forward + backward, every element (the second shape is
    ragged against the 256 x 256 tiles of the large-shape GEMM); then the fold
    into FP32 master gradients starting from non-zero values, exactly."""
    import torch
    run, (X, Wg, Wu, Wd, dY) = _staged(nv, orc, M, D, F, rht, seed=11, step=3, sampled=False)
    rng = np.random.Generator(np.random.PCG64(5))
    c = [rng.standard_normal(w.shape).astype(np.float32) for w in (Wg, Wu, Wd)]
    run2 = Run(nv, M, D, F, 11, 3, rht, X, Wg, Wu, Wd, dY, dw_init=0.0)
    for i in range(3):
        run2.dW[i].copy_(torch.from_numpy(c[i]))
    nv.nvfp4_mlp_bwd(run2.p, H.dev_bf16(dY), run2.saved, run2.dX, *run2.dW, run2.ws)
    nv.check_device_errors()
    for i, name in enumerate(("dWg", "dWu", "dWd")):
        exp = torch.from_numpy(c[i]).cuda() + run.dW[i]   # one FP32 add of the bf16 WGRAD
        assert torch.equal(run2.dW[i], exp), f"{name}: the fold is not c + float(bf16(WGRAD))"
    assert torch.equal(run2.dX, run.dX)                    # the backward is deterministic


def test_mlp_staged_llama8b_sampled(nv, orc):
    """The full SwiGLU MLP at Llama-3-8B shape (M = 32768 tokens, D = 4096,
    F = 14336; FP32 master weights, the RHT on the WGRAD operands), stage by
    stage on sampled 128-row slabs and sampled GEMM outputs."""
    _staged(nv, orc, 32768, 4096, 14336, True, seed=0, step=1, sampled=True)


def test_mlp_rejects_bad_shapes(nv):
    with pytest.raises(nv.NVFP4Error) as e:
        nv.mlp_sizes(100, 128, 128)
    assert e.value.status == nv.ERR_SHAPE


def test_mlp_llama8b_full_size_property(nv):
    """The full SwiGLU MLP at Llama-3-8B shape, a property that holds at any
    size: every output stays within the NVFP4 quantisation noise of the
    unquantised FP32 MLP (computed here with PyTorch FP32 matmuls, TF32 off)
    -- the same 0.45 relative-Frobenius bound the oracle tests pin for the
    oracle's own NVFP4 MLP against the exact one, far below the error of a
    wrong operand or a transposed view (> 1)."""
    import torch
    M, D, F = 32768, 4096, 14336
    torch.backends.cuda.matmul.allow_tf32 = False
    X = H.dev_bf16(syn.activations((M, D), seed=1))
    Wg, Wu = (H.dev_f32(syn.weights((F, D), seed=s, master_fp32=True)) for s in (4, 5))
    Wd = H.dev_f32(syn.weights((D, F), seed=6, master_fp32=True))
    dY = H.dev_bf16(syn.gradients((M, D), seed=3))
    p = nv.mlp_params(M, D, F, Wg, Wu, Wd, seed=0, step=0, rht=True)
    sb, wb = nv.mlp_sizes(M, D, F)
    saved = torch.empty(sb, dtype=torch.uint8, device="cuda")
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    Y = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    dX = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    gWg, gWu = (torch.zeros(F, D, dtype=torch.float32, device="cuda") for _ in range(2))
    gWd = torch.zeros(D, F, dtype=torch.float32, device="cuda")
    nv.nvfp4_mlp_fwd(p, X, Y, saved, ws)
    nv.nvfp4_mlp_bwd(p, dY, saved, dX, gWg, gWu, gWd, ws)
    nv.check_device_errors()
    del saved, ws

    def rel(a, b):
        return float(torch.linalg.norm((a.float() - b).flatten()) / torch.linalg.norm(b.flatten()))

    Xf, dYf = X.float(), dY.float()
    G = Xf @ Wg.t()
    U = Xf @ Wu.t()
    sg = torch.sigmoid(G)
    Hf = G * sg * U
    errs = {"Y": rel(Y, Hf @ Wd.t())}
    dH = dYf @ Wd
    dG = dH * U * (sg * (1 + G * (1 - sg)))
    dU = dH * G * sg
    errs["dWd"] = rel(gWd, dYf.t() @ Hf)
    del Hf, G, U, sg, dH
    errs["dX"] = rel(dX, dG @ Wg + dU @ Wu)
    errs["dWg"] = rel(gWg, dG.t() @ Xf)
    errs["dWu"] = rel(gWu, dU.t() @ Xf)
    assert all(np.isfinite(e) and e < 0.45 for e in errs.values()), errs
