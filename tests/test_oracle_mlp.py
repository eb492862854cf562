"""Pins of the oracle SwiGLU and MLP composition -- CPU only.

The SwiGLU forward/backward are checked against torch autograd in float64 (a
library derivative, not a retyped formula).  The NVFP4 MLP composition is
checked against the unquantised FP64 MLP with autograd: the NVFP4 noise of
three chained quantised operands gives relative errors of 0.2-0.3 at this
size, while a swapped operand, a sign error or a permuted row gives errors
above 1.
"""
import importlib

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_03_gb300 import synthetic as syn


def _f64(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def test_swiglu_matches_autograd(orc):
    rng = np.random.Generator(np.random.PCG64(41))
    g = syn.f32_to_bf16_bits((rng.standard_normal(4096) * 3).astype(np.float32))
    u = syn.f32_to_bf16_bits(rng.standard_normal(4096).astype(np.float32))
    dh = syn.f32_to_bf16_bits(rng.standard_normal(4096).astype(np.float32))
    gt = torch.tensor(_f64(g), requires_grad=True)
    ut = torch.tensor(_f64(u), requires_grad=True)
    h = torch.nn.functional.silu(gt) * ut
    h.backward(torch.tensor(_f64(dh)))
    ref_h = orc.bf16_round_f64(h.detach().numpy())
    ref_dg = orc.bf16_round_f64(gt.grad.numpy())
    ref_du = orc.bf16_round_f64(ut.grad.numpy())
    got_h = orc.swiglu_fwd(g, u)
    got_dg, got_du = orc.swiglu_bwd(dh, g, u)
    # exp() of two libraries may differ in the last FP64 bit: allow 1 bf16 step
    for got, ref in ((got_h, ref_h), (got_dg, ref_dg), (got_du, ref_du)):
        diff = np.abs(got.astype(np.int32) - ref.astype(np.int32))
        assert (diff <= 1).all() and (diff == 0).mean() > 0.999


def test_swiglu_extreme_gates(orc):
    """Gates across the range the outlier rows of the synthetic activations
    reach (|g| up to 129, beyond where an FP32 e^-g overflows), against torch
    autograd in FP64; and at g = 0 the closed forms silu(0) = 0 and
    silu'(0) = 1/2, so dG = dH * u / 2 and dU = 0 there."""
    gv = np.array([-129.0, -100.0, -90.5, -89.0, -88.5, -60.0, -20.0, -1.0, 0.0, 1.0, 20.0,
                   60.0, 89.0, 129.0], np.float32)
    g = np.repeat(syn.f32_to_bf16_bits(gv), 3)
    u = np.tile(syn.f32_to_bf16_bits(np.array([0.875, -1.25, 3.0], np.float32)), len(gv))
    dh = np.tile(syn.f32_to_bf16_bits(np.array([1.0, -0.5, 2.0], np.float32)), len(gv))
    gt = torch.tensor(_f64(g), requires_grad=True)
    ut = torch.tensor(_f64(u), requires_grad=True)
    h = torch.nn.functional.silu(gt) * ut
    h.backward(torch.tensor(_f64(dh)))
    got_h = orc.swiglu_fwd(g, u)
    got_dg, got_du = orc.swiglu_bwd(dh, g, u)
    for got, ref in ((got_h, h.detach().numpy()), (got_dg, gt.grad.numpy()),
                     (got_du, ut.grad.numpy())):
        diff = np.abs(got.astype(np.int32) - orc.bf16_round_f64(ref).astype(np.int32))
        assert (diff <= 1).all()
    # the silu(g) u of the outlier gates is a normal bf16 number, not zero
    i = int(np.where(gv == -89.0)[0][0]) * 3
    assert 1e-38 < abs(_f64(got_h[i:i + 1])[0]) < 1e-36
    z = int(np.where(gv == 0.0)[0][0]) * 3
    np.testing.assert_array_equal(_f64(got_h[z:z + 3]), 0.0)
    np.testing.assert_array_equal(_f64(got_du[z:z + 3]), 0.0)
    np.testing.assert_array_equal(_f64(got_dg[z:z + 3]), _f64(dh[z:z + 3]) * _f64(u[z:z + 3]) / 2)


def _mlp(orc):
    """The MLP composition of the oracle package `orc` (the oracle itself, or
    a copy under test)."""
    return importlib.import_module(orc.__name__ + ".mlp")


def _torch_mlp(X, Wg, Wu, Wd, dY):
    Xt = torch.tensor(_f64(X), requires_grad=True)
    ws = [torch.tensor(w.astype(np.float64), requires_grad=True) for w in (Wg, Wu, Wd)]
    G = Xt @ ws[0].T
    U = Xt @ ws[1].T
    Y = (torch.nn.functional.silu(G) * U) @ ws[2].T
    Y.backward(torch.tensor(_f64(dY)))
    return Y.detach().numpy(), Xt.grad.numpy(), [w.grad.numpy() for w in ws]


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("rht", [False, True])
def test_nvfp4_mlp_tracks_fp64_mlp(orc, rht):
    mlp_bwd, mlp_fwd = _mlp(orc).mlp_bwd, _mlp(orc).mlp_fwd
    M, D, F = 128, 64, 96
    X = syn.activations((M, D), seed=1)
    Wg = syn.weights((F, D), seed=4, master_fp32=True) * np.float32(5)
    Wu = syn.weights((F, D), seed=5, master_fp32=True) * np.float32(5)
    Wd = syn.weights((D, F), seed=6, master_fp32=True) * np.float32(5)
    dY = syn.gradients((M, D), seed=3)
    Y, saved = mlp_fwd(X, Wg, Wu, Wd, seed=0, rht=rht)
    dWg, dWu, dWd = (np.zeros_like(w) for w in (Wg, Wu, Wd))
    dX, _ = mlp_bwd(dY, saved, dWg, dWu, dWd, step=0)
    rY, rdX, (rdWg, rdWu, rdWd) = _torch_mlp(X, Wg, Wu, Wd, dY)
    errs = {"Y": _rel(_f64(Y), rY), "dX": _rel(_f64(dX), rdX), "dWg": _rel(dWg, rdWg),
            "dWu": _rel(dWu, rdWu), "dWd": _rel(dWd, rdWd)}
    for k, e in errs.items():
        assert e < 0.45, (k, errs)   # measured 0.19-0.30 over seeds 0-2
    # a swapped operand, a sign error or a row permutation is far outside it
    assert _rel(dWg, rdWu) > 1.0 and _rel(_f64(dX), -rdX) > 1.5
    assert _rel(_f64(Y), rY[::-1]) > 1.0


# ---- the recipe's per-operand choices inside the composition -------------------
_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _sr_decisions(orc, q, v_bits):
    """For each element of the quantised operand q of the bf16 values v (in
    q's output layout): frac = (|y| - lo) / (hi - lo) of y = v * s_enc / S_b
    on the E2M1 grid, and whether the code took hi; elements on the grid or
    saturated are dropped.  Float64 here: only used to bin fractions."""
    v = np.abs(syn.bf16_bits_to_f32(v_bits).astype(np.float64))
    S = np.array([orc.e4m3_value(int(b)) for b in range(256)])[q["scales"]]
    S = np.repeat(S, 16, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(S > 0, v * float(q["s_enc"]) / S, 0.0)
    codes = q["codes"]
    nib = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    nib[:, 0::2], nib[:, 1::2] = codes & 7, (codes >> 4) & 7
    mag = _GRID[nib]
    hi_i = np.clip(np.searchsorted(_GRID, y, side="right"), 1, 7)
    lo, hi = _GRID[hi_i - 1], _GRID[hi_i]
    keep = (y < 6.0) & (y != lo) & (S > 0)
    frac = (y - lo) / (hi - lo)
    return frac[keep], (mag == hi)[keep], keep


def _rht_of_transpose(orc, x_bits, seed):
    """(1/4) H16 diag(s) applied to each 16-element block of every row of x^T
    (x: bf16 bits [M, N] -> [N, M] float64), H16 = scipy's Sylvester matrix."""
    from scipy.linalg import hadamard
    xt = syn.bf16_bits_to_f32(x_bits).astype(np.float64).T
    T = hadamard(16) @ np.diag(orc.rht_signs(seed).astype(np.float64)) / 4.0
    n, m = xt.shape
    return (xt.reshape(n, m // 16, 16) @ T.T).reshape(n, m)


@pytest.fixture(scope="module")
def mlp_run(orc):
    return make_mlp_run(orc)


def make_mlp_run(orc):
    """One forward and the backward of two steps of a small MLP, through the
    composition of the oracle package `orc`."""
    mlp_bwd, mlp_fwd = _mlp(orc).mlp_bwd, _mlp(orc).mlp_fwd
    M, D, F = 256, 64, 128
    X = syn.activations((M, D), seed=1)
    Wg = syn.weights((F, D), seed=4, master_fp32=True) * np.float32(5)
    Wu = syn.weights((F, D), seed=5, master_fp32=True) * np.float32(5)
    Wd = syn.weights((D, F), seed=6, master_fp32=True) * np.float32(5)
    dY = syn.gradients((M, D), seed=3)
    _, saved = mlp_fwd(X, Wg, Wu, Wd, seed=7, rht=True)
    steps = []
    for step in (0, 1):
        dW = [np.zeros_like(w) for w in (Wg, Wu, Wd)]
        steps.append(mlp_bwd(dY, saved, *dW, step=step)[1])
    return X, dY, saved, steps


def test_mlp_gradient_operands_are_stochastically_rounded(orc, mlp_run):
    """dY, dG, dU (row and column operands) are stochastically rounded: an
    element rounds up with probability equal to its fraction between the
    two grid neighbours (binomial bound per fraction bin), so round-to-
    nearest -- up exactly when frac > 1/2 -- fails every bin."""
    X, dY, saved, steps = mlp_run
    b = steps[0]
    srcs = {"qdY": dY, "qdG": b["dG"], "qdU": b["dU"]}
    for name in ("qdY", "qdG", "qdU"):
        frac, up, _ = _sr_decisions(orc, b[name], srcs[name])
        for lo_f, hi_f in ((0.05, 0.2), (0.2, 0.4), (0.6, 0.8), (0.8, 0.95)):
            sel = (frac >= lo_f) & (frac < hi_f)
            n = int(sel.sum())
            assert n > 500, (name, lo_f, n)
            p, want = up[sel].mean(), frac[sel].mean()
            assert abs(p - want) < 5 * np.sqrt(0.25 / n), (name, lo_f, p, want)


def test_mlp_sr_operands_draw_independent_words(orc, mlp_run):
    """The six SR operands of a step, and one operand across two steps, draw
    their Philox words independently (distinct counter offsets): the rounding
    decisions of any two, paired by output index, are uncorrelated.  Sharing
    an offset would pair identical words, r < T1 and r < T2, a correlation of
    (min(f1, f2) - f1 f2) / sqrt(f1 (1 - f1) f2 (1 - f2)), about 0.5 here."""
    X, dY, saved, steps = mlp_run
    sr_offsets = _mlp(orc).sr_offsets
    assert len(set(sr_offsets(0).values()) | set(sr_offsets(1).values())) == 12
    b0, b1 = steps

    def dec(b, name, src):
        q = b[name]
        if name.endswith("c"):
            return None   # column operands: their fractions need the transformed values
        frac, up, keep = _sr_decisions(orc, q, src)
        f = np.full(keep.shape, np.nan)
        u = np.full(keep.shape, np.nan)
        f[keep], u[keep] = frac, up
        return f.ravel(), u.ravel()

    ops = {("0", "qdY"): dec(b0, "qdY", dY), ("0", "qdG"): dec(b0, "qdG", b0["dG"]),
           ("0", "qdU"): dec(b0, "qdU", b0["dU"]), ("1", "qdG"): dec(b1, "qdG", b1["dG"])}
    keys = list(ops)
    for i in range(len(keys)):
        for j in range(i + 1, len(keys)):
            (f1, u1), (f2, u2) = ops[keys[i]], ops[keys[j]]
            n = min(len(f1), len(f2))
            f1, u1, f2, u2 = f1[:n], u1[:n], f2[:n], u2[:n]
            ok = ~(np.isnan(f1) | np.isnan(f2))
            num = np.sum((u1[ok] - f1[ok]) * (u2[ok] - f2[ok]))
            den = np.sqrt(np.sum(f1[ok] * (1 - f1[ok])) * np.sum(f2[ok] * (1 - f2[ok])))
            c = num / den
            assert abs(c) < 5 / np.sqrt(ok.sum()), (keys[i], keys[j], c)
    # the column operands: same words would make their codes' parity pattern
    # repeat the row operand's at equal linear index; check code agreement is
    # at the level two independent roundings give
    for name in ("qdYc", "qdGc", "qdUc"):
        assert not np.array_equal(b0[name]["codes"], b1[name]["codes"]), name


def test_mlp_wgrad_operands_carry_the_rht(orc, mlp_run):
    """Every column (WGRAD) operand of the composition -- X^T, H^T, dY^T, dG^T,
    dU^T -- encodes (1/4) H16 diag(s) of its tensor's 16-token blocks, with
    the same signs s for all of them (so the transform cancels in each
    product): its dequantisation is within NVFP4 noise of that transform
    (computed here with scipy's Hadamard matrix) and far from the
    untransformed transpose."""
    X, dY, saved, steps = mlp_run
    b = steps[0]
    for name, q, src in (("X^T", saved["qXc"], X), ("H^T", saved["qHc"], saved["H"]),
                         ("dY^T", b["qdYc"], dY), ("dG^T", b["qdGc"], b["dG"]),
                         ("dU^T", b["qdUc"], b["dU"])):
        deq = orc.dequant(q)
        T = _rht_of_transpose(orc, src, 7)
        plain = syn.bf16_bits_to_f32(src).astype(np.float64).T
        assert _rel(deq, T) < 0.3, (name, _rel(deq, T))
        assert _rel(deq, plain) > 0.7, (name, _rel(deq, plain))


# ---- the optimizer step (FP32 master weight, plain SGD) -----------------------------
def test_sgd_step_exact_on_representable_values(orc):
    """Integers times a power of two: every product and difference is exact in
    binary32, so the step must equal the exact FP64 result element for element,
    and the amax the largest magnitude of it."""
    sgd_step = _mlp(orc).sgd_step
    rng = np.random.Generator(np.random.PCG64(61))
    W = rng.integers(-4096, 4096, (48, 64)).astype(np.float32)
    G = rng.integers(-4096, 4096, (48, 64)).astype(np.float32)
    for lr in (0.5, 0.25, 2.0, -1.0):
        Wn, Gn, a = sgd_step(W, G, lr)
        exact = W.astype(np.float64) - lr * G.astype(np.float64)
        assert np.array_equal(Wn.astype(np.float64), exact)
        assert np.array_equal(Gn, G)
        assert a == np.float32(np.abs(exact).max())


def test_sgd_step_rounds_the_product_first(orc):
    """lr = G = 1 + 2^-23: lr * G = 1 + 2^-22 + 2^-46 rounds to 1 + 2^-22, so
    W = 1 + 2^-22 steps exactly to 0; a fused multiply-add would leave -2^-46.
    W = 3 with G = 0.1 (not a binary32 value times lr = 0.1) checks the
    rounding of the difference against an FP64 evaluation of the same two
    rounded operations."""
    sgd_step = _mlp(orc).sgd_step
    one_ulp = np.float32(1 + 2.0 ** -23)
    W = np.array([[np.float32(1 + 2.0 ** -22), 3.0, -0.5, 7.0]], np.float32)
    G = np.array([[one_ulp, 0.1, 0.0, -2.0]], np.float32)
    Wn, _, _ = sgd_step(W[:, :1], G[:, :1], float(one_ulp))
    assert Wn[0, 0] == 0.0 and not np.signbit(Wn[0, 0])
    Wn, _, a = sgd_step(W, G, 0.1)
    prod = np.float32(np.float64(np.float32(0.1)) * np.float64(G[0, 1]))
    assert Wn[0, 1] == np.float32(np.float64(W[0, 1]) - np.float64(prod))
    assert Wn[0, 2] == np.float32(-0.5) and Wn[0, 3] == np.float32(7.0) + np.float32(0.2)
    assert a == np.abs(Wn).max()


def test_sgd_step_zero_grad_and_zero_rate(orc):
    """zero_grad clears the gradient; lr = 0 leaves a weight without negative
    zeros unchanged bit for bit; the amax equals the one the oracle's 16x16
    quantiser takes of the updated weight (its own C reduction)."""
    sgd_step = _mlp(orc).sgd_step
    rng = np.random.Generator(np.random.PCG64(62))
    W = (rng.standard_normal((32, 48)) * 0.02).astype(np.float32)
    W[W == 0] = 1e-3
    G = (rng.standard_normal((32, 48)) * 1e-3).astype(np.float32)
    Wn, Gn, a = sgd_step(W, G, 0.0, zero_grad=True)
    assert np.array_equal(Wn.view(np.uint32), W.view(np.uint32))
    assert not Gn.any()
    Wn, _, a = sgd_step(W, G, 3e-2)
    q = orc.quantize(Wn, orc.BLOCK_16X16, orc.EMIT_T)
    assert a == q["amax"] == np.abs(Wn).max()
