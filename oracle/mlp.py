"""Oracle SwiGLU MLP forward + backward with NVFP4 GEMMs -- TEST INFRASTRUCTURE.

Composition of the oracle primitives in the order the "NVFP4 pretraining
recipe" page's Figure 1 text describes for one linear layer, applied to the
three MLP projections (gate, up, down):

* FPROP:  X (1x16, RNE) x W (16x16, RNE)                    -> BF16
* DGRAD:  dY (1x16, SR) x W read through its transpose       -> BF16
* WGRAD:  (RHT dY)^T (1x16, SR) x (RHT X)^T (1x16, RNE)      -> BF16, then
  folded into the FP32 master gradient (BF16 outputs "folded into an FP32
  master weight on the optimizer step").

The SwiGLU between the GEMMs is evaluated in FP64 and rounded to bf16.  The
two DGRAD products that form dX are summed in FP64 and rounded once.

Stochastic-rounding offsets per step: dY row/col, dG row/col, dU row/col use
offsets 8*step + 0..5; the RHT sign vector depends on the seed only, so every
WGRAD pair shares it.
"""
from __future__ import annotations

import numpy as np

from . import (BLOCK_16X16, COL_1X16, EMIT_T, RHT, ROW_1X16, SR, bf16_round_f64, bf16_to_f32,
               gemm_fp64, quantize, swiglu_bwd, swiglu_fwd, transposed_view)


def _bf16_gemm(qa, qb):
    return bf16_round_f64(gemm_fp64(qa, qb))


def sr_offsets(step: int):
    b = 8 * step
    return {"dy_row": b + 0, "dy_col": b + 1, "dg_row": b + 2, "dg_col": b + 3,
            "du_row": b + 4, "du_col": b + 5}


def mlp_fwd(X, Wg, Wu, Wd, seed: int = 0, rht: bool = True):
    """X bf16 bits [M, D]; Wg, Wu float32 [F, D]; Wd float32 [D, F]."""
    rf = RHT if rht else 0
    qWg = quantize(Wg, BLOCK_16X16, EMIT_T)
    qWu = quantize(Wu, BLOCK_16X16, EMIT_T)
    qWd = quantize(Wd, BLOCK_16X16, EMIT_T)
    qX = quantize(X, ROW_1X16)
    qXc = quantize(X, COL_1X16, rf, seed=seed)
    G = _bf16_gemm(qX, qWg)
    U = _bf16_gemm(qX, qWu)
    H = swiglu_fwd(G, U)
    qH = quantize(H, ROW_1X16)
    qHc = quantize(H, COL_1X16, rf, seed=seed)
    Y = _bf16_gemm(qH, qWd)
    saved = {"G": G, "U": U, "H": H, "qX": qX, "qXc": qXc, "qH": qH, "qHc": qHc, "qWg": qWg,
             "qWu": qWu, "qWd": qWd, "seed": seed, "rht": rht}
    return Y, saved


def mlp_bwd(dY, saved, dWg, dWu, dWd, step: int = 0):
    """dY bf16 bits [M, D]; dWg, dWu, dWd float32 master gradients, updated in place.
    Returns dX and the backward's intermediates (dH, dG, dU as bf16 bits and
    the six quantised gradient operands)."""
    seed, rf = saved["seed"], (RHT if saved["rht"] else 0)
    off = sr_offsets(step)
    qdY = quantize(dY, ROW_1X16, SR, seed=seed, offset=off["dy_row"])
    qdYc = quantize(dY, COL_1X16, rf | SR, seed=seed, offset=off["dy_col"])
    dH = _bf16_gemm(qdY, transposed_view(saved["qWd"]))
    dWd += bf16_to_f32(_bf16_gemm(qdYc, saved["qHc"]))
    dG, dU = swiglu_bwd(dH, saved["G"], saved["U"])
    qdG = quantize(dG, ROW_1X16, SR, seed=seed, offset=off["dg_row"])
    qdGc = quantize(dG, COL_1X16, rf | SR, seed=seed, offset=off["dg_col"])
    qdU = quantize(dU, ROW_1X16, SR, seed=seed, offset=off["du_row"])
    qdUc = quantize(dU, COL_1X16, rf | SR, seed=seed, offset=off["du_col"])
    dX = bf16_round_f64(gemm_fp64(qdG, transposed_view(saved["qWg"])) +
                        gemm_fp64(qdU, transposed_view(saved["qWu"])))
    dWg += bf16_to_f32(_bf16_gemm(qdGc, saved["qXc"]))
    dWu += bf16_to_f32(_bf16_gemm(qdUc, saved["qXc"]))
    return dX, {"dH": dH, "dG": dG, "dU": dU, "qdY": qdY, "qdYc": qdYc, "qdG": qdG,
                "qdGc": qdGc, "qdU": qdU, "qdUc": qdUc}


def sgd_step(W, G, lr: float, zero_grad: bool = False):
    """The optimizer step of an FP32 master weight, with the amax its next
    16x16 quantisation takes.  The page's Figure 1 text folds the GEMMs' BF16
    outputs into an FP32 master weight on the optimizer step, and the weights
    are quantised under a per-tensor scale from their amax every step.  The
    pages name no optimizer; this is plain SGD, elementwise in binary32 with
    the product rounded before the difference (numpy float32 arithmetic
    rounds each operation; no fused multiply-add):
        W_new = W - lr * G,   G_new = 0 (zero_grad) or G,
        amax  = max |W_new| over every element (the per-tensor amax of
                W_new's 16x16 quantisation, which reduces no other way).
    W, G: float32 arrays of one shape.  Returns (W_new, G_new, amax)."""
    W = np.asarray(W, np.float32)
    G = np.asarray(G, np.float32)
    prod = np.multiply(np.float32(lr), G, dtype=np.float32)
    W_new = np.subtract(W, prod, dtype=np.float32)
    G_new = np.zeros_like(G) if zero_grad else G.copy()
    return W_new, G_new, np.float32(np.abs(W_new).max())
