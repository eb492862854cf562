"""GPU parity of the SwiGLU MLP forward + backward (nine NVFP4 GEMMs) and of
the SwiGLU kernels, against the oracle composition.

The composed MLP cannot be bit-identical to the oracle: its GEMMs are within
the GEMM tolerance, not exact, so an intermediate BF16 value (G, U, H, dH)
may differ by an ulp and move a downstream quantisation decision by one grid
step.  The bound below is therefore on the relative Frobenius error of each
output against the oracle's, 2e-2, an order of magnitude under the NVFP4
quantisation noise of the outputs themselves (0.2-0.3 against the
unquantised FP64 MLP, pinned in the oracle tests) and far under the error of
a wrong operand (> 1).
"""
import numpy as np
import pytest

import gpu_helpers as H
from nvfp4_block_scaled_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
REL_FROB = 2e-2


@pytest.fixture(scope="module")
def nv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_03_gb300 import binding
    return binding


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("rht", [True, False])
def test_mlp_fwd_bwd_matches_oracle(nv, orc, rht):
    import torch

    from oracle.mlp import mlp_bwd, mlp_fwd
    M, D, F = 256, 256, 512
    X = syn.activations((M, D), seed=1)
    Wg = syn.weights((F, D), seed=4, master_fp32=True)
    Wu = syn.weights((F, D), seed=5, master_fp32=True)
    Wd = syn.weights((D, F), seed=6, master_fp32=True)
    dY = syn.gradients((M, D), seed=3)
    # oracle
    oY, saved = mlp_fwd(X, Wg, Wu, Wd, seed=11, rht=rht)
    odWg, odWu, odWd = (np.full(w.shape, 0.5, np.float32) for w in (Wg, Wu, Wd))
    odX, _ = mlp_bwd(dY, saved, odWg, odWu, odWd, step=3)
    # GPU
    Wg_d, Wu_d, Wd_d = (H.dev_f32(w) for w in (Wg, Wu, Wd))
    p = nv.mlp_params(M, D, F, Wg_d, Wu_d, Wd_d, seed=11, step=3, rht=rht)
    sb, wb = nv.mlp_sizes(M, D, F)
    saved_d = torch.empty(sb, dtype=torch.uint8, device="cuda")
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    Y = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_mlp_fwd(p, H.dev_bf16(X), Y, saved_d, ws)
    dX = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    gWg, gWu, gWd = (torch.full(w.shape, 0.5, dtype=torch.float32, device="cuda")
                     for w in (Wg, Wu, Wd))
    nv.nvfp4_mlp_bwd(p, H.dev_bf16(dY), saved_d, dX, gWg, gWu, gWd, ws)
    nv.check_device_errors()
    errs = {
        "Y": _rel(H.host_f64(Y), syn.bf16_bits_to_f32(oY).astype(np.float64)),
        "dX": _rel(H.host_f64(dX), syn.bf16_bits_to_f32(odX).astype(np.float64)),
        "dWg": _rel(gWg.cpu().numpy() - 0.5, odWg - 0.5),
        "dWu": _rel(gWu.cpu().numpy() - 0.5, odWu - 0.5),
        "dWd": _rel(gWd.cpu().numpy() - 0.5, odWd - 0.5),
    }
    assert all(e < REL_FROB for e in errs.values()), errs


def test_mlp_rejects_bad_shapes(nv):
    with pytest.raises(nv.NVFP4Error) as e:
        nv.mlp_sizes(100, 128, 128)
    assert e.value.status == nv.ERR_SHAPE


def test_mlp_llama8b_full_size_property(nv):
    """The full SwiGLU MLP at Llama-3-8B shape (M = 32768 tokens, D = 4096,
    F = 14336; FP32 master weights, 9 NVFP4 GEMMs).  The oracle cannot
    compose nine FP64 GEMMs of this size, and a sampled output needs the
    per-tensor amax of the whole intermediate H, so this checks a property
    that holds at any size: every output stays within the NVFP4 quantisation
    noise of the unquantised FP32 MLP (computed here with PyTorch FP32 matmuls,
    TF32 off) -- the same 0.45 relative-Frobenius bound the oracle tests pin
    for the oracle's own NVFP4 MLP against the exact one, far below the
    error of a wrong operand or a transposed view (> 1)."""
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
