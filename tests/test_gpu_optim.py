"""GPU parity of the optimizer step of an FP32 master weight fused with its
amax (nvfp4_sgd_step), and of the MLP forward that takes the weights'
amaxes from it ("NVFP4 pretraining recipe" page, Figure 1 text: BF16
outputs folded into FP32 master weights on the optimizer step; the weights
quantised 16x16 under a per-tensor scale every step).

The update is elementwise binary32 (the product rounded, then the
difference), so the updated weight, the cleared gradient and the amax are
compared bit for bit with the oracle's step on the same inputs.
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


def _weights(shape, seed):
    """A master weight and gradient with the values an update meets: normal
    weights and gradients, exact zeros, negative zeros, tiny and large
    gradients, and the product-first rounding case of the oracle's pin."""
    rng = np.random.Generator(np.random.PCG64(seed))
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    G = (rng.standard_normal(shape) * 1e-3).astype(np.float32)
    flat_w, flat_g = W.reshape(-1), G.reshape(-1)
    n = flat_w.size
    k = rng.integers(0, n, 64)
    flat_g[k[:16]] = 0.0
    flat_g[k[16:24]] = -0.0
    flat_w[k[24:32]] = -0.0
    flat_g[k[32:40]] = rng.standard_normal(8).astype(np.float32) * 1e3
    flat_g[k[40:48]] = rng.standard_normal(8).astype(np.float32) * 1e-30
    flat_w[k[48]] = np.float32(1 + 2.0 ** -22)
    flat_g[k[48]] = np.float32(1 + 2.0 ** -23)
    return W, G


def _step(nv, W, G, lr, zero):
    import torch
    dW, dG = H.dev_f32(W), H.dev_f32(G)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    nv.nvfp4_sgd_step(dW, dG, lr, zero_grad=zero, amax=amax)
    nv.check_device_errors()
    return dW.cpu().numpy(), dG.cpu().numpy(), np.float32(amax.cpu().numpy()[0])


@pytest.mark.parametrize("shape", [(64, 64), (96, 80), (1, 4), (3, 1000), (2048, 2052)])
@pytest.mark.parametrize("lr,zero", [(1e-3, True), (0.5, False), (0.0, True),
                                     (float(np.float32(1 + 2.0 ** -23)), False)])
def test_sgd_step_matches_oracle(nv, shape, lr, zero):
    from oracle.mlp import sgd_step
    W, G = _weights(shape, seed=11 + shape[0])
    gw, gg, ga = _step(nv, W, G, lr, zero)
    ow, og, oa = sgd_step(W, G, lr, zero_grad=zero)
    assert np.array_equal(gw.view(np.uint32), ow.view(np.uint32)), "updated weight differs"
    assert np.array_equal(gg.view(np.uint32), og.view(np.uint32)), "gradient differs"
    assert ga == oa, f"amax {ga} != {oa}"


def test_sgd_step_without_amax_and_full_size(nv):
    """The Llama-3-8B gate projection's master weight [14336, 4096] (235 MB
    each for W and G): bit-exact against the oracle, and the same update
    without the amax output (a single launch) writes the same weight."""
    import torch
    from oracle.mlp import sgd_step
    W, G = _weights((14336, 4096), seed=5)
    gw, gg, ga = _step(nv, W, G, 3e-4, True)
    ow, og, oa = sgd_step(W, G, 3e-4, zero_grad=True)
    assert np.array_equal(gw.view(np.uint32), ow.view(np.uint32))
    assert not gg.any() and ga == oa
    dW, dG = H.dev_f32(W), H.dev_f32(G)
    nv.nvfp4_sgd_step(dW, dG, 3e-4)
    nv.check_device_errors()
    assert np.array_equal(dW.cpu().numpy().view(np.uint32), ow.view(np.uint32))
    assert torch.equal(dG, H.dev_f32(G))


def test_sgd_amax_gives_the_quantiser_its_own_amax(nv, orc):
    """The amax the step writes equals what nvfp4_amax and the 16x16
    quantiser take of the updated weight, and quantising with it given
    (NVFP4_AMAX_GIVEN) writes the same codes and scales as the quantiser's
    own amax pass."""
    import torch
    W, G = _weights((512, 768), seed=3)
    dW, dG = H.dev_f32(W), H.dev_f32(G)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    nv.nvfp4_sgd_step(dW, dG, 1e-2, amax=amax)
    ref = torch.zeros(1, dtype=torch.float32, device="cuda")
    nv.nvfp4_amax(dW, amax_plain=ref)
    assert torch.equal(amax, ref)
    q_own = nv.nvfp4_quantize(dW, nv.BLOCK_16X16, nv.EMIT_T)
    q_given = nv.nvfp4_quantize(dW, nv.BLOCK_16X16, nv.EMIT_T, amax=amax.clone())
    nv.check_device_errors()
    for a, b in ((q_own.codes, q_given.codes), (q_own.scales, q_given.scales),
                 (q_own.codes_t, q_given.codes_t), (q_own.scales_t, q_given.scales_t),
                 (q_own.s_dec, q_given.s_dec)):
        assert torch.equal(a, b)
    H.assert_quant_equal(q_given, orc.quantize(dW.cpu().numpy(), orc.BLOCK_16X16, orc.EMIT_T),
                         "W after the step")


@pytest.mark.parametrize("rht", [True, False])
def test_mlp_forward_with_weight_amaxes_from_the_step(nv, rht):
    """Training-step order: backward folds WGRAD into the FP32 master
    gradients, the optimizer step updates the masters and writes their amaxes
    straight into the next forward's weight-operand slots, the forward takes
    them (NVFP4_AMAX_GIVEN).  Against a forward that takes the amaxes itself
    on the same updated weights: every weight operand and Y identical."""
    import torch
    M, D, F = 256, 256, 512
    X = syn.activations((M, D), seed=1)
    Ws = [syn.weights((F, D), seed=4, master_fp32=True),
          syn.weights((F, D), seed=5, master_fp32=True),
          syn.weights((D, F), seed=6, master_fp32=True)]
    dY = syn.gradients((M, D), seed=3)
    sb, wb = nv.mlp_sizes(M, D, F)

    def buffers():
        return (torch.empty(sb, dtype=torch.uint8, device="cuda"),
                torch.empty(wb, dtype=torch.uint8, device="cuda"))

    # step 0: forward + backward into zeroed master gradients
    W = [H.dev_f32(w) for w in Ws]
    grads = [torch.zeros_like(w) for w in W]
    saved, ws = buffers()
    p = nv.mlp_params(M, D, F, *W, seed=9, step=0, rht=rht)
    Y = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    dX = torch.empty_like(Y)
    nv.nvfp4_mlp_fwd(p, H.dev_bf16(X), Y, saved, ws)
    nv.nvfp4_mlp_bwd(p, H.dev_bf16(dY), saved, dX, *grads, ws)
    # two copies of the masters and gradients: A steps without the amax, B with it
    WA, GA = [w.clone() for w in W], [g.clone() for g in grads]
    slots = [nv.MLP_Q_WG, nv.MLP_Q_WU, nv.MLP_Q_WD]
    for w, g, which in zip(W, grads, slots):
        op = nv.mlp_operand(M, D, F, saved, ws, which)
        nv.nvfp4_sgd_step(w, g, 5e-2, zero_grad=True, amax=op.amax)
    for w, g in zip(WA, GA):
        nv.nvfp4_sgd_step(w, g, 5e-2, zero_grad=True)
    for w, wa in zip(W, WA):
        assert torch.equal(w, wa)
    # step 1: B's forward with the given amaxes, A's forward taking its own
    pB = nv.mlp_params(M, D, F, *W, seed=9, step=1, rht=rht, weight_amax_given=True)
    YB = torch.empty_like(Y)
    nv.nvfp4_mlp_fwd(pB, H.dev_bf16(X), YB, saved, ws)
    savedA, wsA = buffers()
    pA = nv.mlp_params(M, D, F, *WA, seed=9, step=1, rht=rht)
    YA = torch.empty_like(Y)
    nv.nvfp4_mlp_fwd(pA, H.dev_bf16(X), YA, savedA, wsA)
    nv.check_device_errors()
    for which in slots:
        a = nv.mlp_operand(M, D, F, savedA, wsA, which)
        b = nv.mlp_operand(M, D, F, saved, ws, which)
        for x, y in ((a.codes, b.codes), (a.scales, b.scales), (a.codes_t, b.codes_t),
                     (a.scales_t, b.scales_t), (a.amax, b.amax), (a.s_dec, b.s_dec)):
            assert torch.equal(x, y), f"weight operand {which} differs"
    assert torch.equal(YA, YB)
