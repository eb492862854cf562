"""GPU parity of the SwiGLU kernels (nvfp4_swiglu_fwd / _bwd), which also
emit the tensor amaxes of their bf16 outputs for the NVFP4 quantisations
that follow.

Outputs against the oracle's SwiGLU: the kernels evaluate in FP32 with the
CUDA expf and __fdividef (each within 2 FP32 ulp here) and four or five
further FP32 roundings, a relative error below 2^-19 before the one rounding
to bf16; the oracle evaluates in FP64.  The two bf16 results can therefore
differ only where the exact value lies within 2^-19 of a bf16 rounding
boundary, and then by one bf16 ulp: the bound below.

The amaxes: (1) bit for bit equal to nvfp4_amax over the same device output
(itself pinned bit for bit to the oracle's amax in test_gpu_quantize), which
is the contract the fused quantisers rely on; (2) against the oracle's amax
of the oracle's output, within what a one-ulp difference per element can
move it: one bf16 ulp for max |x|; for max |RHT(v)| over 16-value blocks,
(1/4) 16 2^-8 max|v| <= 2^-4 max|RHT(v)| (max|RHT(v)| >= |v|_2 / 4).
"""
import numpy as np
import pytest

import gpu_helpers as H
from nvfp4_block_scaled_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
SEED = 0x5EED


@pytest.fixture(scope="module")
def nv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_03_gb300 import binding
    return binding


def _ulp_bf16(v):
    """Spacing of bf16 values at |v|: 2^(floor(log2|v|) - 7), and 2^-133 among
    the subnormals and at zero."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.maximum(np.where(a > 0, 2.0 ** (e - 7), 0.0), 2.0 ** -133)


def _within_one_ulp(got_t, ref_bits, name):
    got = H.host_f64(got_t)
    ref = syn.bf16_bits_to_f32(ref_bits).astype(np.float64)
    d = np.abs(got - ref)
    bad = np.argwhere(d > _ulp_bf16(ref))
    assert bad.size == 0, f"{name}: {len(bad)} values beyond one bf16 ulp, first {bad[:4].tolist()}"
    return float(np.mean(d > 0))


def _device_amax(nv, t, rht):
    import torch
    p = torch.zeros(1, dtype=torch.float32, device="cuda")
    r = torch.zeros(1, dtype=torch.float32, device="cuda") if rht else None
    nv.nvfp4_amax(t, amax_plain=p, amax_rht=r, seed=SEED)
    return p.item(), (r.item() if rht else p.item())


def _check_amaxes(nv, orc, t_dev, ref_bits, a_row, a_col, rht, name):
    got_row, got_col = a_row.item(), a_col.item()
    want_row, want_col = _device_amax(nv, t_dev, rht)
    assert got_row == want_row, f"{name}: row amax {got_row!r} != nvfp4_amax {want_row!r}"
    assert got_col == want_col, f"{name}: col amax {got_col!r} != nvfp4_amax {want_col!r}"
    o_row = float(orc.amax(ref_bits, orc.COL_1X16))  # max |x| (rows % 16 == 0 for every shape)
    assert abs(got_row - o_row) <= float(_ulp_bf16(np.float64(o_row))), (name, got_row, o_row)
    if rht:
        o_col = float(orc.amax(ref_bits, orc.COL_1X16, orc.RHT, SEED))
        assert abs(got_col - o_col) <= 2.0 ** -4 * o_col, (name, got_col, o_col)


SHAPES = [(16, 8), (48, 136), (64, 256), (272, 520), (128, 1000)]


@pytest.mark.parametrize("rht", [True, False])
@pytest.mark.parametrize("shape", SHAPES)
def test_swiglu_fwd_matches_oracle(nv, orc, shape, rht):
    G = syn.activations(shape, seed=1)
    U = syn.activations(shape, seed=2)
    Hd, a_row, a_col = nv.nvfp4_swiglu_fwd(H.dev_bf16(G), H.dev_bf16(U), rht=rht, seed=SEED)
    nv.check_device_errors()
    ref = orc.swiglu_fwd(G, U)
    frac = _within_one_ulp(Hd, ref, f"H {shape}")
    assert frac < 0.01, f"H {shape}: {frac:.3%} of values off by one ulp"
    _check_amaxes(nv, orc, Hd, ref, a_row, a_col, rht, f"H {shape} rht={rht}")


@pytest.mark.parametrize("rht", [True, False])
@pytest.mark.parametrize("shape", SHAPES)
def test_swiglu_bwd_matches_oracle(nv, orc, shape, rht):
    G = syn.activations(shape, seed=1)
    U = syn.activations(shape, seed=2)
    dH = syn.gradients(shape, seed=3)
    dG, dU, g_row, g_col, u_row, u_col = nv.nvfp4_swiglu_bwd(
        H.dev_bf16(dH), H.dev_bf16(G), H.dev_bf16(U), rht=rht, seed=SEED)
    nv.check_device_errors()
    rg, ru = orc.swiglu_bwd(dH, G, U)
    for t, ref, nm in ((dG, rg, "dG"), (dU, ru, "dU")):
        frac = _within_one_ulp(t, ref, f"{nm} {shape}")
        assert frac < 0.01, f"{nm} {shape}: {frac:.3%} of values off by one ulp"
    _check_amaxes(nv, orc, dG, rg, g_row, g_col, rht, f"dG {shape} rht={rht}")
    _check_amaxes(nv, orc, dU, ru, u_row, u_col, rht, f"dU {shape} rht={rht}")


def test_swiglu_llama8b_intermediate_full_width(nv, orc):
    """The Llama-3-8B MLP intermediate (F = 14336) over 8192 tokens, forward
    and backward with the RHT: every amax bit for bit equal to nvfp4_amax of
    the stored output; outputs on 64 sampled rows within one ulp of the
    oracle's."""
    M, F = 8192, 14336
    G = syn.activations((M, F), seed=1)
    U = syn.activations((M, F), seed=2)
    dH = syn.gradients((M, F), seed=3)
    Gd, Ud, dHd = H.dev_bf16(G), H.dev_bf16(U), H.dev_bf16(dH)
    Hd, h_row, h_col = nv.nvfp4_swiglu_fwd(Gd, Ud, rht=True, seed=SEED)
    dG, dU, g_row, g_col, u_row, u_col = nv.nvfp4_swiglu_bwd(dHd, Gd, Ud, rht=True, seed=SEED)
    nv.check_device_errors()
    for t, a_row, a_col, nm in ((Hd, h_row, h_col, "H"), (dG, g_row, g_col, "dG"),
                                (dU, u_row, u_col, "dU")):
        assert (a_row.item(), a_col.item()) == _device_amax(nv, t, True), nm
    rows = np.unique(np.random.default_rng(4).integers(0, M, 64))
    ref_h = orc.swiglu_fwd(G[rows], U[rows])
    ref_g, ref_u = orc.swiglu_bwd(dH[rows], G[rows], U[rows])
    import torch
    idx = torch.from_numpy(rows).cuda()
    for t, ref, nm in ((Hd, ref_h, "H"), (dG, ref_g, "dG"), (dU, ref_u, "dU")):
        _within_one_ulp(t[idx], ref, f"{nm} sampled rows")


def test_swiglu_rejects_bad_arguments(nv):
    import torch
    x = torch.zeros(40, 64, dtype=torch.bfloat16, device="cuda")   # 40 rows: not a multiple of 16
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_swiglu_fwd(x, x)
    assert e.value.status == nv.ERR_SHAPE
    y = torch.zeros(32, 64, dtype=torch.bfloat16, device="cuda")
    a = torch.zeros(4, dtype=torch.float32, device="cuda")
    ws = torch.zeros(nv.lib.nvfp4_swiglu_workspace_bytes(), dtype=torch.uint8, device="cuda")
    p = y.data_ptr()
    st = nv.lib.nvfp4_swiglu_fwd(p, p, p, 32, 64, 0x80, 0, a.data_ptr(), a.data_ptr(),
                                 ws.data_ptr(), ws.numel(), None)
    assert st == nv.ERR_INVALID_ARG                                 # unknown flag bit
    st = nv.lib.nvfp4_swiglu_bwd(p, p, p, p, p, 32, 64, 0, 0, *([a.data_ptr()] * 4),
                                 ws.data_ptr(), ws.numel() - 16, None)
    assert st == nv.ERR_WORKSPACE                                   # workspace too small
    st = nv.lib.nvfp4_swiglu_fwd(p, p, None, 32, 64, 0, 0, a.data_ptr(), a.data_ptr(),
                                 ws.data_ptr(), ws.numel(), None)
    assert st == nv.ERR_INVALID_ARG                                 # NULL output
    nv.check_device_errors()
