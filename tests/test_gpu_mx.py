"""GPU parity of the MX comparison quantisers (MXFP4, MXFP8: 32-element
blocks, E8M0 scales) against the CPU oracle: codes and scales bit for bit."""
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


def _check(nv, orc, x_bits_or_f32, mode, fmt, name):
    x = x_bits_or_f32
    dev = H.dev_bf16(x) if x.dtype == np.uint16 else H.dev_f32(x)
    codes, scales = nv.nvfp4_mx_quantize(dev, mode, fmt)
    nv.check_device_errors()
    o = orc.mx_quantize(x, mode, fmt)
    got_c, got_s = codes.cpu().numpy(), scales.cpu().numpy()
    assert got_s.shape == o["scales"].shape and got_c.shape == o["codes"].shape, name
    bad_s = np.argwhere(got_s != o["scales"])
    assert bad_s.size == 0, f"{name}: {len(bad_s)} scale bytes differ, first {bad_s[:4].tolist()}"
    bad_c = np.argwhere(got_c != o["codes"])
    assert bad_c.size == 0, f"{name}: {len(bad_c)} code bytes differ, first {bad_c[:4].tolist()}"


@pytest.mark.parametrize("fmt", ["MXFP4", "MXFP8"])
@pytest.mark.parametrize("mode,shape", [("ROW", (128, 256)), ("ROW", (100, 96)), ("ROW", (1, 32)),
                                        ("ROW", (333, 1056)), ("COL", (64, 136)),
                                        ("COL", (32, 8)), ("COL", (96, 264)),
                                        ("COL", (320, 1000))])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_mx_quantize_matches_oracle(nv, orc, fmt, mode, shape, dtype):
    x = syn.activations(shape, seed=7)
    if dtype == "fp32":
        x = orc.bf16_to_f32(x) * np.float32(1.0001)  # values bf16 cannot hold
    m = {"ROW": nv.MX_ROW, "COL": nv.MX_COL}[mode]
    f = {"MXFP4": nv.MXFP4, "MXFP8": nv.MXFP8}[fmt]
    _check(nv, orc, np.ascontiguousarray(x), m, f, f"{fmt} {mode} {shape} {dtype}")


@pytest.mark.parametrize("fmt", ["MXFP4", "MXFP8"])
@pytest.mark.parametrize("mode", ["ROW", "COL"])
def test_mx_special_values(nv, orc, fmt, mode):
    """All-zero and negative-zero blocks, blocks holding inf or NaN, values
    that round to zero or saturate, tiny (subnormal) and huge magnitudes."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-30, 30, (64, 1)))).astype(np.float32)
    x[0, :] = 0.0
    x[1, :] = -0.0
    x[2, 5] = np.inf
    x[3, 40] = -np.inf
    x[4, 70] = np.nan
    x[5, :32] = np.float32(1e-42)          # subnormal block
    x[6, :4] = [7.0, 5.0, -2.5, -1e-20]    # saturation, ties, negative tiny
    x[7, 64:96] = np.float32(3.0e38)       # huge
    if mode == "COL":
        x = np.ascontiguousarray(x.T)      # the same blocks along the columns of x^T
    m = {"ROW": nv.MX_ROW, "COL": nv.MX_COL}[mode]
    f = {"MXFP4": nv.MXFP4, "MXFP8": nv.MXFP8}[fmt]
    _check(nv, orc, x, m, f, f"{fmt} {mode} special")


@functools.lru_cache(maxsize=1)
def _x405b():
    return syn.activations((8192, 16384), seed=1)


@pytest.mark.parametrize("fmt", ["MXFP4", "MXFP8"])
@pytest.mark.parametrize("mode", ["ROW", "COL"])
def test_mx_405b_activation_full_size(nv, orc, fmt, mode):
    """The Llama-3.1-405B MLP input X [8192, 16384] in both block directions
    (the FPROP operand and the WGRAD operand), bit for bit."""
    x = _x405b()
    m = {"ROW": nv.MX_ROW, "COL": nv.MX_COL}[mode]
    f = {"MXFP4": nv.MXFP4, "MXFP8": nv.MXFP8}[fmt]
    _check(nv, orc, x, m, f, f"{fmt} {mode} [8192, 16384]")


def test_mx_rejects_bad_arguments(nv):
    import torch
    x = torch.zeros(64, 48, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_mx_quantize(x, nv.MX_ROW, nv.MXFP4)    # 48 columns: not a multiple of 32
    assert e.value.status == nv.ERR_SHAPE
    y = torch.zeros(40, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_mx_quantize(y, nv.MX_COL, nv.MXFP8)    # 40 rows: not a multiple of 32
    assert e.value.status == nv.ERR_SHAPE
    z = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_mx_quantize(z, nv.MX_ROW, 7)
    assert e.value.status == nv.ERR_INVALID_ARG
    nv.check_device_errors()
