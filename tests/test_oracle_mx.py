"""Pins of the oracle's MX comparison formats (MXFP4: E2M1 elements, MXFP8:
E4M3 elements; 32-element blocks with power-of-two E8M0 scales, per the
"NVFP4 pretraining recipe" page's comparison of NVFP4 with MXFP4 and the OCP
Microscaling conversion it links).  Checked against closed forms, an
exhaustive nearest-value search, exact round trips and the page's stated
ordering of the formats' errors -- not against the oracle's own formula."""
import math

import numpy as np
import pytest

from nvfp4_block_scaled_03_gb300 import synthetic as syn

pytestmark = pytest.mark.filterwarnings("ignore")

MXFP4, MXFP8 = 0, 1   # the oracle's format codes (checked below)
EMAX = {MXFP4: 2, MXFP8: 8}


def test_format_codes(orc):
    assert (orc.MXFP4, orc.MXFP8) == (MXFP4, MXFP8)


def _values(orc, fmt):
    """Decoded value of every element code (from the format tables)."""
    if fmt == orc.MXFP4:
        return np.array([orc.e2m1_value(c) for c in range(16)])
    return np.array([orc.e4m3_value(c) for c in range(256)])


@pytest.mark.parametrize("fmt", [MXFP4, MXFP8])
def test_e8m0_scale_closed_forms(orc, fmt):
    e = EMAX[fmt]
    for k in range(-60, 61):
        p = math.ldexp(1.0, k)
        # amax exactly 2^k: shared exponent k - emax
        assert orc.e8m0_scale(p, fmt) == k - e + 127
        # anything in [2^k, 2^(k+1)) shares it; just below 2^k drops by one
        assert orc.e8m0_scale(p * 1.75, fmt) == k - e + 127
        assert orc.e8m0_scale(float(np.nextafter(np.float32(p), np.float32(0))), fmt) \
            == k - 1 - e + 127
    assert orc.e8m0_scale(0.0, fmt) == 0
    assert orc.e8m0_scale(math.ldexp(1.0, -140), fmt) == 0          # clamped at -127
    assert orc.e8m0_scale(float(np.finfo(np.float32).max), fmt) == 127 - e + 127
    assert orc.e8m0_scale(float("inf"), fmt) == 0xFF
    assert orc.e8m0_scale(float("nan"), fmt) == 0xFF


def test_e8m0_values(orc):
    for b in range(255):
        assert orc.e8m0_value(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(orc.e8m0_value(0xFF))


def _nearest_code(v, scale, vals):
    """Exhaustive search: the code whose value (times the block scale) is
    nearest to v; ties to the code with an even mantissa (low) bit; values
    beyond the largest finite magnitude saturate to it; the sign of v is kept."""
    best, best_d = None, None
    for c, cv in enumerate(vals):
        if not np.isfinite(cv) or (cv != 0 and np.sign(cv) != np.sign(v)):
            continue
        if cv == 0 and (c & (len(vals) >> 1)) != (0 if not np.signbit(v) else len(vals) >> 1):
            continue  # the zero code of v's sign
        d = abs(cv * scale - v)
        if best is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    return best


@pytest.mark.parametrize("fmt", [MXFP4, MXFP8])
def test_elements_are_the_nearest_code(orc, fmt):
    rng = np.random.default_rng(11)
    vals = _values(orc, fmt)
    x = (rng.standard_normal((6, 64)) * np.exp(rng.uniform(-6, 6, (6, 1)))).astype(np.float32)
    x[0, :8] = [0.0, -0.0, 1e-30, -1e-30, 3.0, -3.0, 2.5, 5.0]  # zeros, tiny values, ties
    x[1, 5] = 0.0
    q = orc.mx_quantize(x, orc.MX_ROW, fmt)
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 32):
            blk = x[r, b * 32:(b + 1) * 32].astype(np.float64)
            amax = np.max(np.abs(blk))
            _, ex = math.frexp(amax)               # amax = m 2^ex, m in [0.5, 1)
            shared = max(-127, min(127, ex - 1 - EMAX[fmt]))
            assert q["scales"][r, b] == shared + 127
            scale = math.ldexp(1.0, shared)
            for i, v in enumerate(blk):
                c = b * 32 + i
                got = (q["codes"][r, c // 2] >> (4 * (c & 1))) & 15 if fmt == orc.MXFP4 \
                    else q["codes"][r, c]
                assert got == _nearest_code(v, scale, vals), (r, c, v)


@pytest.mark.parametrize("fmt", [MXFP4, MXFP8])
def test_representable_blocks_round_trip(orc, fmt):
    rng = np.random.default_rng(5)
    vals = _values(orc, fmt)
    finite = vals[np.isfinite(vals)]
    top = np.max(np.abs(finite))
    for k in (-20, -3, 0, 7, 30):
        blk = rng.choice(finite, size=32) * math.ldexp(1.0, k)
        blk[0] = top * math.ldexp(1.0, k)          # block maximum = largest finite value
        x = blk.astype(np.float32)[None, :]
        q = orc.mx_quantize(x, orc.MX_ROW, fmt)
        np.testing.assert_array_equal(orc.mx_dequant(q)[0], blk)


@pytest.mark.parametrize("fmt", [MXFP4, MXFP8])
def test_column_mode_is_row_mode_of_transpose(orc, fmt):
    x = syn.activations((64, 96), seed=3)
    qc = orc.mx_quantize(x, orc.MX_COL, fmt)
    qr = orc.mx_quantize(np.ascontiguousarray(x.T), orc.MX_ROW, fmt)
    np.testing.assert_array_equal(qc["codes"], qr["codes"])
    np.testing.assert_array_equal(qc["scales"], qr["scales"])


def test_bf16_and_fp32_inputs_agree(orc):
    x = syn.activations((32, 128), seed=4)
    xf = orc.bf16_to_f32(x)
    for fmt in (orc.MXFP4, orc.MXFP8):
        a, b = orc.mx_quantize(x, orc.MX_ROW, fmt), orc.mx_quantize(xf, orc.MX_ROW, fmt)
        np.testing.assert_array_equal(a["codes"], b["codes"])
        np.testing.assert_array_equal(a["scales"], b["scales"])


def test_zero_and_nonfinite_blocks(orc):
    x = np.zeros((3, 32), np.float32)
    x[1, :] = -0.0
    x[2, 3] = np.inf
    x[2, 4] = 1.0
    for fmt, neg0 in ((orc.MXFP4, 0x88), (orc.MXFP8, 0x80)):
        q = orc.mx_quantize(x, orc.MX_ROW, fmt)
        assert list(q["scales"][:, 0]) == [0, 0, 0xFF]
        assert not q["codes"][0].any() and not q["codes"][2].any()
        assert (q["codes"][1] == neg0).all()


def test_nvfp4_error_below_mxfp4_on_outlier_data(orc):
    """The page's comparison: 16-element blocks with E4M3 scales (under a
    per-tensor scale) encode the outlier-laden activations with less error
    than MXFP4's 32-element power-of-two blocks; MXFP8 (three mantissa bits)
    stays well below both."""
    x = syn.activations((256, 2048), seed=1)
    ref = orc.bf16_to_f32(x).astype(np.float64)

    def rel_mse(deq):
        return float(np.mean((deq - ref) ** 2) / np.mean(ref ** 2))
    e_nv = rel_mse(orc.dequant(orc.quantize(x, orc.ROW_1X16)))
    e_mx4 = rel_mse(orc.mx_dequant(orc.mx_quantize(x, orc.MX_ROW, orc.MXFP4)))
    e_mx8 = rel_mse(orc.mx_dequant(orc.mx_quantize(x, orc.MX_ROW, orc.MXFP8)))
    assert e_nv < e_mx4
    assert e_mx8 < 0.5 * e_nv
