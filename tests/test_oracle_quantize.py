"""Pins of the oracle quantiser -- CPU only.

Each check compares the oracle with something other than itself: brute-force
argmin encoders over the format value sets, a lossless round trip, the
transpose invariant of 16x16 weight scaling ("NVFP4 pretraining recipe",
bullet 4), an independent reshape formulation of the MMA scale layout, and the
statistical unbiasedness of stochastic rounding (bullet 5).
"""
import numpy as np
import pytest

from nvfp4_block_scaled_03_gb300 import synthetic as syn

GRID = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)
E4M3_POS = np.array([(m * 2.0 ** -9) if e == 0 else (8 + m) * 2.0 ** (e - 10)
                     for e in range(16) for m in range(8)][:127], np.float64)


def bf_e2m1(y):
    """Brute-force E2M1 RNE: argmin over the grid, ties to the even code."""
    y = np.asarray(y, np.float32).astype(np.float64)
    a = np.abs(y)
    d = np.abs(a[..., None] - GRID)
    ties = d == d.min(axis=-1, keepdims=True)
    best = np.where(ties.sum(-1) > 1, np.argmax(ties & ((np.arange(8) & 1) == 0), -1),
                    np.argmin(d, axis=-1))
    best = np.where(a >= 6, 7, best)
    return (best | (np.signbit(y).astype(np.int64) << 3)).astype(np.uint8)


def bf_e4m3(t):
    """Brute-force E4M3FN RNE with saturation (t >= 0)."""
    t = np.asarray(t, np.float32).astype(np.float64)
    d = np.abs(t[..., None] - E4M3_POS)
    ties = d == d.min(axis=-1, keepdims=True)
    best = np.where(ties.sum(-1) > 1, np.argmax(ties & ((np.arange(127) & 1) == 0), -1),
                    np.argmin(d, -1))
    return np.where(t >= 448, 0x7E, best).astype(np.uint8)


def unpack(codes, ncols):
    out = np.empty((codes.shape[0], ncols), np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


def _f32(x):
    return syn.bf16_bits_to_f32(x) if x.dtype == np.uint16 else x.astype(np.float32)


def _brute_quantize_1x16(v):
    """v: float32 [R, C] already in output layout (and transformed)."""
    amax = np.float32(np.abs(v).max())
    s_enc = np.float32(1.0) if amax == 0 else np.float32(np.float32(2688.0) / amax)
    R, C = v.shape
    blocks = v.reshape(R, C // 16, 16)
    a_b = np.abs(blocks).max(axis=-1).astype(np.float32)
    t = (a_b / np.float32(6.0)).astype(np.float32) * s_enc
    sc = bf_e4m3(t.astype(np.float32))
    S = E4M3_POS[sc].astype(np.float32)
    enc = np.where(S == 0, np.float32(0), (s_enc / np.where(S == 0, 1, S)).astype(np.float32))
    y = (blocks * enc[..., None].astype(np.float32)).astype(np.float32).reshape(R, C)
    return bf_e2m1(y), sc, amax, s_enc, y


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("shape", [(32, 64), (16, 256), (48, 16)])
def test_row_quantize_brute_force(orc, dtype, shape):
    x = syn.activations(shape, seed=21)
    if dtype == "fp32":
        x = syn.bf16_bits_to_f32(x) * np.float32(1.37)
    q = orc.quantize(x, orc.ROW_1X16)
    codes, sc, amax, s_enc, _ = _brute_quantize_1x16(_f32(x))
    assert q["amax"] == amax and q["s_enc"] == s_enc
    assert q["s_dec"] == np.float32(np.float32(1.0) / s_enc)
    assert np.array_equal(q["scales"], sc)
    assert np.array_equal(unpack(q["codes"], shape[1]), codes)


def test_col_quantize_is_row_quantize_of_transpose(orc):
    x = syn.activations((64, 48), seed=22)
    qc = orc.quantize(x, orc.COL_1X16)
    qr = orc.quantize(np.ascontiguousarray(x.T), orc.ROW_1X16)
    assert qc["rows"] == 48 and qc["cols"] == 64
    for k in ("codes", "scales", "scales_sw"):
        assert np.array_equal(qc[k], qr[k])


def test_col_rht_brute_force_on_integer_inputs(orc):
    """Integer-valued inputs make the butterfly exact, so the matrix form in
    FP64 gives the same binary32 values; then brute-force encode."""
    rng = np.random.Generator(np.random.PCG64(23))
    x = rng.integers(-40, 40, (64, 32)).astype(np.float32)
    seed = 99
    q = orc.quantize(x, orc.COL_1X16, orc.RHT, seed=seed)
    s = orc.rht_signs(seed).astype(np.float64)
    H = np.array([[(-1) ** bin(i & j).count("1") for j in range(16)] for i in range(16)], float)
    xt = x.T.astype(np.float64)  # [32, 64] output layout
    v = np.empty_like(xt)
    for r in range(xt.shape[0]):
        for b in range(4):
            v[r, b * 16:(b + 1) * 16] = 0.25 * H @ (s * xt[r, b * 16:(b + 1) * 16])
    codes, sc, amax, s_enc, _ = _brute_quantize_1x16(v.astype(np.float32))
    assert q["amax"] == amax
    assert orc.amax(x, orc.COL_1X16, orc.RHT, seed=seed) == amax
    assert np.array_equal(q["scales"], sc)
    assert np.array_equal(unpack(q["codes"], 64), codes)


def test_lossless_round_trip(orc):
    """Inputs built as code * S_b * 2^-p with a +-6 in every block and one block
    at S = 448 dequantise back exactly."""
    rng = np.random.Generator(np.random.PCG64(24))
    R, C, p = 32, 128, 10
    codes = rng.integers(0, 16, (R, C))
    Sb = rng.integers(1, 0x7E, (R, C // 16))
    Sb[0, 0] = 0x7E
    for r in range(R):
        for b in range(C // 16):
            codes[r, b * 16 + rng.integers(0, 16)] = 7 | (rng.integers(0, 2) << 3)
    vals = np.array([orc.e2m1_value(c) for c in range(16)])[codes]
    exact = vals * np.repeat(E4M3_POS[Sb], 16, axis=1) * 2.0 ** -p
    x = exact.astype(np.float32)
    assert np.all(x.astype(np.float64) == exact)
    q = orc.quantize(x, orc.ROW_1X16)
    assert q["s_enc"] == np.float32(2.0 ** p)
    assert np.array_equal(q["scales"], Sb.astype(np.uint8))
    assert np.array_equal(orc.dequant(q), exact)


def test_16x16_one_scale_per_tile_and_transpose_invariant(orc):
    w = syn.weights((64, 96), seed=25, master_fp32=True)
    q = orc.quantize(w, orc.BLOCK_16X16, orc.EMIT_T)
    sc = q["scales"].reshape(4, 16, 6)
    assert np.all(sc == sc[:, :1, :])               # 16 rows of a tile share a scale
    st = q["scales_t"].reshape(6, 16, 4)
    assert np.array_equal(st[:, 0, :], sc[:, 0, :].T)
    # FPROP and DGRAD see identical weight values (bit for bit)
    assert np.array_equal(orc.dequant(q), orc.dequant(orc.transposed_view(q)).T)
    tiles = w.reshape(4, 16, 6, 16).transpose(0, 2, 1, 3).reshape(4, 6, 256)
    s_enc = np.float32(np.float32(2688.0) / np.float32(np.abs(w).max()))
    t = (np.abs(tiles).max(-1).astype(np.float32) / np.float32(6)).astype(np.float32) * s_enc
    assert np.array_equal(sc[:, 0, :], bf_e4m3(t))
    # codes: brute-force encode with the tile's factor
    S = E4M3_POS[np.repeat(np.repeat(sc[:, 0, :], 16, 0), 16, 1)].astype(np.float32)
    enc = (s_enc / S).astype(np.float32)
    assert np.array_equal(unpack(q["codes"], 96), bf_e2m1((w * enc).astype(np.float32)))


def test_swizzle_matches_reshape_formulation(orc):
    """Atom layout as a reshape: row = rb*128 + q*32 + i, col = cb*4 + j stored
    at [rb][cb][i][q][j] (32 lines of 16 bytes: 4 row groups x 4 scales)."""
    x = syn.activations((200, 16 * 10), seed=26)   # ragged rows and scale cols
    q = orc.quantize(x, orc.ROW_1X16)
    R, nsc = q["scales"].shape
    pr, pc = (R + 127) // 128 * 128, (nsc + 3) // 4 * 4
    padded = np.zeros((pr, pc), np.uint8)
    padded[:R, :nsc] = q["scales"]
    exp = padded.reshape(pr // 128, 4, 32, pc // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    assert np.array_equal(q["scales_sw"], exp)


def test_sr_quantize_unbiased_and_deterministic(orc):
    """Constant tensor: SR codes dequantise to x on average; P(up) = frac."""
    R, C = 256, 256
    x = np.full((R, C), 0.37, np.float32)
    x[0, 0] = 6.0
    q = orc.quantize(x, orc.ROW_1X16, orc.SR, seed=5, offset=3)
    body = orc.dequant(q)[1:, :]
    assert np.all(q["scales"][1:] == q["scales"][1, 0])
    n = body.size
    vals = np.unique(body)
    assert len(vals) == 2
    lo, hi = vals
    p = (0.37 - lo) / (hi - lo)
    assert abs((body == hi).mean() - p) <= 5 * np.sqrt(p * (1 - p) / n)
    assert abs(body.mean() - 0.37) <= 5 * (hi - lo) * np.sqrt(p * (1 - p) / n) + 1e-6
    q2 = orc.quantize(x, orc.ROW_1X16, orc.SR, seed=5, offset=3)
    assert np.array_equal(q["codes"], q2["codes"])
    q3 = orc.quantize(x, orc.ROW_1X16, orc.SR, seed=5, offset=4)
    assert not np.array_equal(q["codes"], q3["codes"])


def test_sr_uses_the_philox_word_of_each_element(orc):
    x = syn.gradients((16, 64), seed=27)
    seed, off = 8, 2
    q = orc.quantize(x, orc.COL_1X16, orc.SR, seed=seed, offset=off)
    v = np.ascontiguousarray(syn.bf16_bits_to_f32(x).T)  # output layout [64, 16]
    _, _, _, _, y = _brute_quantize_1x16(v)
    got = unpack(q["codes"], 16)
    for r in range(64):
        for c in range(16):
            w = orc.sr_word(seed, off, r * 16 + c)
            assert got[r, c] == orc.e2m1_sr(float(y[r, c]), w)


def test_zero_tensor_and_amax_given(orc):
    q = orc.quantize(np.zeros((16, 32), np.uint16), orc.ROW_1X16)
    assert q["amax"] == 0 and q["s_enc"] == 1 and q["s_dec"] == 1
    assert not q["codes"].any() and not q["scales"].any() and not q["scales_sw"].any()
    x = syn.activations((16, 32), seed=28)
    big = float(np.abs(syn.bf16_bits_to_f32(x)).max()) * 4
    q = orc.quantize(x, orc.ROW_1X16, amax_given=big)
    assert q["amax"] == np.float32(big)
    assert q["s_enc"] == np.float32(np.float32(2688.0) / np.float32(big))


def test_invalid_arguments_rejected(orc):
    with pytest.raises(ValueError):
        orc.quantize(syn.activations((32, 40)), orc.ROW_1X16)    # 40 % 16 != 0
    with pytest.raises(ValueError):
        orc.quantize(syn.activations((24, 32)), orc.COL_1X16)    # rows % 16
    with pytest.raises(ValueError):
        orc.quantize(syn.activations((32, 32)), orc.BLOCK_16X16, orc.RHT)
    with pytest.raises(ValueError):
        orc.quantize(syn.activations((32, 32)), orc.ROW_1X16, orc.EMIT_T)


def test_sr_window_equals_slab_of_whole(orc):
    """Quantising a window of output rows with sr_index_base = first row x
    output columns reproduces that window of the whole operand's SR codes
    (row and transposing modes), given the whole operand's amax."""
    x = syn.gradients((96, 64), seed=21)
    for mode, flags in ((orc.ROW_1X16, orc.SR), (orc.COL_1X16, orc.SR | orc.RHT)):
        whole = orc.quantize(x, mode, flags, seed=3, offset=5)
        orows, ocols = orc.out_shape(mode, *x.shape)
        r0, r1 = 16, 48
        xs = x[r0:r1] if mode == orc.ROW_1X16 else x[:, r0:r1]
        win = orc.quantize(np.ascontiguousarray(xs), mode, flags, seed=3, offset=5,
                           amax_given=float(whole["amax"]), sr_index_base=r0 * ocols)
        assert np.array_equal(win["codes"], whole["codes"][r0:r1])
        # without the base the window draws other random words
        other = orc.quantize(np.ascontiguousarray(xs), mode, flags, seed=3, offset=5,
                             amax_given=float(whole["amax"]))
        assert not np.array_equal(other["codes"], whole["codes"][r0:r1])
