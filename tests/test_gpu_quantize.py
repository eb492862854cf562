"""GPU parity of the quantisers against the CPU oracle: codes, MMA-layout
scales (with padding), amax and s_dec bit for bit."""
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

# (mode name, flags) in both libraries' terms
MODES = [
    ("ROW", 0), ("ROW", "SR"), ("ROW", "RHT"), ("ROW", "RHT|SR"),
    ("COL", 0), ("COL", "SR"), ("COL", "RHT"), ("COL", "RHT|SR"),
    ("BLK", "EMIT_T"), ("BLK", "SR|EMIT_T"), ("BLK", 0),
]


def _mode(lib, name):
    return {"ROW": lib.ROW_1X16, "COL": lib.COL_1X16, "BLK": lib.BLOCK_16X16}[name]


def _flags(lib, spec):
    if not spec:
        return 0
    f = 0
    for part in spec.split("|"):
        f |= getattr(lib, part)
    return f


def _input(shape, kind, dtype):
    if kind == "x":
        a = syn.activations(shape, seed=1)
    elif kind == "w":
        a = syn.weights(shape, seed=2)
    else:
        a = syn.gradients(shape, seed=3)
    if dtype == "fp32":
        a = syn.bf16_bits_to_f32(a) * np.float32(1.0 + 2.0 ** -12)  # not bf16-representable
    return a


def _run(nv, orc, x, mode_name, spec, seed=7, offset=3):
    xt = H.dev_bf16(x) if x.dtype == np.uint16 else H.dev_f32(x)
    q = nv.nvfp4_quantize(xt, _mode(nv, mode_name), _flags(nv, spec), seed=seed, offset=offset)
    o = orc.quantize(x, _mode(orc, mode_name), _flags(orc, spec), seed=seed, offset=offset)
    H.assert_quant_equal(q, o, f"{mode_name}/{spec}/{x.shape}")


@pytest.mark.parametrize("mode_name,spec", MODES)
@pytest.mark.parametrize("shape,kind", [((128, 256), "x"), ((512, 256), "w"), ((128, 512), "dy"),
                                        ((208, 80), "x"), ((16, 16), "dy"), ((48, 32), "x"),
                                        ((336, 400), "dy")])
def test_quantize_small(nv, orc, mode_name, spec, shape, kind):
    _run(nv, orc, _input(shape, kind, "bf16"), mode_name, spec)


@pytest.mark.parametrize("mode_name,spec", [("ROW", 0), ("COL", "RHT|SR"), ("BLK", "EMIT_T"),
                                            ("BLK", "SR|EMIT_T")])
def test_quantize_fp32_input(nv, orc, mode_name, spec):
    _run(nv, orc, _input((256, 384), "w", "fp32"), mode_name, spec)


def test_quantize_amax_given_and_zero(nv, orc):
    import torch
    x = _input((128, 256), "x", "bf16")
    big = float(np.abs(syn.bf16_bits_to_f32(x)).max()) * 3.0
    q = nv.nvfp4_quantize(H.dev_bf16(x), nv.ROW_1X16, amax=big)
    o = orc.quantize(x, orc.ROW_1X16, amax_given=big)
    H.assert_quant_equal(q, o, "amax_given")
    z = np.zeros((64, 64), np.uint16)
    q = nv.nvfp4_quantize(H.dev_bf16(z), nv.COL_1X16, nv.RHT | nv.SR, seed=1)
    o = orc.quantize(z, orc.COL_1X16, orc.RHT | orc.SR, seed=1)
    H.assert_quant_equal(q, o, "zeros")
    assert float(q.s_dec.cpu()[0]) == 1.0
    torch.cuda.synchronize()


def test_quantize_rejects_bad_shapes(nv):
    import torch
    x = torch.zeros(40, 24, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_quantize(x, nv.ROW_1X16)            # 24 % 16
    assert e.value.status == nv.ERR_SHAPE
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_quantize(x, nv.COL_1X16)            # 40 % 16
    assert e.value.status == nv.ERR_SHAPE
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_quantize(torch.zeros(32, 32, dtype=torch.bfloat16, device="cuda"),
                          nv.BLOCK_16X16, nv.RHT)
    assert e.value.status == nv.ERR_INVALID_ARG


@pytest.mark.parametrize("shape,kind,mode_name,spec", [
    ((8192, 4096), "x", "ROW", 0),             # FPROP X
    ((8192, 4096), "x", "COL", "RHT"),         # WGRAD X^T
    ((14336, 4096), "w", "BLK", "EMIT_T"),     # W for FPROP and DGRAD
    ((8192, 14336), "dy", "ROW", "SR"),        # DGRAD dY
    ((8192, 14336), "dy", "COL", "RHT|SR"),    # WGRAD dY^T
])
def test_quantize_llama8b_full(nv, orc, shape, kind, mode_name, spec):
    """The bench workload's quantiser calls at full size, every byte compared."""
    _run(nv, orc, _input(shape, kind, "bf16"), mode_name, spec, seed=0, offset=1)


@functools.lru_cache(maxsize=2)
def _activations_32k(R, Cn):
    return syn.activations((R, Cn), seed=5)


@pytest.mark.parametrize("R,Cn", [(32768, 14336), (32768, 4096)])
@pytest.mark.parametrize("mode_name,spec", [("ROW", 0), ("ROW", "SR"), ("COL", "RHT|SR"),
                                            ("BLK", "EMIT_T")])
def test_quantize_32k_tokens_sampled(nv, orc, R, Cn, mode_name, spec):
    """The quantiser-only sweep's 32k-token shapes: the GPU quantises the whole
    tensor; the oracle computes the tensor amax itself and quantises sampled
    128-row output slabs with it (each element's stochastic-rounding index
    taken in the whole output), compared bit for bit: codes, the slab's scale
    atoms and, for 16x16, its columns of the transposed codes."""
    x = _activations_32k(R, Cn)
    mode, flags = _mode(orc, mode_name), _flags(orc, spec)
    q = nv.nvfp4_quantize(H.dev_bf16(x), _mode(nv, mode_name), _flags(nv, spec), seed=2, offset=4)
    amax = orc.amax(x, mode, flags & orc.RHT, seed=2)
    assert q.amax.cpu().numpy()[0] == amax
    orows, ocols = orc.out_shape(mode, R, Cn)
    codes = q.codes.cpu().numpy().reshape(orows, ocols // 2)
    scales = q.scales.cpu().numpy()
    codes_t = q.codes_t.cpu().numpy().reshape(ocols, orows // 2) if flags & orc.EMIT_T else None
    atom_bytes = ((ocols // 16 + 3) // 4) * 512
    rng = np.random.Generator(np.random.PCG64(9))
    for rb in sorted(set(rng.integers(0, orows // 128, 3).tolist()) | {0, orows // 128 - 1}):
        sl = slice(rb * 128, rb * 128 + 128)
        xs = np.ascontiguousarray(x[:, sl] if mode == orc.COL_1X16 else x[sl])
        o = orc.quantize(xs, mode, flags, seed=2, offset=4, amax_given=float(amax),
                         sr_index_base=rb * 128 * ocols)
        assert np.array_equal(scales[rb * atom_bytes:(rb + 1) * atom_bytes], o["scales_sw"]), rb
        assert np.array_equal(codes[sl], o["codes"]), rb
        if codes_t is not None:
            assert np.array_equal(codes_t[:, rb * 64:(rb + 1) * 64], o["codes_t"]), rb


@pytest.mark.parametrize("shape,kind,dtype", [((336, 400), "dy", "bf16"), ((128, 256), "x", "fp32"),
                                              ((8192, 14336), "dy", "bf16")])
def test_amax_one_read_matches_oracle_and_quantise(nv, orc, shape, kind, dtype):
    """nvfp4_amax: max |x| and the column-RHT amax from one read equal the
    oracle's; quantising with them given reproduces the self-computed codes."""
    import torch
    x = _input(shape, kind, dtype)
    xt = H.dev_bf16(x) if x.dtype == np.uint16 else H.dev_f32(x)
    seed = 5
    a_plain = torch.zeros(1, dtype=torch.float32, device="cuda")
    a_rht = torch.zeros(1, dtype=torch.float32, device="cuda")
    nv.nvfp4_amax(xt, a_plain, a_rht, seed=seed)
    assert float(a_plain.cpu()[0]) == orc.amax(x, orc.ROW_1X16, 0, seed=seed)
    assert float(a_rht.cpu()[0]) == orc.amax(x, orc.COL_1X16, orc.RHT, seed=seed)
    # each output alone takes another kernel path; same values
    b_plain = torch.zeros(1, dtype=torch.float32, device="cuda")
    b_rht = torch.zeros(1, dtype=torch.float32, device="cuda")
    nv.nvfp4_amax(xt, amax_plain=b_plain, seed=seed)
    nv.nvfp4_amax(xt, amax_rht=b_rht, seed=seed)
    assert float(b_plain.cpu()[0]) == float(a_plain.cpu()[0])
    assert float(b_rht.cpu()[0]) == float(a_rht.cpu()[0])
    for mode, flags, a in ((nv.ROW_1X16, nv.SR, a_plain), (nv.COL_1X16, nv.RHT | nv.SR, a_rht)):
        ref = nv.nvfp4_quantize(xt, mode, flags, seed=seed, offset=2)
        q = nv.alloc_qtensor(shape[0], shape[1], mode, flags)
        q.amax.copy_(a)
        nv.nvfp4_quantize(xt, mode, flags | nv.AMAX_GIVEN, seed=seed, offset=2, out=q)
        for name in ("codes", "scales", "amax", "s_dec"):
            assert torch.equal(getattr(q, name), getattr(ref, name)), name
    if shape[0] * shape[1] <= 1 << 20:  # and against the oracle directly
        q = nv.alloc_qtensor(shape[0], shape[1], nv.COL_1X16, nv.RHT)
        q.amax.copy_(a_rht)
        nv.nvfp4_quantize(xt, nv.COL_1X16, nv.RHT | nv.AMAX_GIVEN, seed=seed, out=q)
        H.assert_quant_equal(q, orc.quantize(x, orc.COL_1X16, orc.RHT, seed=seed), "rht given")


def test_amax_rejects_bad_arguments(nv):
    import torch
    x = torch.zeros(40, 32, dtype=torch.bfloat16, device="cuda")
    a = torch.zeros(1, dtype=torch.float32, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_amax(x, amax_rht=a)                 # 40 % 16: no whole RHT blocks
    assert e.value.status == nv.ERR_SHAPE
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_amax(x)                             # no output asked for
    assert e.value.status == nv.ERR_INVALID_ARG
    nv.nvfp4_amax(x, amax_plain=a)                   # the plain amax has no row constraint
    assert float(a.cpu()[0]) == 0.0


def _edge_rows(C):
    """bf16 [64, C] whose 16-element row blocks (and, because the 16 rows of
    each 16-row strip repeat one pattern, whose 16x16 tiles) reach the rarely
    taken branches of the quantiser: with the tensor amax given as 2688
    (s_enc = 1, so a block's scale is E4M3(max/6)) --
      T        every E2M1 tie (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, signed)
               under a block maximum of 6 (scale 1, encode factor 1);
      Z        -0 and negative values that round to zero in a non-zero block;
      T * 2^-8 a subnormal E4M3 scale (2^-8);
      T * 2^-9 the smallest subnormal scale (2^-9);
      T * 2^-10 a scale exactly halfway to zero (rounds to 0: codes 0 / -0);
      T * 2^-12 a scale far below (0);
      T * 16   a large normal scale;
    and a Gaussian strip.  With the amax given as 26.88 (s_enc = 100, below
    the true maximum) block scales clamp at 448 and elements saturate at 6."""
    T = np.array([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -.25, -.75, -1.25, -1.75, -2.5, -3.5,
                  -5, .5], np.float32)
    Z = np.array([6, -0.0, -0.1, -0.2, -0.24, 0.1, 0.2, -0.0, 0.0, -6, -0.3, 0.3, -0.26, 0.26,
                  -0.01, -0.0], np.float32)
    pats = [T, Z, T * 2.0 ** -8, T * 2.0 ** -9, T * 2.0 ** -10, T * 2.0 ** -12, T * 16,
            Z * 2.0 ** -8]
    rng = np.random.Generator(np.random.PCG64(17))
    x = np.empty((64, C), np.float32)
    for r in range(64):
        for j in range(C // 16):
            k = ((r // 16) * (C // 16) + j) % (len(pats) + 1)
            x[r, 16 * j:16 * j + 16] = (pats[k] if k < len(pats)
                                        else rng.standard_normal(16).astype(np.float32) * 3)
    return syn.f32_to_bf16_bits(x)


@pytest.mark.parametrize("amax", [2688.0, 26.88, None])
@pytest.mark.parametrize("mode_name,spec", MODES)
def test_quantize_edge_cases(nv, orc, mode_name, spec, amax):
    """Ties, signed zeros, subnormal and zero block scales, saturation: codes,
    scales, amax and s_dec bit for bit against the oracle, in every mode (the
    column mode reads the transpose, so its 16-row blocks hold the patterns)."""
    x = _edge_rows(256)
    if mode_name == "COL":
        x = np.ascontiguousarray(x.T)
    mode, flags = _mode(nv, mode_name), _flags(nv, spec)
    q = nv.nvfp4_quantize(H.dev_bf16(x), mode, flags, seed=9, offset=1, amax=amax)
    o = orc.quantize(x, _mode(orc, mode_name), _flags(orc, spec), seed=9, offset=1,
                     amax_given=amax)
    H.assert_quant_equal(q, o, f"edge {mode_name}/{spec}/amax={amax}")
    if amax == 2688.0 and not (flags & nv.RHT):
        codes = q.codes.cpu().numpy()
        # the patterns reach what they are there for: negative zeros (code 8)
        # and, in the blocks under a zero scale, all-zero magnitudes
        assert ((codes & 0xF) == 8).any() or ((codes >> 4) == 8).any()
        assert (q.scales.cpu().numpy() == 0).any()
