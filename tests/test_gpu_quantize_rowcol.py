"""GPU parity of the one-read row + column quantiser (nvfp4_quantize_rowcol):
its two operands equal, byte for byte, the two nvfp4_quantize calls it
replaces (codes, MMA-layout scales with their padding, amax, s_dec), and the
oracle's quantisations ("NVFP4 pretraining recipe" page, bullets 1-5)."""
import numpy as np
import pytest

import gpu_helpers as H
from nvfp4_block_scaled_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

# (row flags, column flags): activations (X, H) and gradients (dY, dG, dU),
# with and without the RHT
FORMS = [("", "RHT"), ("SR", "RHT|SR"), ("", ""), ("SR", "SR"), ("SR", "RHT")]


@pytest.fixture(scope="module")
def nv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_03_gb300 import binding
    return binding


def _flags(lib, spec):
    f = 0
    for part in filter(None, spec.split("|")):
        f |= getattr(lib, part)
    return f


def _same(a, b, name):
    for f in ("codes", "scales", "amax", "s_dec"):
        ga, gb = getattr(a, f), getattr(b, f)
        assert ga.numel() == gb.numel() and bool((ga == gb).all()), f"{name}: {f} differ"
    assert (a.rows, a.cols, a.desc.mode) == (b.rows, b.cols, b.desc.mode), name


def _run(nv, x, rs, cs, seed=5, ro=2, co=3):
    import torch
    xt = H.dev_bf16(x)
    rf, cf = _flags(nv, rs), _flags(nv, cs)
    a_plain = torch.zeros(1, dtype=torch.float32, device="cuda")
    a_col = torch.zeros(1, dtype=torch.float32, device="cuda")
    if cf & nv.RHT:
        nv.nvfp4_amax(xt, a_plain, a_col, seed=seed)
    else:
        nv.nvfp4_amax(xt, amax_plain=a_plain, seed=seed)
        a_col.copy_(a_plain)
    row, col = nv.nvfp4_quantize_rowcol(xt, rf, cf, seed=seed, row_offset=ro, col_offset=co,
                                        amax_row=a_plain, amax_col=a_col)
    ref_r = nv.nvfp4_quantize(xt, nv.ROW_1X16, rf, seed=seed, offset=ro)
    ref_c = nv.nvfp4_quantize(xt, nv.COL_1X16, cf, seed=seed, offset=co)
    nv.check_device_errors()
    _same(row, ref_r, f"row {rs}")
    _same(col, ref_c, f"col {cs}")
    return row, col


@pytest.mark.parametrize("rs,cs", FORMS)
@pytest.mark.parametrize("shape,kind", [((128, 256), "x"), ((208, 80), "dy"), ((336, 400), "x"),
                                        ((16, 16), "dy"), ((64, 1040), "x"), ((400, 48), "dy")])
def test_rowcol_matches_two_calls_and_oracle(nv, orc, rs, cs, shape, kind):
    x = syn.activations(shape, seed=1) if kind == "x" else syn.gradients(shape, seed=3)
    row, col = _run(nv, x, rs, cs)
    H.assert_quant_equal(row, orc.quantize(x, orc.ROW_1X16, _flags(orc, rs), seed=5, offset=2),
                         f"row {rs}")
    H.assert_quant_equal(col, orc.quantize(x, orc.COL_1X16, _flags(orc, cs), seed=5, offset=3),
                         f"col {cs}")


@pytest.mark.parametrize("shape,kind,rs,cs", [((8192, 4096), "x", "", "RHT"),
                                              ((8192, 14336), "dy", "SR", "RHT|SR")])
def test_rowcol_llama8b_full(nv, orc, shape, kind, rs, cs):
    """The bench workload's X and dY at full size: equal to the two separate
    calls (themselves checked bit for bit against the oracle at this size)."""
    x = syn.activations(shape, seed=1) if kind == "x" else syn.gradients(shape, seed=3)
    _run(nv, x, rs, cs, seed=0, ro=0, co=1)


def test_rowcol_rejects_bad_arguments(nv):
    import torch
    x = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_quantize_rowcol(torch.zeros(40, 64, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == nv.ERR_SHAPE                      # 40 rows: no whole 16-row blocks
    r, c = nv.alloc_qtensor(64, 64, nv.ROW_1X16), nv.alloc_qtensor(64, 64, nv.COL_1X16)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_quantize_rowcol(x, nv.RHT, 0, row_out=r, col_out=c)   # RHT on the row operand
    assert e.value.status == nv.ERR_INVALID_ARG


@pytest.mark.parametrize("rs,cs", [("", "RHT"), ("SR", "RHT|SR")])
def test_rowcol_strided_input(nv, orc, rs, cs):
    """x is a column slice of a wider tensor (leading dimension 208 > 144
    columns): both operands equal the oracle's quantisation of the slice."""
    import torch
    wide = syn.activations((96, 208), seed=4)
    x = np.ascontiguousarray(wide[:, 32:176])
    xt = H.dev_bf16(wide)[:, 32:176]
    assert xt.stride(0) == 208
    rf, cf = _flags(nv, rs), _flags(nv, cs)
    a_plain = torch.zeros(1, dtype=torch.float32, device="cuda")
    a_col = torch.zeros(1, dtype=torch.float32, device="cuda")
    nv.nvfp4_amax(xt, a_plain, a_col, seed=5)
    row, col = nv.nvfp4_quantize_rowcol(xt, rf, cf, seed=5, row_offset=2, col_offset=3,
                                        amax_row=a_plain, amax_col=a_col)
    nv.check_device_errors()
    H.assert_quant_equal(row, orc.quantize(x, orc.ROW_1X16, _flags(orc, rs), seed=5, offset=2),
                         "row strided")
    H.assert_quant_equal(col, orc.quantize(x, orc.COL_1X16, _flags(orc, cs), seed=5, offset=3),
                         "col strided")
