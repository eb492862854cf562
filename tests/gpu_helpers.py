"""Helpers for the GPU parity tests: device transfer of oracle operands and
the comparison rules.

Comparison rules (the tolerance the hot-path contract states):
* quantiser outputs (codes, MMA-layout scales including padding, amax, s_dec)
  are compared bit for bit;
* a BF16 GEMM output D against the oracle's FP64 product ref of the
  dequantised operands must satisfy max|D - ref| / max|ref| <= 1e-2 and, per
  element, |D - ref| <= 4 ulp_bf16(ref) + 1e-3 rms(ref), with
  ulp_bf16(v) = 2^(floor(log2|v|) - 7) (2^-133 for v = 0).
"""
import ctypes as C

import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def upload(nv, q: dict):
    """An oracle-quantised operand as a library QTensor (codes/scales/s_dec)."""
    codes = torch.from_numpy(q["codes"].reshape(-1).copy()).cuda()
    scales = torch.from_numpy(q["scales_sw"].copy()).cuda()
    amax = torch.tensor([float(q["amax"])], dtype=torch.float32, device="cuda")
    s_dec = torch.tensor([float(q["s_dec"])], dtype=torch.float32, device="cuda")
    t = nv.QTensor(codes=codes, scales=scales, amax=amax, s_dec=s_dec)
    t.desc.codes, t.desc.scales = codes.data_ptr(), scales.data_ptr()
    t.desc.amax, t.desc.s_dec = amax.data_ptr(), s_dec.data_ptr()
    t.desc.rows, t.desc.cols = q["rows"], q["cols"]
    return t


def assert_quant_equal(q, o: dict, name: str = ""):
    """GPU QTensor vs oracle dict, bit for bit."""
    codes = q.codes.cpu().numpy()
    exp = o["codes"].reshape(-1)
    if not np.array_equal(codes, exp):
        bad = np.nonzero(codes != exp)[0]
        raise AssertionError(f"{name}: {bad.size} code bytes differ, first at {bad[:8]} "
                             f"(gpu {codes[bad[:8]]}, oracle {exp[bad[:8]]})")
    sc = q.scales.cpu().numpy()
    if not np.array_equal(sc, o["scales_sw"]):
        bad = np.nonzero(sc != o["scales_sw"])[0]
        raise AssertionError(f"{name}: {bad.size} scale bytes differ, first at {bad[:8]} "
                             f"(gpu {sc[bad[:8]]}, oracle {o['scales_sw'][bad[:8]]})")
    assert q.amax.cpu().numpy()[0].view(np.uint32) == np.float32(o["amax"]).view(np.uint32), name
    assert q.s_dec.cpu().numpy()[0].view(np.uint32) == np.float32(o["s_dec"]).view(np.uint32), name
    assert (q.rows, q.cols) == (o["rows"], o["cols"]), name
    if "codes_t" in o:
        assert np.array_equal(q.codes_t.cpu().numpy(), o["codes_t"].reshape(-1)), name + " codes_t"
        assert np.array_equal(q.scales_t.cpu().numpy(), o["scales_t_sw"]), name + " scales_t"


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def assert_gemm_close(got: np.ndarray, ref: np.ndarray, name: str = "", rms=None):
    err = np.abs(got - ref)
    rel = err.max() / max(np.abs(ref).max(), 1e-300)
    if rms is None:
        rms = np.sqrt(np.mean(ref ** 2))
    bound = 4 * bf16_ulp(ref) + 1e-3 * rms
    bad = err > bound
    assert rel <= 1e-2, f"{name}: max relative error {rel:.3e} > 1e-2"
    assert not bad.any(), (f"{name}: {int(bad.sum())} elements beyond 4 ulp + 1e-3 rms; worst "
                           f"err {err[bad].max():.3e} at ref {ref[bad][np.argmax(err[bad])]:.3e}")
    return rel


# ---- sampled comparisons at sizes the oracle cannot take whole -------------
# An operand row of a 1x16 or 16x16 quantisation depends only on its own input
# row (ROW_1X16, BLOCK_16X16) or input column (COL_1X16), the tensor amax and,
# for stochastic rounding, its own Philox counters: the oracle quantises
# 128-row slabs of the operand with the tensor amax given and each element's
# SR index taken in the whole operand (sr_index_base), and those slabs must
# equal the GPU's bytes.  The GEMM is then checked on sampled outputs whose
# rows and columns lie in the checked slabs.
def oracle_slabs(orc, x, mode, flags, amax, slabs, seed=0, offset=0):
    """Oracle quantisation of 128-row slabs `slabs` of the operand that
    quantising x [R, C] (bf16 bits or float32) in `mode` gives."""
    R, Cn = x.shape
    _, ocols = orc.out_shape(mode, R, Cn)
    out = []
    for sl in slabs:
        r0 = sl * 128
        xs = np.ascontiguousarray(x[:, r0:r0 + 128] if mode == orc.COL_1X16 else x[r0:r0 + 128])
        out.append(orc.quantize(xs, mode, flags, seed=seed, offset=offset,
                                amax_given=float(amax), sr_index_base=r0 * ocols))
    return out


def oracle_slabs_transposed(orc, w, amax, slabs):
    """Slabs of the transposed view of a 16x16 weight quantisation of w [R, C]:
    operand rows c0 .. c0 + 127 are input columns, quantised from w[:, c0:]."""
    out = []
    for sl in slabs:
        ws = np.ascontiguousarray(w[:, sl * 128:sl * 128 + 128])
        o = orc.quantize(ws, orc.BLOCK_16X16, orc.EMIT_T, amax_given=float(amax))
        out.append({"codes": o["codes_t"], "scales": o["scales_t"], "scales_sw": o["scales_t_sw"],
                    "s_dec": o["s_dec"], "rows": 128, "cols": o["rows"]})
    return out


def assert_slabs_equal(codes, scales_sw, amax, s_dec, oslabs, slabs, name):
    """GPU operand (codes [rows, cols/2] uint8, MMA-layout scales, amax, s_dec
    as numpy) against oracle slabs, bit for bit."""
    ocols = codes.shape[1] * 2
    atom_bytes = ((ocols // 16 + 3) // 4) * 512
    for sl, o in zip(slabs, oslabs):
        if not np.array_equal(codes[sl * 128:sl * 128 + 128], o["codes"]):
            bad = np.argwhere(codes[sl * 128:sl * 128 + 128] != o["codes"])
            raise AssertionError(f"{name}: slab {sl}: {len(bad)} code bytes differ, first {bad[:4]}")
        got = scales_sw[sl * atom_bytes:(sl + 1) * atom_bytes]
        assert np.array_equal(got, o["scales_sw"]), f"{name}: slab {sl}: scale atoms differ"
        assert np.float32(o["s_dec"]).view(np.uint32) == np.float32(s_dec).view(np.uint32), name
        if "amax" in o:
            assert np.float32(o["amax"]).view(np.uint32) == np.float32(amax).view(np.uint32), name


def compact_operand(oslabs):
    """The oracle slabs as one operand dict of their rows (row-major scales)."""
    return {"codes": np.ascontiguousarray(np.concatenate([o["codes"] for o in oslabs])),
            "scales": np.ascontiguousarray(np.concatenate([o["scales"] for o in oslabs])),
            "s_dec": oslabs[0]["s_dec"], "rows": 128 * len(oslabs), "cols": oslabs[0]["cols"]}


def sampled_positions(a_slabs, b_slabs, n=4096, seed=11):
    """(local m, local n, global m, global n): every output of the first
    slab pair and of the last slab pair, plus n random outputs over all the
    slabs' rows and columns."""
    rng = np.random.Generator(np.random.PCG64(seed))
    na, nb = 128 * len(a_slabs), 128 * len(b_slabs)
    g0 = np.meshgrid(np.arange(128), np.arange(128), indexing="ij")
    lm = np.concatenate([g0[0].ravel(), na - 128 + g0[0].ravel(), rng.integers(0, na, n)])
    ln = np.concatenate([g0[1].ravel(), nb - 128 + g0[1].ravel(), rng.integers(0, nb, n)])
    to_g = lambda loc, slabs: np.asarray(slabs)[loc // 128] * 128 + loc % 128  # noqa: E731
    return lm, ln, to_g(lm, a_slabs), to_g(ln, b_slabs)
