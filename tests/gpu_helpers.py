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
