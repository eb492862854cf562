"""Seeded synthetic inputs for the NVFP4 linear layer (shared by tests, bench
and the CPU oracle; holds none of the quantisation or GEMM arithmetic).

Recipe (the pages name no dataset for this path; the Llama-3 MaxText runs of
the "Performance results" section supply only the shapes):

* generator: ``numpy.random.Generator(PCG64(seed))``, values drawn in float32;
* activations X ~ N(0, 1), each entry independently multiplied by 50 with
  probability 1e-3 (the outliers the recipe's RHT and 1x16 blocks address);
* weights W ~ N(0, 0.02) (bf16, or the FP32 master copy);
* upstream gradients dY ~ N(0, 1e-3);
* bf16 tensors are the float32 draws rounded to nearest-even bf16, returned as
  uint16 bit patterns (numpy has no bf16 dtype).

Default seeds: X=1, W=2, dY=3, Wg/Wu/Wd=4/5/6, the SR/RHT seed is 0.
"""
from __future__ import annotations

import numpy as np

SEED_X, SEED_W, SEED_DY = 1, 2, 3
SEED_WG, SEED_WU, SEED_WD = 4, 5, 6
OUTLIER_RATE, OUTLIER_MULT = 1e-3, 50.0

_CHUNK = 1 << 24


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_f32(shape, seed: int, sigma: float, outliers: bool) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if sigma != 1.0:
            v *= np.float32(sigma)
        if outliers:
            mask = rng.random(e - s, dtype=np.float32) < np.float32(OUTLIER_RATE)
            v[mask] *= np.float32(OUTLIER_MULT)
        out[s:e] = v
    return out.reshape(shape)


def activations(shape, seed: int = SEED_X, outliers: bool = True) -> np.ndarray:
    """X ~ N(0,1) with x50 outliers at rate 1e-3, as bf16 bits."""
    return f32_to_bf16_bits(_normal_f32(shape, seed, 1.0, outliers))


def weights(shape, seed: int = SEED_W, master_fp32: bool = False) -> np.ndarray:
    """W ~ N(0, 0.02): bf16 bits, or the float32 master copy."""
    w = _normal_f32(shape, seed, 0.02, False)
    return w if master_fp32 else f32_to_bf16_bits(w)


def gradients(shape, seed: int = SEED_DY) -> np.ndarray:
    """dY ~ N(0, 1e-3) as bf16 bits."""
    return f32_to_bf16_bits(_normal_f32(shape, seed, 1e-3, False))


def linear_layer(M: int, K: int, N: int):
    """(X [M,K], W [N,K], dY [M,N]) for one linear layer, bf16 bits."""
    return activations((M, K)), weights((N, K)), gradients((M, N))
