"""The seeded input generators: determinism and distribution -- CPU only."""
import numpy as np

from nvfp4_block_scaled_03_gb300 import synthetic as syn


def test_deterministic_and_seed_dependent():
    a = syn.activations((64, 256), seed=1)
    assert np.array_equal(a, syn.activations((64, 256), seed=1))
    assert not np.array_equal(a, syn.activations((64, 256), seed=2))


def test_distributions():
    x = syn.bf16_bits_to_f32(syn.activations((512, 2048), seed=1)).astype(np.float64)
    big = np.abs(x) > 8
    assert 0.5e-3 < big.mean() < 1.5e-3              # x50 outliers at rate 1e-3
    assert abs(x[~big].std() - 1.0) < 0.02
    w = syn.bf16_bits_to_f32(syn.weights((512, 512))).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.001 and abs(w.mean()) < 0.001
    d = syn.bf16_bits_to_f32(syn.gradients((512, 512))).astype(np.float64)
    assert abs(d.std() - 1e-3) < 5e-5
    wm = syn.weights((64, 64), master_fp32=True)
    assert wm.dtype == np.float32


def test_bf16_rounding_is_nearest_even():
    v = np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5], np.float32)
    b = syn.f32_to_bf16_bits(v)
    assert list(syn.bf16_bits_to_f32(b)) == [1.0, 1.0 + 2**-6, 1.0, -2.5]
