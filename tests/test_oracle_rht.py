"""Pins of the oracle's 16-point random Hadamard transform -- CPU only.

Closed forms: the Sylvester Hadamard H16[i][j] = (-1)^popcount(i & j),
H16 H16^T = 16 I, (1/4) H16 D orthogonal, and the cancellation that lets the
WGRAD GEMM use transformed operands without an inverse ("NVFP4 pretraining
recipe", bullet 3: RHT on the WGRAD inputs only).
"""
import numpy as np


def _sylvester():
    return np.array([[(-1) ** bin(i & j).count("1") for j in range(16)] for i in range(16)],
                    dtype=np.float64)


def test_butterfly_builds_the_sylvester_matrix(orc):
    ones = np.ones(16, np.float32)
    cols = np.stack([orc.rht16(np.eye(16, dtype=np.float32)[j], ones) for j in range(16)], axis=1)
    H = 4.0 * cols.astype(np.float64)
    assert np.array_equal(H, _sylvester())
    assert np.array_equal(H @ H.T, 16.0 * np.eye(16))


def test_signs_are_applied_before_the_transform(orc):
    rng = np.random.Generator(np.random.PCG64(3))
    s = np.where(rng.random(16) < 0.5, -1.0, 1.0).astype(np.float32)
    v = rng.integers(-50, 50, 16).astype(np.float32)
    got = orc.rht16(v, s).astype(np.float64)
    exp = 0.25 * _sylvester() @ (s.astype(np.float64) * v.astype(np.float64))
    assert np.array_equal(got, exp)  # integer inputs: every step is exact


def test_butterfly_rounding_is_small_on_random_floats(orc):
    rng = np.random.Generator(np.random.PCG64(4))
    s = orc.rht_signs(0)
    for _ in range(200):
        v = rng.standard_normal(16).astype(np.float32)
        got = orc.rht16(v, s).astype(np.float64)
        exp = 0.25 * _sylvester() @ (s.astype(np.float64) * v.astype(np.float64))
        assert np.all(np.abs(got - exp) <= 4 * 2.0 ** -24 * np.abs(v).sum())
        assert abs(np.linalg.norm(got) - np.linalg.norm(v.astype(np.float64))) <= \
            1e-6 * np.linalg.norm(v)


def test_rht_cancels_in_the_wgrad_product(orc):
    """(RHT A)^T (RHT B) == A^T B along the token dim, same signs for both."""
    rng = np.random.Generator(np.random.PCG64(5))
    M, p, q = 64, 5, 7
    A = rng.integers(-8, 8, (M, p)).astype(np.float32)
    B = rng.integers(-8, 8, (M, q)).astype(np.float32)

    def rht_cols(X, s):
        Y = np.empty_like(X)
        for c in range(X.shape[1]):
            for b in range(M // 16):
                Y[b * 16:(b + 1) * 16, c] = orc.rht16(X[b * 16:(b + 1) * 16, c], s)
        return Y.astype(np.float64)

    s = orc.rht_signs(123)
    rhs = A.astype(np.float64).T @ B.astype(np.float64)
    assert np.array_equal(rht_cols(A, s).T @ rht_cols(B, s), rhs)
    # with different signs on the two sides the product no longer cancels
    assert not np.allclose(rht_cols(A, s).T @ rht_cols(B, orc.rht_signs(124)), rhs)
