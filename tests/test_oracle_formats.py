"""Pins of the oracle's element formats (E2M1, E4M3, bf16) -- CPU only."""
import math
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _golden(name):
    rows = []
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_e2m1_table_matches_golden(orc):
    for code, val in _golden("e2m1_grid.txt"):
        got = orc.e2m1_value(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e4m3_points_match_golden(orc):
    for val, code in _golden("e4m3_points.txt"):
        assert orc.e4m3_value(int(code, 16)) == float(val)
        assert orc.e4m3_rne_sat(float(val)) == int(code, 16)


def test_e4m3_saturation_and_subnormals(orc):
    assert orc.e4m3_rne_sat(448.0) == 0x7E
    assert orc.e4m3_rne_sat(464.0) == 0x7E      # halfway to 480: saturates
    for t in (449.0, 470.0, 479.0, 480.0, 500.0):  # above the largest finite value
        assert orc.e4m3_rne_sat(t) == 0x7E, t      # saturates, never the NaN code
    assert orc.e4m3_rne_sat(1e30) == 0x7E
    assert orc.e4m3_rne_sat(float("inf")) == 0x7E
    assert orc.e4m3_rne_sat(2.0 ** -9) == 0x01
    assert orc.e4m3_rne_sat(2.0 ** -10) == 0x00  # tie between 0 and 2^-9 -> even (0)
    assert orc.e4m3_rne_sat(1.5 * 2.0 ** -10) == 0x01
    assert orc.e4m3_rne_sat(3 * 2.0 ** -10) == 0x02  # tie between 1 and 2 -> even (2)
    assert math.isnan(orc.e4m3_value(0x7F))
    for c in range(0x7F):                         # every finite code round-trips
        assert orc.e4m3_rne_sat(orc.e4m3_value(c)) == c


def test_e2m1_ties_to_even(orc):
    # (input, expected code): midpoints go to the code with mantissa bit 0
    cases = [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
             (0.2500001, 1), (5.0000005, 7), (6.5, 7), (1e9, 7), (float("inf"), 7),
             (-0.25, 8), (-0.75, 10), (-5.0, 14), (-7.0, 15), (-0.1, 8), (0.0, 0), (-0.0, 8)]
    for y, code in cases:
        assert orc.e2m1_rne(y) == code, (y, code, orc.e2m1_rne(y))


def test_e2m1_e4m3_exhaustive_against_brute_force(tmp_path):
    """Every binary32 pattern through the oracle encoders vs an argmin encoder."""
    exe = str(tmp_path / "exh")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-pthread", "-o", exe,
                           os.path.join(HERE, "pins", "exhaustive_formats.c"),
                           os.path.join(ROOT, "oracle", "nvfp4_oracle.c"), "-lm"])
    out = subprocess.check_output([exe, str(max(1, os.cpu_count() or 1))], text=True)
    res = {l.split()[0]: (int(l.split()[1]), int(l.split()[2])) for l in out.splitlines()}
    assert res["e2m1"][0] == (1 << 32) - 2 * ((1 << 23) - 1)  # all non-NaN patterns
    assert res["e2m1"][1] == 0
    assert res["e4m3"][0] > 1_000_000_000
    assert res["e4m3"][1] == 0


def test_e2m1_sr_rule(orc):
    for code in range(8):                 # grid points never move
        v = orc.e2m1_value(code)
        for r in (0, 1, 2**31, 2**32 - 1):
            assert orc.e2m1_sr(v, r) == code
    # 1.25 sits half way between 1 and 1.5: up iff r < 2^31
    assert orc.e2m1_sr(1.25, 2**31 - 1) == 3
    assert orc.e2m1_sr(1.25, 2**31) == 2
    assert orc.e2m1_sr(7.0, 0) == 7 and orc.e2m1_sr(-7.0, 0) == 15
    assert orc.e2m1_sr(-0.3, 2**32 - 1) == 8   # rounds down to -0


@pytest.mark.parametrize("y", [0.3, 1.1, 2.5, 5.9, -0.7])
def test_e2m1_sr_unbiased(orc, y):
    """Mean of SR draws converges to y (|mean - y| <= 5 sigma / sqrt(n))."""
    rng = np.random.Generator(np.random.PCG64(7))
    n = 1 << 16
    r = rng.integers(0, 2**32, size=n, dtype=np.uint64)
    vals = np.array([orc.e2m1_value(orc.e2m1_sr(y, int(x))) for x in r])
    a = abs(y)
    grid = [0, .5, 1, 1.5, 2, 3, 4, 6]
    lo = max(g for g in grid if g <= a)
    hi = min(g for g in grid if g > a)
    p = (a - lo) / (hi - lo)
    sigma = (hi - lo) * math.sqrt(p * (1 - p))
    assert abs(vals.mean() - y) <= 5 * sigma / math.sqrt(n)


def _bf16_val(bits):
    return float((np.array([bits & 0xFFFF], np.uint16).astype(np.uint32) << 16).view(np.float32)[0])


def test_bf16_from_double_is_nearest_even(orc):
    rng = np.random.Generator(np.random.PCG64(11))
    xs = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                         [1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 0.0, 1e-45]])
    for x in xs:
        b = orc.bf16_from_double(float(x))
        v = _bf16_val(b)
        for nb in (b - 1, b + 1):          # neighbours one bf16 step away
            if nb < 0 or (nb & 0x7F80) == 0x7F80 or ((nb ^ b) & 0x8000):
                continue
            w = _bf16_val(nb)
            d0, d1 = abs(x - v), abs(x - w)
            assert d0 < d1 or (d0 == d1 and (b & 1) == 0), (x, hex(b), hex(nb))


def test_bf16_matches_f32_rounding_for_f32_values(orc):
    from nvfp4_block_scaled_03_gb300.synthetic import f32_to_bf16_bits
    rng = np.random.Generator(np.random.PCG64(12))
    x = (rng.standard_normal(4096) * 3).astype(np.float32)
    got = orc.bf16_round_f64(x.astype(np.float64))
    assert np.array_equal(got, f32_to_bf16_bits(x))
