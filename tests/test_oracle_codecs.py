"""Pins for the oracle's E2M1 / E4M3 codecs (CPU only).

Every check compares the oracle with something other than itself: the OCP
format table (golden fixture), torch's float8_e4m3fn and ml_dtypes'
float4_e2m1fn / float8_e4m3fn conversions (library routines), and an exact
rational brute force written here in Python.
"""
import math
import pathlib
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = pathlib.Path(__file__).parent / "golden" / "e2m1_e4m3_formats.txt"


def _golden():
    rows = []
    for line in GOLDEN.read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        fmt, code, val = line.split()
        rows.append((fmt, int(code, 0), float(val)))
    return rows


def _same(a, b):
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1, a) == math.copysign(1, b)


def test_decode_matches_ocp_table(oracle):
    for fmt, code, val in _golden():
        got = oracle.e2m1_value(code) if fmt == "e2m1" else oracle.e4m3_value(code)
        assert _same(got, val), (fmt, hex(code), got, val)


def test_e4m3_decode_all_codes_vs_torch(oracle):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().tolist()
    for c in range(256):
        assert _same(oracle.e4m3_value(c), ref[c]), hex(c)


def test_e2m1_decode_all_codes_vs_ml_dtypes(oracle):
    mld = pytest.importorskip("ml_dtypes")
    ref = np.arange(16, dtype=np.uint8).view(mld.float4_e2m1fn).astype(np.float64)
    for c in range(16):
        assert _same(oracle.e2m1_value(c), float(ref[c])), c


@pytest.mark.parametrize("bit_level", [False, True])
def test_exhaustive_round_trip(oracle, bit_level):
    enc2 = oracle.e2m1_encode_bits if bit_level else oracle.e2m1_encode
    enc8 = oracle.e4m3_encode_bits if bit_level else oracle.e4m3_encode
    for c in range(16):
        assert enc2(oracle.e2m1_value(c)) == c
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(v):
            assert enc8(v) & 0x7F == 0x7F          # NaN maps to NaN
        else:
            assert enc8(v) == c, hex(c)             # includes -0 -> 0x80


def _e2m1_grid():
    return [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2),
            Fraction(3), Fraction(4), Fraction(6)]


def _e4m3_grid():
    g = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        g.append(Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7))
    return g


def _rational_encode(x: float, grid, sign_bit, sat):
    """Exact brute force in rationals: nearest grid value, ties to even code."""
    sign = sign_bit if math.copysign(1.0, x) < 0 else 0
    a = abs(Fraction(x))
    if a > grid[-1]:
        return sign | (len(grid) - 1)
    best = min(range(len(grid)), key=lambda c: (abs(grid[c] - a), c & 1))
    return sign | best


def _tricky_inputs(grid):
    """Grid points, midpoints and their fp32 neighbours, both signs."""
    vals = set()
    pts = [float(g) for g in grid] + [float((grid[i] + grid[i + 1]) / 2)
                                     for i in range(len(grid) - 1)]
    pts += [float(grid[-1]) * 1.03, float(grid[-1]) * 2, 1e30]
    for p in pts:
        f = np.float32(p)
        for k in (-2, -1, 0, 1, 2):
            v = f
            step = np.float32(np.inf) if k > 0 else np.float32(-np.inf)
            for _ in range(abs(k)):
                v = np.nextafter(v, step)
            vals.add(float(v))
            vals.add(-float(v))
    return sorted(vals)


def test_e2m1_encode_vs_exact_rationals(oracle):
    grid = _e2m1_grid()
    for x in _tricky_inputs(grid):
        want = _rational_encode(x, grid, 0x8, True)
        assert oracle.e2m1_encode(x) == want, x
        assert oracle.e2m1_encode_bits(x) == want, x


def test_e4m3_encode_vs_exact_rationals(oracle):
    grid = _e4m3_grid()
    for x in _tricky_inputs(grid):
        want = _rational_encode(x, grid, 0x80, True)
        assert oracle.e4m3_encode(x) == want, x
        assert oracle.e4m3_encode_bits(x) == want, x


def test_documented_e2m1_ties(oracle):
    # ties go to the even code: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2,
    # 3.5->4, 5->4; above 6 saturates; the sign of a value rounding to 0 is kept.
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 7.0: 7,
             1e9: 7, float("inf"): 7, -0.2: 0x8, -0.0: 0x8, -5.0: 0xE}
    for x, c in cases.items():
        assert oracle.e2m1_encode(x) == c, x
        assert oracle.e2m1_encode_bits(x) == c, x


def _random_f32(n, seed):
    rng = np.random.default_rng(seed)
    # random bit patterns (all exponents) plus values concentrated near the
    # formats' ranges
    a = rng.integers(0, 2**32, size=n // 2, dtype=np.uint64).astype(np.uint32).view(np.float32)
    b = (rng.standard_normal(n - n // 2) * np.exp2(rng.uniform(-14, 10, n - n // 2)))
    x = np.concatenate([a, b.astype(np.float32)])
    return x[~np.isnan(x)]


def test_bit_level_equals_brute_force_random(oracle):
    x = _random_f32(10_000_000, 1)
    assert np.array_equal(oracle.e2m1_encode_array(x, False), oracle.e2m1_encode_array(x, True))
    assert np.array_equal(oracle.e4m3_encode_array(x, False), oracle.e4m3_encode_array(x, True))


def test_e2m1_encode_vs_ml_dtypes(oracle):
    mld = pytest.importorskip("ml_dtypes")
    x = _random_f32(2_000_000, 2)
    x = np.concatenate([x, np.array(_tricky_inputs(_e2m1_grid()), np.float32)])
    x = x[np.isfinite(x)]
    ref = x.astype(mld.float4_e2m1fn).view(np.uint8) & 0xF
    # ml_dtypes saturates finite overflow to +-6 for this format as well
    assert np.array_equal(oracle.e2m1_encode_array(x, False), ref)


def test_e4m3_encode_vs_torch_float8(oracle):
    # torch's float -> float8_e4m3fn rounds to nearest even; it does not
    # saturate (|x| >= 464 gives NaN), so compare on |x| < 464 and check the
    # saturated region separately.
    x = _random_f32(2_000_000, 3)
    x = np.concatenate([x, np.array(_tricky_inputs(_e4m3_grid()), np.float32)])
    x = x[np.isfinite(x)]
    inside = np.abs(x) < 464
    ref = torch.from_numpy(x[inside]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_array(x, False)
    assert np.array_equal(got[inside], ref)
    sat = got[~inside]
    assert np.all((sat & 0x7F) == 0x7E)
