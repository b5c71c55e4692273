"""Pins for the oracle's single-precision helpers, against exact arithmetic."""
import math
from fractions import Fraction

import numpy as np

from oracle.fp32 import F32, fma32, weight


def round_f32_exact(fr: Fraction) -> np.float32:
    """Nearest-even float32 of an exact rational (normal range)."""
    if fr == 0:
        return F32(0.0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    m = a * Fraction(2) ** (23 - e)          # in [2^23, 2^24)
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return F32(sign * n * 2.0 ** (e - 23))


def exact_fma(a, b, c):
    return round_f32_exact(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def test_fma32_matches_exact_rounding_random():
    rng = np.random.default_rng(1)
    n = 4000
    a = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(F32)
    b = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(F32)
    c = (rng.standard_normal(n) * np.exp2(rng.integers(-40, 40, n))).astype(F32)
    got = fma32(a, b, c)
    want = np.array([exact_fma(x, y, z) for x, y, z in zip(a, b, c)], dtype=F32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_fma32_double_rounding_midpoints():
    # 2^36 + 1 = 4097 * 16773121 and 2^36 - 1 = (2^18 - 1)(2^18 + 1): products just off a
    # float32 midpoint by 2^-60, which a plain double sum rounds onto the midpoint.
    up = (F32(4097 * 2.0 ** -12), F32(16773121 * 2.0 ** -48), F32(1.0))          # 1 + 2^-24 + 2^-60
    dn = (F32((2 ** 18 - 1) * 2.0 ** -18), F32((2 ** 18 + 1) * 2.0 ** -42), F32(1.0 + 2.0 ** -23))  # 1 + 3*2^-24 - 2^-60
    for a, b, c in (up, dn):
        naive = F32(np.float64(a) * np.float64(b) + np.float64(c))
        good = exact_fma(a, b, c)
        assert naive != good            # the case really exercises the correction
        assert fma32(a, b, c) == good
    assert fma32(*up) == F32(1.0 + 2.0 ** -23)
    assert fma32(*dn) == F32(1.0 + 2.0 ** -23)


def test_weight_special_values():
    assert weight(F32(0.0)) == F32(1.0)
    assert weight(F32(-64.0)) > 0
    assert weight(np.nextafter(F32(-64.0), F32(-np.inf))) == 0
    assert weight(F32(-1000.0)) == 0


def test_weight_error_bound():
    # the exponent t = fl32(d * log2 e) carries a relative error of at most 2^-23 (two roundings),
    # the degree-7 Taylor remainder is below 6e-9 and the Horner FMAs add a few ulps
    d = np.linspace(-64.0, 0.0, 200001).astype(F32)
    w = weight(d).astype(np.float64)
    ref = np.exp(d.astype(np.float64))
    rel = np.abs(w - ref) / ref
    t = np.abs(d.astype(np.float64)) / math.log(2.0)
    bound = math.log(2.0) * t * 2.0 ** -23 + 8 * 2.0 ** -24
    assert np.all(rel <= bound)
    # near the maximum the weight is within 2 ulp of the exponential
    small = np.abs(d) < 1
    assert np.max(rel[small]) < 2 * 2.0 ** -23
