"""Host checks of the identities the fp8 quantisation kernel relies on to avoid per-element
division (exact rational arithmetic, no GPU):

- block scale: for every bf16 amax from 2^-100 up, RN(amax / 448) equals Markstein's
  corrected product RN(q0 + RN(amax - 448 q0) * c), q0 = RN(amax * c), c = RN(1/448);
- the quotient bracket: RN(x * RN(r (1 -+ 2^-19))) lies strictly below / above RN(x / s)
  for any r within 2^-23 of 1/s, so equal e4m3 codes at both ends fix the quotient's code.
"""
from fractions import Fraction as F

import numpy as np
import pytest


def rn32(q: F) -> F:
    """q rounded to the nearest fp32 value, ties to even (normal range)."""
    if q == 0:
        return F(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    assert e >= -126
    scaled = a / F(2) ** (e - 23)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > F(1, 2) or (rem == F(1, 2) and n % 2 == 1):
        n += 1
    return sign * F(n) * F(2) ** (e - 23)


def test_rn32_matches_numpy_division():
    rng = np.random.default_rng(0)
    a = rng.standard_normal(2000).astype(np.float32)
    b = (rng.random(2000) + 0.1).astype(np.float32)
    for x, y in zip(a, b):
        assert rn32(F(float(x)) / F(float(y))) == F(float(np.float32(x) / np.float32(y)))


def test_block_scale_correction_is_exact_for_every_bf16():
    c = rn32(F(1, 448))
    checked = 0
    for hi in range(0x0001, 0x7F80):
        x = float(np.array([hi << 16], np.uint32).view(np.float32)[0])
        if x < 2.0 ** -100:
            continue
        X = F(x)
        q0 = rn32(X * c)
        r = rn32(X - q0 * 448)
        assert rn32(r * c + q0) == rn32(X / 448), hex(hi)
        checked += 1
    assert checked == 29184


@pytest.mark.parametrize("seed", [0, 1])
def test_quotient_bracket_is_strict(seed):
    rng = np.random.default_rng(seed)
    lo_f, hi_f = F(1) - F(1, 2 ** 19), F(1) + F(1, 2 ** 19)
    for _ in range(3000):
        s = F(float(np.float32(abs(rng.standard_normal()) * 2.0 ** rng.integers(-60, 60) + 1e-30)))
        x = F(float(np.float32(rng.standard_normal() * 2.0 ** rng.integers(-20, 20))))
        r = rn32(F(1) / s * (1 + F(int(rng.integers(-2 ** 20, 2 ** 20)), 2 ** 43)))   # within 2^-23 of 1/s
        q = rn32(x / s)
        lo, hi = rn32(x * rn32(r * lo_f)), rn32(x * rn32(r * hi_f))
        if x > 0:
            assert lo < q < hi
        elif x < 0:
            assert hi < q < lo
