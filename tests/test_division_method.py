"""The E2M1 quantising epilogue divides by the block scale without a division
instruction per element: it takes the correctly rounded reciprocal r = rn(1/sc)
once per 32-element block, then q0 = rn(|x| r), the exact residual
e = |x| - q0 sc (one FMA) and q = rn(q0 + e r) (one FMA), with the sign of x
-- Markstein's final step of FMA-based division.  The codes then equal those
of the IEEE quotient only if q == rn(x / sc) for every x and scale.

This test replays the method in exact rational arithmetic (every fp32
operation rounded once, to nearest even, from its exact value) and compares
it with the exactly rounded quotient: every positive finite E4M3 scale
against seeded random fp32 significands, plus the significands nearest to
each E2M1 rounding boundary times each scale.  It checks the method, not the
kernel; the kernel's codes are compared bit for bit with the oracle's
quantiser on the GPU."""
from fractions import Fraction

import numpy as np
import torch


def _rn32(v: Fraction) -> Fraction:
    """v rounded to the nearest fp32 value, ties to even (normal and
    subnormal range; the values here never overflow)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                      # subnormals share the smallest exponent
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp                           # significand in ulps, exact
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def _e4m3_scales():
    codes = torch.arange(1, 0x7F, dtype=torch.uint8)          # positive finite codes
    return [Fraction(float(v)) for v in codes.view(torch.float8_e4m3fn).float().tolist()]


def _method(x: Fraction, sc: Fraction) -> Fraction:
    ax = abs(x)
    r = _rn32(1 / sc)
    q0 = _rn32(ax * r)
    e = _rn32(ax - q0 * sc)               # the FMA's single rounding (exact here)
    q = _rn32(q0 + e * r)
    return q if x >= 0 else -q


def test_e4m3_scales_are_the_126_positive_finite_codes():
    sc = _e4m3_scales()
    assert len(sc) == 126 and sc[0] == Fraction(1, 512) and sc[-1] == 448


def test_reciprocal_step_equals_ieee_division_random_significands():
    rng = np.random.default_rng(20251203)
    # fp32 values of |x| / sc within the E2M1 range and beyond, both signs
    xs = (rng.uniform(1.0, 2.0, 60).astype(np.float32) *
          np.float32(2.0) ** rng.integers(-8, 9, 60).astype(np.float32)) * rng.choice([-1, 1], 60)
    bad = []
    for sc in _e4m3_scales():
        for xf in xs.astype(np.float32):
            x = Fraction(float(xf))
            want = _rn32(x / sc)
            if _method(x, sc) != want:
                bad.append((float(xf), float(sc)))
    assert not bad, bad[:5]


def test_reciprocal_step_equals_ieee_division_at_e2m1_boundaries():
    # x whose quotient lies on, or one ulp either side of, each E2M1 rounding
    # boundary (0.25, 0.75, ..., 5) and on the largest magnitude 6
    bad = []
    for sc in _e4m3_scales():
        for b in (Fraction(1, 4), Fraction(3, 4), Fraction(5, 4), Fraction(7, 4), Fraction(5, 2),
                  Fraction(7, 2), Fraction(5), Fraction(6)):
            c = np.float32(float(_rn32(b * sc)))
            near = [c]
            for _ in range(2):
                near.append(np.nextafter(near[-1], np.float32(np.inf)))
                near.insert(0, np.nextafter(near[0], np.float32(0)))
            for xf in near:
                x = Fraction(float(xf))
                if _method(x, sc) != _rn32(x / sc):
                    bad.append((float(x), float(sc)))
                if _method(-x, sc) != _rn32(-x / sc):
                    bad.append((float(-x), float(sc)))
    assert not bad, bad[:5]
