"""The CUDA FP4 encoder forms fl32(amax_b / 6) without a division, as
q = fl32(amax_b * r), e = fma(-q, 6, amax_b), q' = fma(e, r, q) with
r = fl32(1/6).  amax_b is always a bf16 value, so every case can be checked:
this test does it with exact rational arithmetic (each FMA rounded once, to
nearest even, as the hardware does) against the correctly rounded quotient
the encode rule asks for."""

from fractions import Fraction

import numpy as np


def _round_f32(x: Fraction) -> Fraction:
    """Round a rational to the nearest float32 (ties to even), finite range."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                       # subnormals share the 2^-149 quantum
    q = Fraction(2) ** (e - 23)
    m = a / q
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * q


def test_fma_corrected_quotient_matches_division_for_every_bf16():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    r = _round_f32(Fraction(1, 6))
    assert float(r) == float(np.float32(1.0) / np.float32(6.0))
    bad = 0
    for v in vals:
        a = Fraction(float(v))
        q = _round_f32(a * r)
        e = _round_f32(a - q * 6)
        q2 = _round_f32(e * r + q)
        if q2 != _round_f32(a / 6):
            bad += 1
    assert bad == 0


def test_rounding_helper_against_numpy():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(2000).astype(np.float32) * np.float32(2.0) ** rng.integers(-60, 60, 2000)
    for a, b in zip(x[:1000], x[1000:]):
        if b == 0:
            continue
        want = np.float32(a) / np.float32(b)
        assert float(_round_f32(Fraction(float(a)) / Fraction(float(b)))) == float(want)
