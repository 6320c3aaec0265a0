"""The activation quantisers divide by the block scale without a division
instruction: with r = RN(1/s), q0 = RN(v*r), rem = v - s*q0 (exact by FMA),
q = RN(q0 + rem*r) (Markstein's correction step).  The E2M1 code taken from q
must be the code of the correctly rounded quotient RN(v/s), the rule of
NVFP4 activation quantisation.  Checked here in exact rational arithmetic
(no GPU) for every positive E4M3 scale s: every FP32 v within 48 ulps of
each code decision point t*s (t the midpoints 0.25, 0.75, ... 5), both signs,
where the quotient could round across a decision point; plus a random sample
of (v, s) elsewhere, where q must equal RN(v/s) as well."""
from fractions import Fraction

import numpy as np

THRESHOLDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def rn32(x: Fraction) -> Fraction:
    """x rounded to the nearest FP32 value, ties to even (normal and
    subnormal range; no overflow in this use)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def e4m3_positive_values():
    out = []
    for code in range(1, 127):
        e, m = code >> 3, code & 7
        out.append(Fraction(m, 8) * Fraction(2) ** -6 if e == 0
                   else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return out


def fast_div(v: Fraction, s: Fraction, r: Fraction) -> Fraction:
    q0 = rn32(v * r)
    rem = rn32(v - s * q0)
    return rn32(q0 + rem * r)


def f32_neighbours(x: float, k: int):
    """FP32 values k ulps below .. k ulps above the FP32 value x."""
    b = np.array([x], np.float32).view(np.int32)[0]
    ints = np.arange(b - k, b + k + 1, dtype=np.int64)
    return [Fraction(float(f)) for f in ints.astype(np.int32).view(np.float32)]


def test_rn32_matches_numpy_on_exact_doubles():
    rng = np.random.default_rng(0)
    for x in rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000):
        assert rn32(Fraction(float(x))) == Fraction(float(np.float32(x)))


def test_division_shortcut_decides_every_code_like_exact_division():
    for s in e4m3_positive_values():
        r = rn32(1 / s)
        for t in THRESHOLDS:
            c = float(np.float32(float(t * s)))  # t*s is exact in FP32
            for v in f32_neighbours(c, 48):
                for sv in (v, -v):
                    assert fast_div(sv, s, r) == rn32(sv / s), (float(sv), float(s))


def test_division_shortcut_is_correctly_rounded_on_a_random_sample():
    rng = np.random.default_rng(1)
    scales = e4m3_positive_values()
    for _ in range(20000):
        s = scales[rng.integers(len(scales))]
        v = Fraction(float(np.float32(float(s) * rng.uniform(-8.0, 8.0))))
        assert fast_div(v, s, rn32(1 / s)) == rn32(v / s)
