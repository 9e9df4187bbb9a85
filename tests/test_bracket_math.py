"""The arithmetic argument behind the expert-major quantiser's codes (the
kernel quantises y = v / scale through two reciprocals rh > 1/scale > rl
instead of dividing), checked exactly on the CPU with rational arithmetic:

* from a maximum a, r0 within two units in the last place of 1/a (the PTX ISA
  bounds the hardware's approximate reciprocal by one), one Newton step
  r1 = fma(r0, fma(-a, r0, 1), r0), r = F * r1, rh = r * (1 + 2^-21) and
  rl = r * (1 - 2^-21), each rounded to fp32 once, satisfy
  rh * scale > 1 + 2^-24 and rl * scale < 1 - 2^-24 for scale = fl(a / F);
* so for any v, v * rh and v * rl bracket Q = fl(v / scale), and where the
  per-token int8 rounding (fl(v * r + 1.5 * 2^23), one rounding of the exact
  product) or the FP8 conversion of both ends agree, Q's code is the same.

Every fp32 rounding here is done exactly (Fraction -> nearest fp32, ties to
even), not through float64, so that no double rounding hides a failure."""
import math
from fractions import Fraction

import numpy as np
import pytest

TWO = Fraction(2)


def rn32(x: Fraction) -> Fraction:
    """x rounded to the nearest fp32 value, ties to even (normal and subnormal
    range; no overflow in the values used here)."""
    if x == 0:
        return Fraction(0)
    s = -1 if x < 0 else 1
    m = abs(x)
    e = math.floor(math.log2(m.numerator) - math.log2(m.denominator))
    # correct the estimate so that 2^e <= m < 2^(e+1)
    while TWO ** e > m:
        e -= 1
    while TWO ** (e + 1) <= m:
        e += 1
    e = max(e, -126)
    ulp = TWO ** (e - 23)
    q = m / ulp
    f = q.numerator // q.denominator
    rem = q - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return s * f * ulp


def f32(x: float) -> Fraction:
    return Fraction(float(np.float32(x)))


def ulp32(x: Fraction) -> Fraction:
    e = math.floor(math.log2(abs(float(x))))
    return TWO ** (max(e, -126) - 23)


def brackets(a: Fraction, F: Fraction, k: int):
    r0 = rn32(1 / a) + k * ulp32(1 / a)
    r1 = rn32(r0 * rn32(1 - a * r0) + r0)  # fma(r0, fma(-a, r0, 1), r0): each fma rounds once
    r = rn32(F * r1)
    return rn32(r * (1 + TWO ** -21)), rn32(r * (1 - TWO ** -21))


def maxima(n: int, seed: int):
    rng = np.random.default_rng(seed)
    out = [Fraction(1), Fraction(127), Fraction(448), TWO ** -100, TWO ** 100, f32(np.nextafter(np.float32(1), 2))]
    e = rng.integers(-100, 100, size=n)
    m = rng.uniform(1.0, 2.0, size=n)
    out += [f32(float(mi) * 2.0 ** int(ei)) for mi, ei in zip(m, e)]
    return out


@pytest.mark.parametrize("F", [127, 448, 57344])
def test_reciprocal_brackets_enclose_one_over_scale(F):
    F = Fraction(F)
    for a in maxima(300, 11 + int(F)):
        scale = rn32(a / F)
        for k in (-2, -1, 0, 1, 2):
            rh, rl = brackets(a, F, k)
            assert rh * scale > 1 + TWO ** -24, (a, k)
            assert rl * scale < 1 - TWO ** -24, (a, k)


def rne_int(x: Fraction) -> int:
    f = x.numerator // x.denominator
    rem = x - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def test_int8_codes_agree_with_the_division_where_the_brackets_agree():
    """Per-token int8: t = fl(v * r + 1.5 * 2^23) rounds the exact product once;
    both ends' integers equal => the quotient's integer equals them. Values on
    and next to half-integers included (they must disagree, not mis-round)."""
    rng = np.random.default_rng(5)
    M = Fraction(3, 2) * TWO ** 23
    agreed = 0
    for trial in range(400):
        a = f32(rng.uniform(0.5, 300.0) * 2.0 ** int(rng.integers(-20, 20)))
        scale = rn32(a / 127)
        rh, rl = brackets(a, Fraction(127), int(rng.integers(-2, 3)))
        for _ in range(8):
            if rng.random() < 0.5:
                v = f32(float(rng.uniform(-1, 1)) * float(a))
            else:  # v / scale near a half-integer
                n = int(rng.integers(-127, 127))
                v = rn32((n + Fraction(1, 2)) * scale) + int(rng.integers(-2, 3)) * ulp32(a)
                if abs(v) > a:
                    continue
            q = rne_int(rn32(v / scale))
            th, tl = rn32(v * rh + M), rn32(v * rl + M)
            if th == tl:
                agreed += 1
                assert th - M == q, (a, v)
    assert agreed > 1500


def fp8_e4m3(x: Fraction) -> Fraction:
    """fp32 value -> nearest OCP E4M3 value (ties to even), saturating at 448."""
    if x == 0:
        return Fraction(0)
    s = -1 if x < 0 else 1
    m = abs(x)
    if m >= 448:
        return s * Fraction(448)
    e = max(math.floor(math.log2(float(m))), -6)
    ulp = TWO ** (e - 3)
    q = m / ulp
    f = q.numerator // q.denominator
    rem = q - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return s * min(f * ulp, Fraction(448))


def test_fp8_codes_agree_with_the_division_where_the_brackets_agree():
    """Per-group FP8 E4M3: y = fl(v * rh), fl(v * rl) converted to FP8; both
    ends equal => the quotient's FP8 value equals them (midpoints included)."""
    rng = np.random.default_rng(6)
    agreed = 0
    for trial in range(400):
        a = f32(rng.uniform(0.5, 300.0) * 2.0 ** int(rng.integers(-20, 20)))
        scale = rn32(a / 448)
        rh, rl = brackets(a, Fraction(448), int(rng.integers(-2, 3)))
        for _ in range(8):
            if rng.random() < 0.5:
                v = f32(float(rng.uniform(-1, 1)) * float(a))
            else:  # v / scale near an E4M3 midpoint
                e = int(rng.integers(-6, 9))
                m = int(rng.integers(8, 16))
                mid = min((m + Fraction(1, 2)) * TWO ** (e - 3), Fraction(448))
                v = rn32(mid * scale) + int(rng.integers(-2, 3)) * ulp32(a)
                if abs(v) > a:
                    continue
            c = fp8_e4m3(rn32(v / scale))
            ch, cl = fp8_e4m3(rn32(v * rh)), fp8_e4m3(rn32(v * rl))
            if ch == cl:
                agreed += 1
                assert ch == c, (a, v)
    assert agreed > 1500
