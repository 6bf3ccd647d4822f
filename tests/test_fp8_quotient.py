"""The FP8 grouped GEMM encodes its intermediate, and the FP8 dispatch its
token rows, with x / s computed from the reciprocal rs = RN(1/s) as
q = RN(x * rs), then q + RN(x - q*s) * rs rounded once (Markstein's correction
step; the residual is exact under fma).  Emulated
here with exact rational arithmetic on fp32 inputs: over the range the kernel
uses (s = amax / 448, |x| <= amax) the result equals the correctly rounded
fp32 quotient, i.e. what an IEEE division gives."""
import math
from fractions import Fraction

import numpy as np


def rn32(v: Fraction) -> np.float32:
    """Round an exact rational to the nearest fp32 (ties to even), normal range."""
    if v == 0:
        return np.float32(0.0)
    a = abs(v)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    scale = Fraction(2) ** (23 - e)
    m = a * scale
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    out = float(Fraction(fl) / scale)
    return np.float32(out if v > 0 else -out)


def F(x) -> Fraction:
    return Fraction(float(x))


def test_rn32_against_numpy_cast():
    """Pin of the rounding helper: doubles exactly representable in 53 bits round
    like numpy's float64 -> float32 cast (itself round-to-nearest-even)."""
    rng = np.random.default_rng(1)
    for v in rng.standard_normal(2000) * 10.0 ** rng.uniform(-6, 6, 2000):
        assert rn32(Fraction(float(v))) == np.float32(v)


def test_reciprocal_quotient_is_correctly_rounded():
    rng = np.random.default_rng(0)
    for _ in range(4000):
        amax = np.float32(abs(rng.standard_normal()) * 10.0 ** rng.uniform(-3, 3))
        s = np.float32(amax / np.float32(448.0))
        x = np.float32(rng.uniform(-1.0, 1.0) * amax)
        rs = rn32(1 / F(s))
        q = np.float32(x * rs)                     # one fp32 product
        r = rn32(F(x) - F(q) * F(s))              # fma(-q, s, x): exact residual, rounded once
        got = rn32(F(r) * F(rs) + F(q))           # fma(r, rs, q)
        assert got == rn32(F(x) / F(s)), (x, s)
