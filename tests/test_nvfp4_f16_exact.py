"""The NVFP4 grouped GEMM expands E2M1 values times their E4M3 block scale to
f16 in shared memory and multiplies in f16; that expansion is only exact if
every such product is representable in f16.  These tests enumerate all code
pairs with decoders written from the two formats' bit-level definitions
(E2M1: sign, 2 exponent bits with bias 1, 1 mantissa bit, subnormal when the
exponent field is 0; E4M3: sign, 4 exponent bits with bias 7, 3 mantissa bits,
subnormal when the exponent field is 0, S.1111.111 is NaN), independently of
the oracle's decoders.
"""
import numpy as np


def e2m1_value(code: int) -> float:
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5  # subnormal: m * 2^(1 - bias) * 2^-1
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


def e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6  # subnormal
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def exact_in_f16(x: float) -> bool:
    return float(np.float16(x)) == x


def test_decoders_reach_the_formats_extremes():
    e2m1 = sorted({abs(e2m1_value(c)) for c in range(16)})
    assert e2m1 == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    finite = [e4m3_value(c) for c in range(128) if c != 0x7F]
    assert max(finite) == 448.0
    assert min(v for v in finite if v > 0) == 2.0 ** -9


def test_every_scale_and_value_is_exact_in_f16():
    for c in range(256):
        v = e4m3_value(c)
        if not np.isnan(v):
            assert exact_in_f16(v), hex(c)
    for c in range(16):
        assert exact_in_f16(e2m1_value(c)), hex(c)


def test_every_product_is_exact_in_f16_and_in_range():
    """Block scales are non-negative E4M3 codes (0x00..0x7E); the product of
    a 2-significant-bit value and a 4-significant-bit scale has at most 6
    significant bits, and magnitudes lie in [2^-10, 6 * 448 = 2688]."""
    smallest, largest = np.inf, 0.0
    for sc in range(0x7F):
        s = e4m3_value(sc)
        for vc in range(16):
            p = e2m1_value(vc) * s  # exact in float64
            assert exact_in_f16(p), (hex(vc), hex(sc))
            # the f16 multiply of the two exact f16 operands returns the product unrounded
            assert float(np.float16(e2m1_value(vc)) * np.float16(s)) == p, (hex(vc), hex(sc))
            if p != 0.0:
                smallest = min(smallest, abs(p))
                largest = max(largest, abs(p))
    assert smallest == 2.0 ** -10
    assert largest == 2688.0
