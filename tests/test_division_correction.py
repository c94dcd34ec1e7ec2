"""The prefill epilogue's division (bw_gemm.cu, div_by_recip): a / s as
the product with r = RN(1 / s), corrected twice by its fma residual.  By
P. Markstein's theorem on the final correction step of division, once the
quotient is within one ulp the residual is exact and the corrected value is
the correctly rounded quotient.  This test replays the steps in exact
rational arithmetic, rounding to binary32 after every operation as the GPU
does (one rounding per fma), on seeded integers a (|a| <= 2^23, the exact
accumulators) and activation scales s = 127 / absmax, and checks every
result against RN(a / s) -- and that the second residual is exact."""
import math
import random
from fractions import Fraction

import numpy as np


def rn32(v: Fraction) -> Fraction:
    """v rounded to the nearest binary32 value, ties to even (normal range)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    v = abs(v)
    e = v.numerator.bit_length() - v.denominator.bit_length()
    if Fraction(2) ** e > v:
        e -= 1
    unit = Fraction(2) ** (e - 23)           # 24-bit significand
    m = v / unit
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * unit


def test_corrected_reciprocal_product_is_the_rounded_quotient():
    rng = random.Random(20240607)
    for i in range(3000):
        a = Fraction(rng.randint(-(1 << 23), 1 << 23))
        if i % 5 == 0:
            a = Fraction(rng.randint(-300, 300))
        absmax = float(np.float32(math.exp(rng.uniform(math.log(1e-6),
                                                       math.log(1e6)))))
        s = Fraction(float(np.float32(127.0 / absmax)))
        r = rn32(1 / s)                                  # the IEEE division
        q0 = rn32(a * r)                                 # a * r
        q1 = rn32(rn32(a - q0 * s) * r + q0)             # fma(fma(-q0,s,a),r,q0)
        res = a - q1 * s
        assert rn32(res) == res, (a, s)                  # exact residual
        q2 = rn32(res * r + q1)                          # fma(fma(-q1,s,a),r,q1)
        assert q2 == rn32(a / s), (a, s, q2)


def test_the_bare_product_is_not_the_quotient():
    """The product a r alone is often off (so a correction is needed) and
    can be more than one ulp off, where the theorem's precondition fails
    for a single correction: hence the two steps."""
    rng = random.Random(7)
    misses = beyond_one_ulp = 0
    for _ in range(3000):
        a = Fraction(rng.randint(1, 1 << 23))
        absmax = float(np.float32(math.exp(rng.uniform(math.log(1e-3),
                                                       math.log(1e4)))))
        s = Fraction(float(np.float32(127.0 / absmax)))
        r = rn32(1 / s)
        q0 = rn32(a * r)
        exact = a / s
        misses += q0 != rn32(exact)
        e = exact.numerator.bit_length() - exact.denominator.bit_length()
        if Fraction(2) ** e > exact:
            e -= 1
        beyond_one_ulp += abs(q0 - exact) > Fraction(2) ** (e - 23)
    assert misses > 0 and beyond_one_ulp > 0
