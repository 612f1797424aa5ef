"""The FP8 1x128 cast divides each value by its block scale s = amax/448.
The CUDA kernels form that quotient without a division per element, by
Markstein's correction step (P. Markstein, "Computation of elementary
functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
1990): r = RN(1/s), q0 = RN(x*r), e = RN(s*q0 - x), q = RN(q0 - e*r).

This checks, in exact rational arithmetic, that q is the IEEE quotient
RN(x/s) for every pair of bf16 significands (x and amax) and both signs.
Exponent gaps of 0 and 1 between x and amax are enough: every operation
scales exactly by powers of two, so a larger gap repeats the gap-1 case
scaled, as long as nothing underflows (the kernels take the IEEE division
for scales below 2^-90, and quotients below 2^-11 code to zero either way).
The GPU test of every bf16 value at every relative scale checks the device
codes themselves."""
from fractions import Fraction as F


def rn32(v):
    """Round an exact rational to the nearest fp32 value (ties to even);
    normal range only."""
    if v == 0:
        return F(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    elif F(2) ** (e + 1) <= a:
        e += 1
    assert F(2) ** e <= a < F(2) ** (e + 1) and e >= -126
    scaled = a * F(2) ** (23 - e)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > F(1, 2) or (rem == F(1, 2) and n % 2 == 1):
        n += 1
    return sign * F(n) * F(2) ** (e - 23)


def test_rn32_rounds_like_fp32():
    import numpy as np
    rng = np.random.default_rng(1)
    for a, b in rng.uniform(0.5, 4.0, (200, 2)):
        a32, b32 = np.float32(a), np.float32(b)
        assert rn32(F(float(a32)) / F(float(b32))) == F(float(a32 / b32))
    assert rn32(F(1) + F(1, 2 ** 24)) == 1                       # tie to even (down)
    assert rn32(F(1) + F(3, 2 ** 24)) == F(1) + F(2, 2 ** 23)    # tie to even (up)


def test_corrected_quotient_is_the_ieee_quotient():
    mismatches = []
    for ia in range(128):
        amax = F(128 + ia, 128)
        s = rn32(amax / 448)
        r = rn32(1 / s)
        for ix in range(128):
            for gap in (0, 1):
                x = F(128 + ix, 128) / 2 ** gap
                if x > amax:
                    continue
                for xs in (x, -x):
                    q0 = rn32(xs * r)
                    e = rn32(q0 * s - xs)
                    q = rn32(q0 - e * r)
                    if q != rn32(xs / s):
                        mismatches.append((ia, ix, gap))
    assert not mismatches, mismatches[:5]
