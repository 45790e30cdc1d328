"""The int8 payload's quantizer divides every value of a 256-element block by
the block's scale with Markstein's correction instead of a full IEEE division
(P. Markstein, IBM J. Res. Dev. 34(1), 1990), so that the code
rint(p / scale) is taken from the correctly rounded quotient: from
y = RN(1/b) and q0 = RN(a*y), two corrections q' = RN(q + RN(a - q*b)*y) (each
two fmas), falling back to IEEE division outside 2^-100 <= |a| <= 2^100.
Markstein's theorem needs a faithful q; q0 alone is not always faithful (an
example is pinned below), the first correction makes it so, and the second is
then the correctly rounded quotient.  Checked in exact rational arithmetic
with binary32 round-to-nearest-even on random operands and on the corner where
q0 is furthest off (both significands just below 2: 1/b sits just above a
power of two, where RN(1/b) has its largest relative error, and a/b near the
top of its binade)."""
import math
import random
from fractions import Fraction as Fr


def rn32(x):
    """x (exact rational, normal binary32 range) rounded to binary32, ties to even."""
    if x == 0:
        return Fr(0)
    s = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fr(2) ** e > x:
        e -= 1
    while Fr(2) ** (e + 1) <= x:
        e += 1
    q = x / Fr(2) ** (e - 23)
    n, rem = divmod(q.numerator, q.denominator)
    rem = Fr(rem, q.denominator)
    if rem > Fr(1, 2) or (rem == Fr(1, 2) and n % 2):
        n += 1
    return s * n * Fr(2) ** (e - 23)


def f32(sig, exp):
    """sig in [2^23, 2^24): the binary32 sig * 2^(exp - 23)."""
    return Fr(sig) * Fr(2) ** (exp - 23)


def ulp_above(v):
    """Gap from binary32 v > 0 to the next larger binary32 (normal range)."""
    e = v.numerator.bit_length() - v.denominator.bit_length()
    while Fr(2) ** e > v:
        e -= 1
    while Fr(2) ** (e + 1) <= v:
        e += 1
    return Fr(2) ** (e - 23)


def faithful(q, x):
    """q is one of the two binary32 numbers that bracket x (x, q > 0)."""
    r = rn32(x)
    if r == x:
        return q == r
    if r < x:
        lo, hi = r, r + ulp_above(r)
    else:
        hi = r
        is_pow2 = r.denominator & (r.denominator - 1) == 0 and \
            r.numerator & (r.numerator - 1) == 0
        lo = r - (ulp_above(r) / 2 if is_pow2 else ulp_above(r))
    return q in (lo, hi)


def markstein(a, b):
    """The kernels' division; asserts the premises of Markstein's theorem for
    the second correction (a faithful q1, an exact remainder)."""
    y = rn32(1 / b)
    q0 = rn32(a * y)
    q1 = rn32(q0 + rn32(a - q0 * b) * y)
    assert faithful(abs(q1), abs(a / b))
    r1 = rn32(a - q1 * b)
    assert r1 == a - q1 * b                   # the second remainder is exact
    return rn32(q1 + r1 * y)


def test_one_correction_can_start_from_an_unfaithful_quotient():
    a, b = Fr(15197189, 2 ** 37), Fr(16291847, 2 ** 25)
    y = rn32(1 / b)
    q0 = rn32(a * y)
    assert not faithful(q0, a / b)
    assert faithful(rn32(a / b), a / b)
    assert rn32(a - q0 * b) != a - q0 * b     # its remainder is not exact


def test_rn32_reference():
    assert rn32(Fr(1, 3)) == Fr(11184811, 2 ** 25)           # 0x3EAAAAAB
    assert rn32(Fr(2 ** 24 + 1)) == 2 ** 24                  # tie to even
    assert rn32(Fr(2 ** 24 + 3)) == 2 ** 24 + 4
    assert math.isclose(float(rn32(Fr(1, 10))), 0.1, rel_tol=1e-7)


def test_markstein_quotient_is_correctly_rounded():
    rng = random.Random(20261202)
    cases = []
    for _ in range(3000):                          # random significands, divisor in [2^-10, 1]
        cases.append((f32(rng.randrange(1 << 23, 1 << 24), rng.randrange(-20, 20)),
                      f32(rng.randrange(1 << 23, 1 << 24), rng.randrange(-10, 0))))
    for _ in range(6000):                          # the corner: both significands just below 2
        cases.append((f32((1 << 24) - rng.randrange(1, 20000), rng.randrange(-20, 20)),
                      f32((1 << 24) - rng.randrange(1, 20000), rng.randrange(-10, 0))))
    for _ in range(1000):                          # divisors of the form 1 - beta^t
        t = rng.randrange(1, 20000)
        b = rn32(Fr(1) - Fr(rng.choice([0.9, 0.999])) ** t) if t < 400 else Fr(1)
        cases.append((f32(rng.randrange(1 << 23, 1 << 24), rng.randrange(-40, 0)), b))
    for a, b in cases:
        for sa in (a, -a):
            assert markstein(sa, b) == rn32(sa / b), (sa, b)
