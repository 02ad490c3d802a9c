"""The key path's division-free quotient, checked on the host in exact
arithmetic (no GPU).

The encode kernel forms RN(a / b) for the keys' scale, zero point and codes
(encodeKeys divides by the level count and by scale + eps) without a
division (div_by_recip): y = RN(1 / b), q0 = RN(a y), q = RN(q0 + RN(a - q0 b) y)
(two fmas). q0 can be 1.5 ulp from a / b, and its remainder is then not
exact; q is still RN(a / b): a wrong q needs a rounding midpoint m within
3 2^-24 ulp of a / b, and there q0 = m +- ulp / 2 (one ulp at most from
a / b, so the remainder is exact) and the corrected value moves by less than
a / b's distance to m (the argument is written out at div_by_recip). The
argument is scale-free, so these checks use integer significands: random
pairs; divisors with all-ones and near-one significands, where y's error is
largest; quotients as close to a midpoint as two fp32 values allow (a - m b =
k units of the last place of m b, small k); and, exhaustively, the corner
where |a y - m| can come near one ulp (m near the top of its binade, b's
significand near 2^24). Each case is evaluated with exact rationals rounded
once per operation to fp32.
"""
from fractions import Fraction

import numpy as np

from oracle.lloyd_fit import round_f32


def _rn(q):
    return Fraction(float(round_f32(q)))


def _one_step(a, b):
    y = _rn(1 / b)
    q0 = _rn(a * y)
    r = _rn(a - q0 * b)
    return q0, r, _rn(q0 + r * y)


def _check(a, b):
    q0, r, q = _one_step(a, b)
    assert q == _rn(a / b), (a, b)
    return r != a - q0 * b


def _near_midpoint(Bi, k):
    """a (a 24-bit integer times 2^25) with a / Bi = M - k / Bi for the odd
    25-bit M = k Bi^-1 mod 2^25, or None: a / b is then k / Bi from the
    midpoint M of the fp32 grid of spacing 2 on [2^24, 2^25)."""
    M = (k * pow(Bi, -1, 1 << 25)) % (1 << 25)
    if M < (1 << 24) or M % 2 == 0:
        return None
    ai = M * Bi - k
    A = ai >> 25
    if A < (1 << 23) or A >= (1 << 24):
        return None
    return Fraction(ai)


def test_random_and_wide_error_divisors():
    rng = np.random.default_rng(12)
    inexact = 0
    divisors = [Fraction(int(b)) for b in rng.integers(1 << 23, 1 << 24, 200)]
    divisors += [Fraction((1 << 24) - j) for j in range(1, 40)] + [Fraction((1 << 23) + j) for j in range(1, 40)]
    divisors += [Fraction(3), Fraction(15), Fraction(31), Fraction(255), Fraction(254)]  # the level counts
    for b in divisors:
        for A in rng.integers(1 << 23, 1 << 24, 40):
            inexact += _check(Fraction(int(A)) * Fraction(2) ** int(rng.integers(-30, 30)), b)
    assert inexact > 0  # q0 is sometimes 1.5 ulp off; q is right all the same


def test_quotients_next_to_midpoints():
    rng = np.random.default_rng(13)
    n = 0
    for Bi in list(rng.integers((1 << 23) + 1, 1 << 24, 150) | 1) + [(1 << 24) - 1 - 2 * j for j in range(50)]:
        for k in range(-12, 13):
            a = _near_midpoint(int(Bi), k) if k else None
            if a is not None:
                _check(a, Fraction(int(Bi)))
                n += 1
    assert n > 500


def test_corner_where_the_first_guess_can_reach_one_ulp():
    """|a y - m| can only come near one ulp when M Bi >= 2^49 - 3 2^25
    (M >= 2^25 - 6 and Bi >= 2^24 - 3); exhaustive over a wider corner, odd M
    in [2^25 - 256, 2^25) and Bi in [2^24 - 256, 2^24), for every a within 8
    units of M Bi that is a 24-bit value times 2^25 (a quotient within
    3 2^-24 ulp of the midpoint M needs |k| <= 6). Such pairs are rare: every
    one found is checked."""
    for M in range((1 << 25) - 255, 1 << 25, 2):
        for Bi in range((1 << 24) - 256, 1 << 24):
            p = M * Bi
            for k in range(-8, 9):
                if (p - k) % (1 << 25) == 0:
                    _check(Fraction(p - k), Fraction(Bi))
