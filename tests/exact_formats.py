"""Exact-rational definitions of the FP4 / FP8 / E8M0 formats, for pinning the
oracle.  Everything here is derived from the bit-field definitions with
Python's fractions, independently of the oracle's float tables and loops.

E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0 is
subnormal (value m/2).  E4M3 (OCP "FN"): sign bit 7, exponent bits 6..3
(bias 7), mantissa bits 2..0; exponent 0 subnormal (m/8 * 2^-6); S.1111.111
is NaN; no infinities.  E8M0: value 2^(code - 127), 0xFF NaN.
"""
from fractions import Fraction
import math


def e2m1_exact(code: int) -> Fraction:
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    if e == 0:
        v = Fraction(m, 2)
    else:
        v = (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return -v if s else v


def e4m3_exact(code: int):
    s, e, m = (code >> 7) & 1, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return None  # NaN
    if e == 0:
        v = Fraction(m, 8) * Fraction(1, 2 ** 6)
    else:
        v = (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def e8m0_exact(code: int):
    if code == 0xFF:
        return None
    return Fraction(2) ** (code - 127)


E2M1_POS = sorted({e2m1_exact(c) for c in range(8)})          # 0 .. 6
E4M3_POS = [(c, e4m3_exact(c)) for c in range(0x7F)]          # codes 0..0x7E


def nearest_even(a: Fraction, table):
    """Nearest entry of `table` [(code, value)] to a; ties to the even code."""
    best = None
    for code, v in table:
        d = abs(a - v)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return best[1]


def e2m1_rne_exact(y: float) -> int:
    sign = 8 if math.copysign(1.0, y) < 0 else 0
    a = abs(Fraction(y))
    if a >= 6:
        return sign | 7
    return sign | nearest_even(a, [(c, e2m1_exact(c)) for c in range(8)])


def e4m3_encode_exact(s: float) -> int:
    a = Fraction(s)
    if a >= 448:
        return 0x7E
    return nearest_even(a, E4M3_POS)


def sr_up_count_exact(y: float) -> int:
    """Number of 16-bit u (of 65536) for which stochastic rounding of |y| < 6
    goes up: ceil(frac * 65536) with frac the exact position in the gap."""
    a = abs(Fraction(y))
    grid = [e2m1_exact(c) for c in range(8)]
    lo = max(i for i in range(8) if grid[i] <= a)
    frac = (a - grid[lo]) / (grid[lo + 1] - grid[lo])
    return math.ceil(frac * 65536)


def floor_log2_exact(a: float) -> int:
    f = Fraction(a)
    k = f.numerator.bit_length() - f.denominator.bit_length()
    if Fraction(2) ** k > f:
        k -= 1
    return k
