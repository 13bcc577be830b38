"""Exact rational arithmetic used to pin the oracle.

Nothing here calls the oracle or the CUDA library.  Every rounding is done
on ``fractions.Fraction`` values from the definition of the target format,
so a mistake in the oracle's C arithmetic (a dropped term, a wrong rounding
rule, a wrong exponent) shows up as a disagreement with these functions.
"""

from __future__ import annotations

import bisect
import math
import struct
from fractions import Fraction

HALF = Fraction(1, 2)


def f32(x: float) -> float:
    """The fp32 value nearest to a Python float (numpy-free)."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def f32_from_bits(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def bf16_to_float(b: int) -> float:
    return f32_from_bits((b & 0xFFFF) << 16)


def is_neg(x: float) -> bool:
    return math.copysign(1.0, x) < 0


def _floor_log2(a: Fraction) -> int:
    """floor(log2 a) for a > 0, exactly."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    # 2^e <= a < 2^(e+1) after at most one correction each way
    if _pow2(e) > a:
        e -= 1
    if _pow2(e + 1) <= a:
        e += 1
    return e


def _pow2(e: int) -> Fraction:
    return Fraction(1 << e) if e >= 0 else Fraction(1, 1 << -e)


def _round_half_even(n: Fraction) -> int:
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > HALF or (rem == HALF and fl % 2 == 1):
        fl += 1
    return fl


def rn32(fr: Fraction, negative_zero: bool = False) -> float:
    """Round an exact rational to the nearest binary32 value, ties to even.

    Subnormals are produced (quantum 2^-149 below 2^-126); results beyond the
    largest finite value round to infinity as IEEE round-to-nearest does.
    """
    if fr == 0:
        return -0.0 if negative_zero else 0.0
    sign = -1.0 if fr < 0 else 1.0
    a = abs(fr)
    e = max(_floor_log2(a), -126)
    quantum = _pow2(e - 23)
    n = _round_half_even(a / quantum)
    val = n * quantum
    if val >= _pow2(128):
        return sign * math.inf
    return sign * float(val)  # exact: n <= 2^24 fits a double


def sqrt_rn32(x: float) -> float:
    """Correctly rounded binary32 square root of a non-negative binary32 x."""
    a = Fraction(x)
    if a == 0:
        return x
    E = _floor_log2(a) // 2  # floor(log2 sqrt(a))
    E = max(E, -126)
    quantum = _pow2(E - 23)
    Y = a / (quantum * quantum)  # sqrt(a)/quantum = sqrt(Y)
    n0 = math.isqrt(Y.numerator // Y.denominator)
    # round: compare Y with (n0 + 1/2)^2
    mid = (Fraction(2 * n0 + 1, 2)) ** 2
    n = n0 + 1 if Y > mid else n0
    if Y == mid and n0 % 2 == 1:
        n = n0 + 1
    return float(n * quantum)


# ------------------------------------------------------------- e4m3 table --


def e4m3_decode(code: int) -> Fraction | None:
    """Value of a float8_e4m3fn code (None for NaN): 1 sign, 4 exponent bits
    with bias 7, 3 mantissa bits; exponent field 0 is subnormal (M * 2^-9)."""
    E = (code >> 3) & 0xF
    M = code & 0x7
    if E == 0xF and M == 0x7:
        return None
    mag = Fraction(M, 512) if E == 0 else Fraction(8 + M) * _pow2(E - 10)
    return -mag if code & 0x80 else mag


_POS = [(e4m3_decode(c), c) for c in range(0x7F)]
_POS.sort()
_POS_VALS = [v for v, _ in _POS]
MAX_E4M3 = Fraction(448)


def e4m3_nearest(value: Fraction, negative: bool) -> int:
    """Brute-force rounding to float8_e4m3fn: the nearest of the finite
    values, ties to the code with an even mantissa, magnitudes above 448
    saturating to 448, the sign carried separately (so -0 keeps its sign)."""
    sign = 0x80 if negative else 0x00
    a = abs(value)
    if a >= MAX_E4M3:
        return sign | 0x7E
    i = bisect.bisect_left(_POS_VALS, a)
    if _POS_VALS[i] == a:
        return sign | _POS[i][1]
    lo_v, lo_c = _POS[i - 1]
    hi_v, hi_c = _POS[i]
    dl, dh = a - lo_v, hi_v - a
    if dl < dh:
        c = lo_c
    elif dh < dl:
        c = hi_c
    else:
        c = lo_c if lo_c % 2 == 0 else hi_c
    return sign | c


def e4m3_of_float(x: float) -> int:
    return e4m3_nearest(Fraction(x), is_neg(x))


# ------------------------------------------ exact transcription of op A --


def group_scale(amax: float, ue8m0: bool, eps: float = f32(1e-10)) -> tuple[float, float]:
    """(scale, scale before the power-of-two rounding), from exact rationals."""
    m = max(Fraction(amax), Fraction(eps))
    pre = rn32(m / 448)
    if not ue8m0:
        return pre, pre
    # smallest power of two >= pre
    a = Fraction(pre)
    e = _floor_log2(a)
    s = a if _pow2(e) == a else _pow2(e + 1)
    return float(s), pre


def quant_value(x: float, s: float) -> int:
    """e4m3(RN32(x / s)) with both roundings done on exact rationals."""
    p = rn32(Fraction(x) / Fraction(s), negative_zero=is_neg(x) != is_neg(s))
    return e4m3_of_float(p)


def quant_group_exact(vals, ue8m0: bool):
    amax = max(abs(v) for v in vals)
    s, pre = group_scale(amax, ue8m0)
    return [quant_value(v, s) for v in vals], s, pre
