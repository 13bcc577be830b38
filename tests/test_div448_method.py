"""The two-instruction division by 448 of the kernels' group scale, checked
on the CPU in exact integer arithmetic (no GPU, no oracle).

The kernels form RN32(a / 448) as q = RN(a zh + RN(a zl)) with
zh = RN(1/448), zl = RN(1/448 - zh) (Brisebarre, Muller and Raina,
"Accelerating correctly rounded floating-point division when the divisor is
known in advance", IEEE Trans. Computers 53(8), 2004).  That method is exact
for some divisors only.  For a normal a and quotient, scaling a by a power
of two scales every intermediate exactly, so it suffices to check all 2^23
significands a in [1, 2).  Every product and sum below fits in int64.
"""

from fractions import Fraction

import numpy as np

ZH = float.fromhex("0x1.24924ap-9")    # the constants in csrc/fp8q_rounding.cuh
ZL = float.fromhex("-0x1.b6db6ep-34")


def _split(x: float):
    """x = M * 2^e with M a signed integer of at most 24 bits."""
    f = Fraction(x)
    s = -1 if f < 0 else 1
    f = abs(f)
    e = f.numerator.bit_length() - f.denominator.bit_length()
    while Fraction(2) ** e > f:
        e -= 1
    while Fraction(2) ** (e + 1) <= f:
        e += 1
    M = f / Fraction(2) ** (e - 23)
    assert M.denominator == 1 and M.numerator < (1 << 24)
    return s * M.numerator, e - 23


def _bitlen(v: np.ndarray) -> np.ndarray:
    """Bit length of positive int64 values (exact)."""
    n = np.floor(np.log2(v.astype(np.float64))).astype(np.int64) + 1
    n = np.where((np.int64(1) << np.minimum(n, 62)) <= v, n + 1, n)
    n = np.where((np.int64(1) << (n - 1)) > v, n - 1, n)
    return n


def _rn24(v: np.ndarray):
    """Round positive int64 values to 24 significant bits, ties to even:
    returns (mantissa, shift) with value ~ mantissa * 2^shift."""
    sh = np.maximum(_bitlen(v) - 24, 0)
    m = v >> sh
    rem = v - (m << sh)
    half = np.where(sh > 0, np.int64(1) << np.maximum(sh - 1, 0), 0)
    up = (sh > 0) & ((rem > half) | ((rem == half) & (m & 1 == 1)))
    m = m + up
    carry = m >= (1 << 24)
    return np.where(carry, m >> 1, m), sh + carry


def test_constants_are_the_rounded_reciprocal_and_remainder():
    inv = Fraction(1, 448)
    assert Fraction(ZH) == Fraction(round(inv * 2 ** 32), 2 ** 32)   # 1/448 in [2^-9, 2^-8): ulp 2^-32
    rem = inv - Fraction(ZH)
    # zl is rem rounded to 24 bits
    m, e = _split(ZL)
    assert abs(rem - Fraction(ZL)) <= Fraction(2) ** e / 2


def test_division_by_448_is_correctly_rounded_for_every_significand():
    m = np.arange(1 << 23, 1 << 24, dtype=np.int64)          # a = m 2^-23
    Mh, eh = _split(ZH)
    Ml, el = _split(ZL)
    # p = RN(a zl): |a zl| = m |Ml| 2^(el - 23), m |Ml| < 2^48
    P, psh = _rn24(m * abs(Ml))
    ep = psh + el - 23                                        # p = sign(Ml) P 2^ep
    A = m * Mh                                                # a zh = A 2^(eh - 23), A < 2^48
    g = (eh - 23) - ep
    assert g.min() >= 0 and g.max() <= 14                     # A 2^g < 2^62
    S = (A << g) + np.sign(Ml) * P                            # a zh + p = S 2^ep, exactly
    Q, qsh = _rn24(S)                                         # q = Q 2^(ep + qsh)
    qe = ep + qsh
    # RN(a / 448) = RN(m / 7) 2^-29: m / 7 in [2^20, 2^22), written as N 2^k, N 24 bits
    k = np.where(m >= 7 << 21, -2, -3)
    num = m << (-k)                                           # m 2^-k, divided by 7
    N = num // 7
    r = num - 7 * N
    N = N + ((2 * r > 7) | ((2 * r == 7) & (N & 1 == 1)))
    assert np.all((N >= 1 << 23) & (N < 1 << 24))
    te = k - 29
    # both sides as (24-bit mantissa, exponent)
    bad = (Q != N) | (qe != te)
    assert not bad.any(), (int(bad.sum()), m[bad][:5])


def test_ue8m0_scale_from_the_bits_of_amax():
    """The kernels' UE8M0 scale skips the division: for a = m 2^e (m in
    [1, 2)) the smallest power of two >= RN32(a / 448) is 2^(e - 8), doubled
    when m > 1.75.  Checked exactly for every significand (the identity is
    invariant under scaling a by powers of two while everything stays
    normal): 2^j >= RN32(a / 448) must hold for the formula's j and fail for
    j - 1."""
    M = np.arange(1 << 23, dtype=np.int64)             # mantissa field; a = (2^23 + M) 2^-23
    j = np.where(M > 0x600000, 1, 0) - 8                 # exponent of the scale, for e = 0
    # RN32(a/448) <= 2^j  <=>  a/448 <= 2^j + ulp(2^j)/2 = 2^j (1 + 2^-24)  (ties go to the even 2^j)
    #                     <=>  (2^23 + M) 2^-23 <= 448 2^j (1 + 2^-24)
    #                     <=>  (2^23 + M) 2^25 <= 7 2^(j + 54) + 7 2^(j + 30)     [times 2^48]
    lhs = (np.int64(1 << 23) + M) << 25

    def bound(jj):
        return 7 * ((np.int64(1) << (jj + 54)) + (np.int64(1) << (jj + 30)))
    assert np.all(lhs <= bound(j))                       # 2^j is an upper bound
    assert np.all(lhs > bound(j - 1))                    # 2^(j-1) is not
