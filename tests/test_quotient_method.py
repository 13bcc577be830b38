"""The kernels' correctly rounded quotient RN32(v / s) for a non-power-of-two
scale, checked on the CPU in exact rational arithmetic (no GPU, no oracle).

The method: r = RN(1/s); rd = r if 1 - s r >= 0, else r's predecessor (so
rd <= 1/s); rl = RN(RN(1 - s rd) r) >= 0.  With w = -v:
y0 = RN(w (-rd) + RN(w (-rl))), e = RN(s y0 + w), y1 = RN(y0 + e (-r)),
every step one fp32 operation (an FMA where a product meets a third value).
y0 is a faithful quotient and one Markstein step with the exact residual
makes it correctly rounded.  The cases put quotients next to rounding
midpoints, where a wrong step shows, and cover signed zeros and quotients
that underflow.  Values are modelled as (exact rational, sign bit), with
IEEE 754's rules for the sign of a zero result under rounding to nearest.
"""

from dataclasses import dataclass
from fractions import Fraction

import numpy as np

TWO = Fraction(2)


def _rn(x: Fraction) -> Fraction:
    """x rounded to the nearest fp32 value, ties to even (subnormals kept)."""
    if x == 0:
        return Fraction(0)
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while TWO ** e > a:
        e -= 1
    while TWO ** (e + 1) <= a:
        e += 1
    ulp = TWO ** (max(e, -126) - 23)
    m = a / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return (n * ulp) if x > 0 else -(n * ulp)


@dataclass(frozen=True)
class F:
    """An fp32 value: its exact value and its sign bit."""
    v: Fraction
    neg: bool

    @staticmethod
    def of(x: Fraction) -> "F":
        x = _rn(Fraction(x))
        return F(x, x < 0)

    def __neg__(self):
        return F(-self.v, not self.neg)


def _round(exact: Fraction, zero_neg: bool) -> F:
    """Round an exact result; a zero result (exact or by underflow) gets the
    sign IEEE gives it: that of the exact value when nonzero, else zero_neg."""
    y = _rn(exact)
    if y != 0:
        return F(y, y < 0)
    return F(Fraction(0), exact < 0 if exact != 0 else zero_neg)


def mul(a: F, b: F) -> F:
    return _round(a.v * b.v, a.neg != b.neg)


def fma(a: F, b: F, c: F) -> F:
    """RN(a b + c).  An exact zero sum is -0 only if the product and c are
    both negative zeros; a zero sum of nonzero terms is +0."""
    p = a.v * b.v
    pneg = a.neg != b.neg
    exact = p + c.v
    zero_neg = (p == 0 and c.v == 0 and pneg and c.neg)
    return _round(exact, zero_neg)


def pred(x: Fraction) -> Fraction:
    """The fp32 value just below a positive normal fp32 x."""
    b = np.array([np.float32(float(x))], dtype=np.float32).view(np.uint32)
    return Fraction(float((b - np.uint32(1)).view(np.float32)[0]))


def quotient(v: F, s: Fraction) -> F:
    one = F(Fraction(1), False)
    sf = F(s, False)
    r = F.of(1 / s)
    rem = fma(-sf, r, one)
    assert rem.v == 1 - s * r.v                              # the residual is exact
    rd = r if rem.v >= 0 else F(pred(r.v), False)
    assert rd.v <= 1 / s < rd.v + TWO ** -20 * r.v
    ed = fma(-sf, rd, one)
    assert ed.v == 1 - s * rd.v and ed.v >= 0
    rl = mul(ed, r)
    w = -v
    y0 = fma(w, -rd, mul(w, -rl))
    e = fma(sf, y0, w)
    return fma(e, -r, y0)


def _scales(rng, n):
    """Group scales RN32(amax / 448), amax spread over the binades; powers of
    two (the UE8M0 path) left out."""
    out = []
    while len(out) < n:
        amax = Fraction(float(np.float32(rng.uniform(1, 2)))) * TWO ** int(rng.integers(-40, 40))
        s = _rn(amax / 448)
        if s.numerator & (s.numerator - 1) == 0 and s.denominator & (s.denominator - 1) == 0:
            continue
        out.append((amax, s))
    return out


def test_random_quotients_are_correctly_rounded():
    rng = np.random.default_rng(11)
    for amax, s in _scales(rng, 300):
        for _ in range(20):
            v = F.of(amax * Fraction(float(rng.uniform(-1, 1))))
            y = quotient(v, s)
            assert y.v == _rn(v.v / s), (float(v.v), float(s))
            assert y.v == 0 or y.neg == (v.v < 0)


def test_quotients_next_to_rounding_midpoints():
    """v/s within a few ulp of a midpoint between two fp32 values, where a
    step that is off by one shows."""
    rng = np.random.default_rng(12)
    n = 0
    for amax, s in _scales(rng, 300):
        for _ in range(10):
            q = _rn(Fraction(float(rng.uniform(1, 448))) * TWO ** int(rng.integers(-12, 1)))
            if q > amax / s:
                continue
            e = q.numerator.bit_length() - q.denominator.bit_length()
            while TWO ** e > q:
                e -= 1
            mid = q + TWO ** (e - 24)                       # halfway to the next fp32 up
            base = _rn(s * mid)
            be = base.numerator.bit_length() - base.denominator.bit_length()
            while TWO ** be > base:
                be -= 1
            for k in range(-3, 4):
                v = F.of(base + k * TWO ** (be - 23))
                if abs(v.v) > amax:
                    continue
                for sv in (v, -v):
                    y = quotient(sv, s)
                    assert y.v == _rn(sv.v / s), (float(sv.v), float(s))
                    n += 1
    assert n > 10000


def test_signed_zeros_and_underflow_keep_the_sign_of_v():
    rng = np.random.default_rng(13)
    for amax, s in _scales(rng, 60):
        for neg in (False, True):
            y = quotient(F(Fraction(0), neg), s)
            assert y.v == 0 and y.neg == neg
        for v in (TWO ** -149, -(TWO ** -149), TWO ** -126, -(TWO ** -126)):
            y = quotient(F(v, v < 0), s)
            assert y.v == _rn(v / s)
            assert y.neg == (v < 0)


def test_an_early_version_that_dropped_the_sign_fails_the_zero_case():
    """The same steps with v instead of -v (e = RN(-s y0 + v), y1 = RN(y0 +
    e r)) give +0 for v = -0: the case the sign-keeping order exists for."""
    s = _rn(Fraction(3, 448))
    sf = F(s, False)
    r = F.of(1 / s)
    v = F(Fraction(0), True)
    y0 = mul(v, r)
    e = fma(-sf, y0, v)
    y1 = fma(e, r, y0)
    assert y0.neg and not y1.neg
    assert quotient(v, s).neg


def _faithful_start_only(v: F, s: Fraction) -> F:
    """The method without its correction step: y0 = RN(v rd + RN(v rl))."""
    one = F(Fraction(1), False)
    sf = F(s, False)
    r = F.of(1 / s)
    rd = r if fma(-sf, r, one).v >= 0 else F(pred(r.v), False)
    rl = mul(fma(-sf, rd, one), r)
    w = -v
    return fma(w, -rd, mul(w, -rl))


def _near_midpoint_cases(rng, n):
    """(v, s) whose quotient lies within about 2^-47 (relative) of a midpoint
    between two fp32 values, where the start's own 2^-45 error can decide the
    rounding.  For an odd significand S of s and a small odd t, the midpoint
    numerator N = 2^24 + (t S^-1 mod 2^24) (odd, 25 bits) makes S N = V 2^24
    + t, so v = V (scaled) gives v/s = N 2^-24 (1 - t / (S N)) (scaled)."""
    cases = []
    mod = 1 << 24
    while len(cases) < n:
        S = int(rng.integers(1 << 22, 1 << 23)) * 2 + 1            # odd, 24 bits
        t = int(rng.choice([-3, -1, 1, 3]))
        N = mod + (t * pow(S, -1, mod)) % mod
        P = S * N
        assert (P - t) % mod == 0
        V = (P - t) // mod
        if V >= mod:
            continue
        for shift in (-9, -3, 0, 4, 7):                            # quotients from about 2^-9 to 2^8
            a = int(rng.integers(-40, 30))
            s = Fraction(S) * TWO ** (a - 23)
            v = Fraction(V) * TWO ** (a - 23 + shift)
            mid = Fraction(N) * TWO ** (shift - 24)
            assert abs(v / s - mid) <= 3 * mid / (S * N) and _rn(s) == s and _rn(v) == v
            cases.append((F(v, False), s))
    return cases


def test_quotients_within_2_pow_minus_47_of_a_midpoint():
    rng = np.random.default_rng(14)
    cases = _near_midpoint_cases(rng, 4000)
    for v, s in cases:
        for sv in (v, -v):
            assert quotient(sv, s).v == _rn(sv.v / s), (float(sv.v), float(s))
    # the start alone rounds some of them the wrong way, and so does a step
    # taken with rd instead of the correctly rounded r: these cases test both
    wrong = sum(_faithful_start_only(v, s).v != _rn(v.v / s) for v, s in cases)
    assert wrong > 0
    wrong = sum(_step_with_rd(v, s).v != _rn(v.v / s) for v, s in cases)
    assert wrong > 0


def _step_with_rd(v: F, s: Fraction) -> F:
    """The method with rd in the correction step instead of r = RN(1/s)."""
    one = F(Fraction(1), False)
    sf = F(s, False)
    r = F.of(1 / s)
    rd = r if fma(-sf, r, one).v >= 0 else F(pred(r.v), False)
    rl = mul(fma(-sf, rd, one), r)
    w = -v
    y0 = fma(w, -rd, mul(w, -rl))
    return fma(fma(sf, y0, w), -rd, y0)
