"""Pins of the CPU oracle: checks against what the format definition and the
mathematics fix, independent of the oracle's own C arithmetic.

Each ``pin_*`` function takes no argument, calls the oracle through the
``oracle`` module (whichever build of it is active) and raises
``AssertionError`` when the oracle disagrees.  ``test_oracle.py`` runs them
on the real oracle; ``test_oracle_mutations.py`` runs them on copies of the
oracle with a planted mistake and requires that some pin fails for each.
"""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

import oracle
from fp8_token_group_bf16_b300 import inputs

from exact import (
    bf16_to_float,
    e4m3_decode,
    e4m3_nearest,
    e4m3_of_float,
    f32,
    group_scale,
    is_neg,
    quant_group_exact,
    quant_value,
    rn32,
    sqrt_rn32,
)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EPS = f32(1e-10)
RMS_EPS = f32(1e-6)


def load_midpoints():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_midpoints.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            val, code = line.split()[:2]
            rows.append((float(val), int(code, 16)))
    return rows


def all_bf16_finite() -> np.ndarray:
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (b >> 7) & 0xFF
    return b[exp != 0xFF]


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def ordinal(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes on a monotone integer line (sign-magnitude -> integer)."""
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


# ------------------------------------------------------------- e4m3 -----


def pin_e4m3_exhaustive_bf16():
    """Every finite bf16 value against the brute-force nearest e4m3 value."""
    b = all_bf16_finite()
    got = oracle.f32_to_e4m3(bf16_bits_to_f32(b))
    for bits, code in zip(b.tolist(), got.tolist()):
        x = bf16_to_float(bits)
        want = e4m3_nearest(Fraction(x), is_neg(x))
        assert code == want, f"bf16 {bits:#06x} ({x!r}): oracle {code:#04x}, brute force {want:#04x}"


def structured_f32() -> np.ndarray:
    """fp32 values around every e4m3 rounding boundary: for each exponent in
    the range that matters, all 2^8 top-mantissa patterns times low-bit
    patterns that hit exact ties and their neighbours."""
    out = []
    lows = np.array([0, 1, 2, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x7FFFF, 0x80000, 0x80001, 0xFFFFF,
                     0x3FFFF, 0x40000, 0x40001, 0x1FFFFF, 0x200000, 0x200001], np.uint32)
    for e in range(100, 140):
        top = np.arange(256, dtype=np.uint32) << 15
        m = (top[:, None] | lows[None, :]) & 0x7FFFFF
        u = (np.uint32(e) << 23) | m.ravel()
        out.append(u)
        out.append(u | np.uint32(0x80000000))
    return np.concatenate(out).view(np.float32)


def pin_e4m3_torch_cast():
    """Against torch's float8_e4m3fn cast, a third implementation, after
    clamping to +-448 (torch's cast does not saturate)."""
    rng = np.random.default_rng(7)
    rand = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    v = np.concatenate([bf16_bits_to_f32(all_bf16_finite()), structured_f32(), rand.view(np.float32)])
    v = v[~np.isnan(v)]
    got = oracle.f32_to_e4m3(v)
    clamped = torch.from_numpy(np.clip(v, -448.0, 448.0))
    ref = clamped.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first v={v[bad[0]]!r} oracle={got[bad[0]]:#x} torch={ref[bad[0]]:#x}"


def pin_e4m3_structured_exact():
    """Tie and near-tie fp32 inputs against the exact brute force."""
    v = structured_f32()
    got = oracle.f32_to_e4m3(v)
    for x, c in zip(v.tolist()[::7], got.tolist()[::7]):
        want = e4m3_of_float(x)
        assert c == want, f"{x!r}: oracle {c:#x}, exact {want:#x}"


def pin_e4m3_roundtrip():
    """Every finite code decodes to a value the oracle encodes back to it."""
    for c in range(256):
        v = e4m3_decode(c)
        if v is None:
            continue
        x = float(v)
        if c == 0x80:
            x = -0.0
        got = int(oracle.f32_to_e4m3(np.array([x], np.float32))[0])
        assert got == c, f"code {c:#x} value {x!r} -> {got:#x}"


def pin_golden_midpoints():
    rows = load_midpoints()
    v = np.array([r[0] for r in rows], np.float32)
    got = oracle.f32_to_e4m3(v)
    for (val, want), c in zip(rows, got.tolist()):
        assert c == want, f"{val}: oracle {c:#x}, golden {want:#x}"


def pin_ue8m0():
    """Power-of-two ceiling: result is a power of two, >= s, and < 2 s."""
    rng = np.random.default_rng(3)
    s = np.concatenate([
        (rng.random(20000) * 2.0 ** rng.integers(-60, 60, 20000)).astype(np.float32),
        np.array([2.0 ** k for k in range(-60, 60)], np.float32),
        np.array([np.nextafter(np.float32(2.0 ** k), np.float32(np.inf)) for k in range(-60, 60)], np.float32),
        np.array([np.nextafter(np.float32(2.0 ** k), np.float32(0)) for k in range(-60, 60)], np.float32),
    ])
    s = s[s > 0]
    got = oracle.ue8m0_ceil(s)
    for x, y in zip(s.tolist(), got.tolist()):
        a = Fraction(x)
        r = Fraction(y)
        assert r >= a and r / 2 < a, f"ue8m0({x!r}) = {y!r}"
        m, e = math.frexp(y)
        assert m == 0.5, f"ue8m0({x!r}) = {y!r} is not a power of two"


def pin_group_scale_fp32():
    """The scale from an fp32 amax (ops B and C meet any fp32 amax): against
    exact rational division by 448, the floor applied first, and the
    power-of-two ceiling, over amax values spread across the exponent range,
    near the floor, and next to multiples of 448 times powers of two."""
    rng = np.random.default_rng(11)
    a = (1.0 + rng.random(2500)) * 2.0 ** rng.integers(-100, 100, 2500)
    near = np.array([448.0 * 2.0 ** k for k in range(-60, 60, 7)])
    a = np.concatenate([a, near, np.nextafter(near, np.inf), np.nextafter(near, 0),
                        [0.0, 1e-30, 1e-10, 9.99e-11, 1.0000001e-10, 3.0e38]]).astype(np.float32)
    for ue8m0 in (False, True):
        got = oracle.group_scale(a, ue8m0=ue8m0)
        for x, y in zip(a.tolist(), got.tolist()):
            want, _ = group_scale(x, ue8m0)
            assert y == want, f"group_scale({x!r}, ue8m0={ue8m0}) = {y!r}, exact {want!r}"


# -------------------------------------------------- op A (per group) ----


def pin_op_a_hand_rows():
    x = inputs.small_group_quant_input()
    xb = inputs.bits(x)
    golden = [c for _, c in load_midpoints()]
    for ue8m0 in (False, True):
        q, s, _ = oracle.per_token_group_quant(xb, ue8m0=ue8m0)
        # row 18: rounding midpoints; groups 0..3 = mid, 2 mid, -mid, -2 mid
        mid_codes = q[18, : len(golden) - 2]
        assert mid_codes.tolist() == golden[:-2], (ue8m0, mid_codes)
        for g, (scale, flip) in enumerate([(1.0, 0), (2.0, 0), (1.0, 0x80), (2.0, 0x80)]):
            assert s[18, g] == scale, (ue8m0, g, s[18, g])
            assert np.array_equal(q[18, g * 128 : (g + 1) * 128], q[18, :128] ^ flip), (ue8m0, g)
        # row 16 group 0: all-zero group -> floor scale, zero codes with signs
        want_s = group_scale(0.0, ue8m0)[0]
        assert s[16, 0] == np.float32(want_s), (ue8m0, s[16, 0], want_s)
        if ue8m0:
            assert s[16, 0] == np.float32(2.0**-42)
        signs = (xb[16, :128] >> 15).astype(np.uint8) << 7
        assert np.array_equal(q[16, :128], signs)
        # row 17: +-1e4 outlier (bf16 9984) in groups 0 and 1
        top = 0x7E if not ue8m0 else quant_value(9984.0, group_scale(9984.0, True)[0])
        assert q[17, 5] == top and q[17, 128 + 5] == top | 0x80, (ue8m0, q[17, 5])
        assert s[17, 0] == np.float32(group_scale(9984.0, ue8m0)[0])
        d = q[17, :128] ^ q[17, 128:256]
        assert d[5] == 0x80 and np.count_nonzero(d) == 1, d
        # row 19 group 1: bf16 subnormals quantise to signed zeros
        signs = (xb[19, 128:256] >> 15).astype(np.uint8) << 7
        assert np.array_equal(q[19, 128:256], signs)


def _exact_op_a(xb: np.ndarray, ue8m0: bool, group: int = 128):
    T, H = xb.shape
    G = H // group
    q = np.zeros((T, H), np.uint8)
    s = np.zeros((T, G), np.float32)
    for t in range(T):
        for g in range(G):
            vals = [bf16_to_float(int(b)) for b in xb[t, g * group : (g + 1) * group]]
            codes, sc, _ = quant_group_exact(vals, ue8m0)
            q[t, g * group : (g + 1) * group] = codes
            s[t, g] = sc
    return q, s


def pin_op_a_bruteforce():
    """The whole op on small inputs against the exact-rational transcription."""
    rs = np.random.default_rng(11)
    xs = [inputs.bits(inputs.hand_rows(512))]
    for scale in (1.0, 1e-3, 37.0, 3e4):
        f = torch.from_numpy((rs.standard_normal((2, 256)) * scale).astype(np.float32))
        xs.append(inputs.bits(inputs.bf16(f)))
    xs.append(inputs.bits(inputs.heavy_tailed_input(4, 512, seed=99)))
    for xb in xs:
        for ue8m0 in (False, True):
            q, s, _ = oracle.per_token_group_quant(xb, ue8m0=ue8m0)
            qe, se = _exact_op_a(xb, ue8m0)
            assert np.array_equal(s, se), (ue8m0, np.nonzero(s != se))
            bad = np.argwhere(q != qe)
            assert bad.size == 0, (ue8m0, bad[:5], q[tuple(bad[0])], qe[tuple(bad[0])])


def near_midpoint_cases(n_scales: int = 400, seed: int = 5):
    """(amax, x) bf16 pairs whose quotient x / RN32(amax/448) lies within
    2^-19 (relative) of an e4m3 rounding midpoint, found with float64 and
    kept only if the exact quotient is not itself a midpoint-free case.
    These stress the correctly rounded fp32 quotient: a multiply by the
    reciprocal, or a division that is off by one ulp, changes their code."""
    rng = np.random.default_rng(seed)
    b = all_bf16_finite()
    xv = bf16_bits_to_f32(b).astype(np.float64)
    pos = xv > 0
    xb_pos, xv_pos = b[pos], xv[pos]
    # midpoints between consecutive positive e4m3 values
    vals = np.array([float(e4m3_decode(c)) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2.0
    cases = []
    for amax_bits in rng.choice(xb_pos[(xv_pos > 1e-6) & (xv_pos < 1e6)], n_scales, replace=False):
        amax = float(bf16_bits_to_f32(np.array([amax_bits]))[0])
        s = np.float32(np.float32(amax) / np.float32(448.0))
        sel = xv_pos <= amax
        qv = xv_pos[sel] / float(s)
        j = np.clip(np.searchsorted(mids, qv), 1, len(mids) - 1)
        d = np.minimum(np.abs(qv - mids[j]), np.abs(qv - mids[j - 1])) / np.maximum(qv, 1e-30)
        hit = np.nonzero((d < 2.0**-19) & (qv > 2.0**-10))[0]
        for k in hit[:8]:
            cases.append((int(amax_bits), int(xb_pos[sel][k])))
    return cases


def near_midpoint_groups(cases, group: int = 128) -> np.ndarray:
    """Pack the cases into groups: slot 0 holds amax, the rest the x values
    of that amax (repeated), negated in every other group."""
    by_amax = {}
    for a, x in cases:
        by_amax.setdefault(a, []).append(x)
    rows = []
    for a, xsl in sorted(by_amax.items()):
        g = np.empty(group, np.uint16)
        g[0] = a
        g[1:] = np.resize(np.array(xsl, np.uint16), group - 1)
        rows.append(g)
        rows.append(g ^ np.uint16(0x8000))
    if len(rows) % 4:
        rows += rows[: 4 - len(rows) % 4]
    return np.stack(rows).reshape(-1, 4 * group)


def pin_quotient_near_midpoints():
    cases = near_midpoint_cases()
    assert len(cases) > 20, len(cases)
    xb = near_midpoint_groups(cases)
    q, s, _ = oracle.per_token_group_quant(xb, ue8m0=False)
    qe, se = _exact_op_a(xb, False)
    assert np.array_equal(s, se)
    bad = np.argwhere(q != qe)
    assert bad.size == 0, (bad.shape, bad[:5])


def pin_op_a_invariants():
    """Closed forms on heavy-tailed input: amax -> +-448, UE8M0 max in
    [224, 448], per-element dequant error within half an e4m3 ulp, sign
    symmetry and power-of-two scaling invariance."""
    x = inputs.heavy_tailed_input(16, 7168, seed=inputs.SEED_SWEEP + 50)
    xb = inputs.bits(x)
    xf = bf16_bits_to_f32(xb).astype(np.float64)
    T, H = xb.shape
    G = H // 128
    table = np.zeros(256)
    for c in range(256):
        v = e4m3_decode(c)
        table[c] = float(v) if v is not None else np.nan
    for ue8m0 in (False, True):
        q, s, _ = oracle.per_token_group_quant(xb, ue8m0=ue8m0)
        qf = table[q].reshape(T, G, 128)
        sg = s.astype(np.float64)[:, :, None]
        xg = xf.reshape(T, G, 128)
        if not ue8m0:
            idx = np.abs(xg).argmax(axis=2)
            top = np.take_along_axis(q.reshape(T, G, 128), idx[:, :, None], axis=2)[:, :, 0]
            assert np.all((top & 0x7F) == 0x7E)
        else:
            mq = np.abs(qf).max(axis=2)
            assert np.all((mq >= 224) & (mq <= 448)), mq.min()
            m, e = np.frexp(s)
            assert np.all(m == 0.5)
        err = np.abs(qf * sg - xg)
        bound = np.maximum(2.0**-4 * np.abs(xg) * (1 + 2.0**-23), 2.0**-10 * sg) + 2.0**-23 * np.abs(xg)
        assert np.all(err <= bound), np.max(err / bound)
        # sign symmetry
        qn, sn, _ = oracle.per_token_group_quant(xb ^ np.uint16(0x8000), ue8m0=ue8m0)
        assert np.array_equal(qn, q ^ 0x80) and np.array_equal(sn, s)
        # power-of-two scaling: x * 4 (exact in bf16 here) -> same codes, scale * 4
        x4 = inputs.bits(inputs.bf16(torch.from_numpy(xf.astype(np.float32) * 4.0)))
        q4, s4, _ = oracle.per_token_group_quant(x4, ue8m0=ue8m0)
        assert np.array_equal(q4, q) and np.array_equal(s4, s * 4), ue8m0


def pin_scale_layouts():
    """Column-major scales are the transpose of row-major ones (T != G)."""
    xb = inputs.bits(inputs.heavy_tailed_input(3, 7168, seed=123))
    q0, s0, p0 = oracle.per_token_group_quant(xb, col_major=False)
    q1, s1, p1 = oracle.per_token_group_quant(xb, col_major=True)
    assert s0.shape == (3, 56) and s1.shape == (56, 3)
    assert np.array_equal(q0, q1) and np.array_equal(s1, s0.T) and np.array_equal(p1, p0.T)
    x2 = inputs.bits(inputs.silu_input(3, 256, seed=5))
    qa, sa, _ = oracle.silu_and_mul_per_block_quant(x2, col_major=False)
    qb, sb, _ = oracle.silu_and_mul_per_block_quant(x2, col_major=True)
    assert np.array_equal(qa, qb) and np.array_equal(sb, sa.T)
    x3, w3, _ = inputs.rms_input(3, 256, seeds=(1, 2, 3))
    ra = oracle.rms_norm_per_block_quant(inputs.bits(x3), inputs.bits(w3), col_major=False)
    rb = oracle.rms_norm_per_block_quant(inputs.bits(x3), inputs.bits(w3), col_major=True)
    assert np.array_equal(ra[0], rb[0]) and np.array_equal(rb[1], ra[1].T)


def load_packed_golden():
    T = G = None
    words = {}
    with open(os.path.join(GOLDEN, "ue8m0_packed.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "T":
                T = int(parts[1])
            elif parts[0] == "G":
                G = int(parts[1])
            else:
                k, t, *b = (int(v) for v in parts)
                words[(k, t)] = b
    return T, G, words


def pin_ue8m0_packed_golden():
    """The packing of a hand-derived example, byte for byte."""
    T, G, words = load_packed_golden()
    s = np.array([[2.0 ** (t - g) for g in range(G)] for t in range(T)], np.float32)
    got = oracle.pack_ue8m0(s)
    K, T_pad = -(-G // 4), -(-T // 4) * 4
    assert got.shape == (K, T_pad, 4) and len(words) == K * T_pad
    for (k, t), b in words.items():
        assert got[k, t].tolist() == b, ((k, t), got[k, t].tolist(), b)


def pin_ue8m0_packed_decodes():
    """On op A's UE8M0 scales: every byte decodes to its scale exactly, the
    pad bytes are 0, and the bytes are the scales' exponents as a multiset."""
    for T, H in ((7, 896), (4, 512), (1, 7168)):
        xb = inputs.bits(inputs.heavy_tailed_input(T, H, seed=60 + T))
        _, s, _ = oracle.per_token_group_quant(xb, ue8m0=True)
        G = H // 128
        p = oracle.pack_ue8m0(s)
        K, T_pad = -(-G // 4), -(-T // 4) * 4
        assert p.shape == (K, T_pad, 4)
        seen = []
        for k in range(K):
            for t in range(T_pad):
                for j in range(4):
                    g = 4 * k + j
                    b = int(p[k, t, j])
                    if t >= T or g >= G:
                        assert b == 0, (k, t, j)
                    else:
                        assert math.ldexp(1.0, b - 127) == float(s[t, g]), (t, g, b, s[t, g])
                        seen.append(b)
        want = sorted(int(math.frexp(float(v))[1]) + 126 for v in s.reshape(-1))
        assert sorted(seen) == want


def pin_ue8m0_mx_tiles():
    """The MXFP8 tile layout against an independent construction (repeat each
    group's exponent over its four 32-value blocks, pad rows to 128, cut
    128 x 4 tiles, order rows inside a tile as (r % 32, r // 32)), and every
    byte decoded back to its scale."""
    rng = np.random.default_rng(21)
    for T, G in [(1, 1), (5, 3), (128, 2), (130, 7), (300, 40)]:
        s = np.ldexp(1.0, rng.integers(-30, 10, size=(T, G))).astype(np.float32)
        got = oracle.pack_ue8m0_mx(s)
        e = (np.frexp(s)[1] - 1 + 127).astype(np.uint8)              # exponent bytes [T, G]
        T_pad = -(-T // 128) * 128
        full = np.zeros((T_pad, 4 * G), np.uint8)
        full[:T] = np.repeat(e, 4, axis=1)
        tiles = full.reshape(T_pad // 128, 4, 32, G, 4).transpose(0, 3, 2, 1, 4)
        assert np.array_equal(got.reshape(-1), tiles.reshape(-1)), (T, G)
        flat = got.reshape(-1)
        for t in range(0, T, max(1, T // 7)):
            for g in range(G):
                for j in range(4):
                    at = ((t // 128) * G + g) * 512 + (t % 32) * 16 + ((t % 128) // 32) * 4 + j
                    assert np.ldexp(1.0, int(flat[at]) - 127) == s[t, g]


# ------------------------------------------------------- op B (rms) ----


def _bf16_rn(x: float) -> float:
    """bf16 round to nearest even of an fp32 value, by exact rationals."""
    if x == 0:
        return x
    a = Fraction(abs(x))
    e = max(_flog2(a), -126)
    quantum = Fraction(2) ** (e - 7)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2):
        fl += 1
    v = float(fl * quantum)
    return -v if x < 0 else v


def _flog2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def _exact_inv(ss: float, H: int, eps: float = RMS_EPS) -> float:
    mean = rn32(Fraction(ss) / H)
    var = rn32(Fraction(mean) + Fraction(eps))
    r = sqrt_rn32(var)
    return rn32(1 / Fraction(r))


def _exact_op_b(xb, wb, rb, ue8m0, group: int = 128):
    T, H = xb.shape
    G = H // group
    q = np.zeros((T, H), np.uint8)
    s = np.zeros((T, G), np.float32)
    rout = None if rb is None else np.zeros_like(rb)
    for t in range(T):
        x = [bf16_to_float(int(b)) for b in xb[t]]
        if rb is not None:
            r = [bf16_to_float(int(b)) for b in rb[t]]
            z = [_bf16_rn(rn32(Fraction(a) + Fraction(c))) for a, c in zip(x, r)]
            rout[t] = [np.float32(v).view(np.uint32) >> 16 for v in z]
        else:
            z = x
        ss = rn32(sum(Fraction(v) * Fraction(v) for v in z))
        inv = _exact_inv(ss, H)
        w = [bf16_to_float(int(b)) for b in wb]
        v = [rn32(Fraction(rn32(Fraction(zz) * Fraction(inv))) * Fraction(ww)) for zz, ww in zip(z, w)]
        for g in range(G):
            codes, sc, _ = quant_group_exact(v[g * group : (g + 1) * group], ue8m0)
            q[t, g * group : (g + 1) * group] = codes
            s[t, g] = sc
    return q, s, rout


def pin_rms_inv_chain():
    """1/rms of random sums of squares against the exact step chain
    RN(1 / RN(sqrt(RN(RN(ss/H) + eps))))."""
    rng = np.random.default_rng(17)
    for _ in range(3000):
        H = int(rng.choice([128, 256, 4096, 5120, 7168]))
        ss = float(np.float32(rng.random() * H * 10.0 ** rng.integers(-8, 6)))
        got = float(oracle.rms_inv(ss, H))
        want = _exact_inv(ss, H)
        assert got == want, (ss, H, got, want)


def pin_rms_sumsq():
    """Row sums of squares within 1e-6 of the exact rational sum."""
    x, _, _ = inputs.rms_input(8, 4096, seeds=(31, 32, 33))
    xb = inputs.bits(x)
    got = oracle.row_sumsq(xb)
    for t in range(xb.shape[0]):
        exact = sum(Fraction(bf16_to_float(int(b))) ** 2 for b in xb[t])
        assert abs(Fraction(float(got[t])) - exact) <= exact * Fraction(1, 10**6), t


def pin_rms_bruteforce():
    x, w, r = inputs.rms_input(3, 256, seeds=(41, 42, 43))
    xb, wb, rb = inputs.bits(x), inputs.bits(w), inputs.bits(r)
    for res in (None, rb):
        for ue8m0 in (False, True):
            q, s, _, _, ro = oracle.rms_norm_per_block_quant(xb, wb, res, ue8m0=ue8m0)
            qe, se, re_ = _exact_op_b(xb, wb, res, ue8m0)
            assert np.array_equal(s, se), (ue8m0, res is None)
            assert np.array_equal(q, qe), (ue8m0, res is None, np.argwhere(q != qe)[:4])
            if res is not None:
                assert np.array_equal(ro, re_.astype(np.uint16))


def pin_rms_residual_zero():
    x, w, _ = inputs.rms_input(4, 1024, seeds=(51, 52, 53))
    xb, wb = inputs.bits(x), inputs.bits(w)
    zero = np.zeros_like(xb)
    q0, s0, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, None)
    q1, s1, _, _, ro = oracle.rms_norm_per_block_quant(xb, wb, zero)
    assert np.array_equal(ro, xb) and np.array_equal(q0, q1) and np.array_equal(s0, s1)


def pin_rms_constant_row():
    H = 1024
    for c in (0.75, -3.0, 1e-3):
        xb = inputs.bits(inputs.bf16(torch.full((2, H), c)))
        wb = inputs.bits(inputs.bf16(torch.ones(H)))
        q, s, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, None)
        want = 0x7E if c > 0 else 0xFE
        assert np.all(q == want), (c, np.unique(q))
        assert np.all(s == s.flat[0])


def pin_rms_weight_pow2():
    x, w, _ = inputs.rms_input(4, 512, seeds=(61, 62, 63))
    xb, wb = inputs.bits(x), inputs.bits(w)
    q, s, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, None)
    for k in (1, 3, -2):
        wk = inputs.bits(inputs.bf16(w.float() * 2.0**k))
        qk, sk, _, _, _ = oracle.rms_norm_per_block_quant(xb, wk, None)
        assert np.array_equal(qk, q) and np.array_equal(sk, s * np.float32(2.0**k)), k


# ------------------------------------------------------ op C (silu) ----


def pin_silu_reduces_to_group_quant():
    """Gate >= 20 makes 1 + exp(-a) round to 1, so silu(a) = a; with up = 1
    the op is exactly the per-group quantisation of the gate half."""
    rng = np.random.default_rng(71)
    T, I = 4, 512
    a = (20.0 + np.abs(rng.standard_normal((T, I))) * 50.0).astype(np.float32)
    a[1] *= 1000.0
    ab = inputs.bits(inputs.bf16(torch.from_numpy(a)))
    xb = np.concatenate([ab, inputs.bits(inputs.bf16(torch.ones(T, I)))], axis=1)
    for ue8m0 in (False, True):
        for col in (False, True):
            qc, sc, _ = oracle.silu_and_mul_per_block_quant(xb, ue8m0=ue8m0, col_major=col)
            qa, sa, _ = oracle.per_token_group_quant(ab, ue8m0=ue8m0, col_major=col)
            assert np.array_equal(qc, qa) and np.array_equal(sc, sa), (ue8m0, col)


def pin_silu_zero_gate():
    T, I = 2, 256
    xb = np.concatenate([np.zeros((T, I), np.uint16),
                         inputs.bits(inputs.bf16(torch.randn(T, I, generator=torch.Generator().manual_seed(1))))], axis=1)
    q, s, _ = oracle.silu_and_mul_per_block_quant(xb)
    assert np.all((q & 0x7F) == 0)
    assert np.all(s == np.float32(np.float32(1e-10) / np.float32(448.0)))


def _silu_exact(a: float, b: float) -> tuple[float, float]:
    """(value, ulp) of RN(RN(a / RN(1 + E)) * b) with E = exp(-a) correctly
    rounded to fp32 (mpmath at 80 digits); libm's expf may differ from E by
    an ulp, so the oracle is held to within 2 ulps of this value."""
    import mpmath

    mpmath.mp.dps = 80
    e = mpmath.e ** mpmath.mpf(-a)
    if e > mpmath.mpf(2) ** 128:
        E = math.inf
    else:
        E = rn32(_mp_to_fraction(e))
    if math.isinf(E):
        d = math.inf
        sg = -0.0 if a < 0 else 0.0
    else:
        d = rn32(1 + Fraction(E))
        sg = rn32(Fraction(a) / Fraction(d), negative_zero=a < 0)
    v = f32(sg * b) if (sg == 0 or math.isinf(sg)) else rn32(Fraction(sg) * Fraction(b))
    ulp = float(np.spacing(np.float32(abs(v)))) if v != 0 else 2.0**-149
    return v, ulp


def _mp_to_fraction(x) -> Fraction:
    import mpmath

    m, e = mpmath.frexp(x)
    # m in [0.5, 1): scale to a 200-bit integer
    mi = int(mpmath.floor(m * mpmath.mpf(2) ** 200))
    return Fraction(mi) * (Fraction(2) ** (e - 200))


def pin_silu_values():
    rng = np.random.default_rng(81)
    a = np.concatenate([rng.standard_normal(1500) * 2.0, rng.uniform(-100, 100, 300),
                        np.array([0.0, -0.0, 1e-30, -1e-30, 88.0, -87.0, -89.0, -100.0, 17.0, 20.0])])
    a = a.astype(np.float32)
    b = rng.standard_normal(a.size).astype(np.float32)
    got = oracle.silu_mul(a, b)
    exact_hits = 0
    for ai, bi, g in zip(a.tolist(), b.tolist(), got.tolist()):
        v, ulp = _silu_exact(ai, bi)
        assert abs(g - v) <= 2 * ulp, (ai, bi, g, v)
        exact_hits += g == v
    assert exact_hits >= 0.95 * a.size, exact_hits


def pin_silu_bruteforce():
    """Whole op C on a small input: codes within one e4m3 step and scales
    within 2e-6 of an exact transcription (the only freedom is expf)."""
    xb = inputs.bits(inputs.silu_input(2, 256, seed=91))
    T, I = 2, 256
    for ue8m0 in (False, True):
        q, s, sp = oracle.silu_and_mul_per_block_quant(xb, ue8m0=ue8m0)
        for t in range(T):
            for g in range(I // 128):
                vals = []
                for i in range(128):
                    a = bf16_to_float(int(xb[t, g * 128 + i]))
                    b = bf16_to_float(int(xb[t, I + g * 128 + i]))
                    vals.append(_silu_exact(a, b)[0])
                codes, sc, pre = quant_group_exact(vals, ue8m0)
                assert abs(float(sp[t, g]) - pre) <= 2e-6 * pre, (t, g)
                if not ue8m0:
                    assert abs(float(s[t, g]) - sc) <= 2e-6 * sc
                got = q[t, g * 128 : (g + 1) * 128]
                d = np.abs(ordinal(got) - ordinal(np.array(codes, np.uint8)))
                assert d.max() <= 1 and (d > 0).sum() <= 2, (t, g, d.max())


def pin_silu_large_negative_gate():
    T, I = 1, 128
    a = torch.full((T, I), -100.0)
    b = torch.randn(T, I, generator=torch.Generator().manual_seed(2))
    xb = inputs.bits(inputs.bf16(torch.cat([a, b], dim=1)))
    q, _, _ = oracle.silu_and_mul_per_block_quant(xb)
    assert np.all((q & 0x7F) == 0)
    # -0 * b: sign is that of -b
    bneg = (xb[0, I:] >> 15) == 0  # b >= 0 -> product -0
    assert np.array_equal((q[0] >> 7).astype(bool), bneg)


# ------------------------------------------------- per-token variants ----


def pin_per_token_bruteforce():
    """dynamic_per_token_scaled_fp8_quant on small inputs against the exact-
    rational transcription with one group spanning the row."""
    rs = np.random.default_rng(13)
    xs = [inputs.bits(inputs.hand_rows(512))]
    for scale in (1.0, 3e-3, 5e3):
        f = torch.from_numpy((rs.standard_normal((2, 384)) * scale).astype(np.float32))
        xs.append(inputs.bits(inputs.bf16(f)))
    xs.append(inputs.bits(inputs.heavy_tailed_input(3, 256, seed=77)))
    for xb in xs:
        H = xb.shape[1]
        for ue8m0 in (False, True):
            q, s, _ = oracle.dynamic_per_token_scaled_fp8_quant(xb, ue8m0=ue8m0)
            qe, se = _exact_op_a(xb, ue8m0, group=H)
            assert s.shape == (xb.shape[0],) and np.array_equal(s, se[:, 0]), (ue8m0, s, se[:, 0])
            assert np.array_equal(q, qe), (ue8m0, np.argwhere(q != qe)[:4])


def pin_per_token_row_amax():
    """One scale per row: the row's scale is the largest of its 128-groups'
    scales (division by 448 is monotone), the row's largest |x| gets the
    code +-448, and with UE8M0 the largest |code| of a row lies in [224, 448]."""
    xb = inputs.bits(inputs.heavy_tailed_input(12, 7168, seed=inputs.SEED_SWEEP + 60))
    for ue8m0 in (False, True):
        q, s, sp = oracle.dynamic_per_token_scaled_fp8_quant(xb, ue8m0=ue8m0)
        _, _, spg = oracle.per_token_group_quant(xb, ue8m0=ue8m0)
        assert np.array_equal(sp, spg.max(axis=1))
        xf = np.abs(bf16_bits_to_f32(xb))
        top = q[np.arange(q.shape[0]), xf.argmax(axis=1)]
        if ue8m0:
            table = np.array([abs(float(e4m3_decode(c) or 0)) for c in range(256)])
            full = table[q].max(axis=1)
            assert np.all((full >= 224) & (full <= 448)), full
        else:
            assert np.all((top & 0x7F) == 0x7E), top


def pin_rms_per_token_bruteforce():
    x, w, r = inputs.rms_input(3, 256, seeds=(44, 45, 46))
    xb, wb, rb = inputs.bits(x), inputs.bits(w), inputs.bits(r)
    for res in (None, rb):
        for ue8m0 in (False, True):
            q, s, _, _, ro = oracle.rms_norm_dynamic_per_token_quant(xb, wb, res, ue8m0=ue8m0)
            qe, se, re_ = _exact_op_b(xb, wb, res, ue8m0, group=256)
            assert np.array_equal(s, se[:, 0]), (ue8m0, res is None)
            assert np.array_equal(q, qe), (ue8m0, res is None, np.argwhere(q != qe)[:4])
            if res is not None:
                assert np.array_equal(ro, re_.astype(np.uint16))


def pin_silu_per_token_bruteforce():
    """silu_and_mul_dynamic_per_token_quant on a small input: codes within one
    e4m3 step and the scale within 2e-6 of an exact transcription (the only
    freedom is expf)."""
    T, I = 2, 256
    xb = inputs.bits(inputs.silu_input(T, I, seed=92))
    for ue8m0 in (False, True):
        q, s, sp = oracle.silu_and_mul_dynamic_per_token_quant(xb, ue8m0=ue8m0)
        assert s.shape == (T,)
        for t in range(T):
            vals = [_silu_exact(bf16_to_float(int(xb[t, i])), bf16_to_float(int(xb[t, I + i])))[0]
                    for i in range(I)]
            codes, sc, pre = quant_group_exact(vals, ue8m0)
            assert abs(float(sp[t]) - pre) <= 2e-6 * pre, t
            if not ue8m0:
                assert abs(float(s[t]) - sc) <= 2e-6 * sc
            d = np.abs(ordinal(q[t]) - ordinal(np.array(codes, np.uint8)))
            assert d.max() <= 1 and (d > 0).sum() <= 2, (t, d.max())


# ------------------------------------------------ fused_qk_norm_rope ----


def _exact_qk_rope(xb, qwb, kwb, csb, pos, Hq, Hkv, D, is_neox, eps=RMS_EPS):
    """The op in exact rationals with one RN32 per written step."""
    out = xb.copy()
    half = D // 2
    qw = [bf16_to_float(int(b)) for b in qwb]
    kw = [bf16_to_float(int(b)) for b in kwb]
    for t in range(xb.shape[0]):
        cs = [bf16_to_float(int(b)) for b in csb[pos[t]]]
        for h in range(Hq + Hkv):
            z = [bf16_to_float(int(b)) for b in xb[t, h * D : (h + 1) * D]]
            w = qw if h < Hq else kw
            ss = rn32(sum(Fraction(v) * Fraction(v) for v in z))
            inv = _exact_inv(ss, D, eps)
            y = [rn32(Fraction(rn32(Fraction(zz) * Fraction(inv))) * Fraction(ww)) for zz, ww in zip(z, w)]
            for j in range(half):
                ia, ib = (j, j + half) if is_neox else (2 * j, 2 * j + 1)
                c, sn = Fraction(cs[j]), Fraction(cs[half + j])
                a, b = Fraction(y[ia]), Fraction(y[ib])
                a2 = rn32(Fraction(rn32(a * c)) - Fraction(rn32(b * sn)))
                b2 = rn32(Fraction(rn32(b * c)) + Fraction(rn32(a * sn)))
                out[t, h * D + ia] = np.float32(_bf16_rn(a2)).view(np.uint32) >> 16
                out[t, h * D + ib] = np.float32(_bf16_rn(b2)).view(np.uint32) >> 16
    return out


def _qk_case(T, Hq, Hkv, D, P, seed):
    qkv, qw, kw, cs, pos = inputs.qk_norm_rope_input(T, Hq, Hkv, D, P, seed=seed)
    return inputs.bits(qkv), inputs.bits(qw), inputs.bits(kw), inputs.bits(cs), pos.numpy()


def pin_qk_rope_bruteforce():
    """Both pairings on small heads against the exact-rational transcription."""
    for is_neox in (True, False):
        xb, qw, kw, cs, pos = _qk_case(3, 2, 1, 16, 64, seed=71 + is_neox)
        got = oracle.fused_qk_norm_rope(xb, qw, kw, cs, pos, 2, 1, head_dim=16, is_neox=is_neox)
        want = _exact_qk_rope(xb, qw, kw, cs, pos, 2, 1, 16, is_neox)
        bad = np.argwhere(got != want)
        assert bad.size == 0, (is_neox, bad[:4])


def pin_qk_rope_position_zero_is_the_norm():
    """At position 0 the rotation is the identity (cos 1, sin 0), so the op is
    the per-head RMSNorm times the weight, rounded to bf16: checked against a
    float64 evaluation (within one bf16 step) and the value heads unchanged."""
    Hq, Hkv, D = 4, 2, 128
    xb, qw, kw, cs, pos = _qk_case(5, Hq, Hkv, D, 16, seed=73)
    pos[:] = 0
    got = oracle.fused_qk_norm_rope(xb, qw, kw, cs, pos, Hq, Hkv, head_dim=D)
    x = bf16_bits_to_f32(xb).astype(np.float64).reshape(5, Hq + 2 * Hkv, D)
    w = np.concatenate([np.tile(bf16_bits_to_f32(qw), (Hq, 1)), np.tile(bf16_bits_to_f32(kw), (Hkv, 1))])
    qk = x[:, : Hq + Hkv]
    ref = qk / np.sqrt((qk * qk).mean(axis=2, keepdims=True) + float(RMS_EPS)) * w[None]
    g = bf16_bits_to_f32(got).astype(np.float64).reshape(5, Hq + 2 * Hkv, D)
    assert np.all(np.abs(g[:, : Hq + Hkv] - ref) <= 2.0**-7 * np.abs(ref) + 1e-30)
    assert np.array_equal(got[:, (Hq + Hkv) * D :], xb[:, (Hq + Hkv) * D :])


def pin_qk_rope_pairings_are_a_permutation():
    """The neox pairing (j, j + D/2) and the interleaved pairing (2j, 2j + 1)
    are the same rotation on permuted dimensions: interleaving the input and
    the weights maps one result onto the other, bit for bit."""
    Hq, Hkv, D = 3, 1, 64
    xb, qw, kw, cs, pos = _qk_case(4, Hq, Hkv, D, 32, seed=75)
    perm = np.empty(D, np.int64)
    perm[0::2] = np.arange(D // 2)
    perm[1::2] = np.arange(D // 2) + D // 2          # interleaved position i holds neox dim perm[i]
    heads = Hq + 2 * Hkv
    x3 = xb.reshape(4, heads, D)
    xg = np.ascontiguousarray(x3[:, :, perm].reshape(4, heads * D))
    n = oracle.fused_qk_norm_rope(xb, qw, kw, cs, pos, Hq, Hkv, head_dim=D, is_neox=True)
    gj = oracle.fused_qk_norm_rope(xg, np.ascontiguousarray(qw[perm]), np.ascontiguousarray(kw[perm]), cs, pos,
                                   Hq, Hkv, head_dim=D, is_neox=False)
    assert np.array_equal(gj.reshape(4, heads, D), n.reshape(4, heads, D)[:, :, perm])


def pin_qk_rope_rotation_keeps_pair_norms():
    """Each rotated pair keeps its length (cos^2 + sin^2 = 1 up to the bf16
    table, 2^-7), and rotating by the angle of position p moves the pair by
    that angle: the products with the table row give back the normed pair."""
    Hq, Hkv, D = 2, 1, 128
    xb, qw, kw, cs, pos = _qk_case(6, Hq, Hkv, D, 4096, seed=77)
    z = oracle.fused_qk_norm_rope(xb, qw, kw, cs, np.zeros_like(pos), Hq, Hkv, head_dim=D)
    r = oracle.fused_qk_norm_rope(xb, qw, kw, cs, pos, Hq, Hkv, head_dim=D)
    zf = bf16_bits_to_f32(z).astype(np.float64).reshape(6, -1, D)[:, : Hq + Hkv]
    rf = bf16_bits_to_f32(r).astype(np.float64).reshape(6, -1, D)[:, : Hq + Hkv]
    h = D // 2
    nz = np.hypot(zf[..., :h], zf[..., h:])
    nr = np.hypot(rf[..., :h], rf[..., h:])
    assert np.all(np.abs(nr - nz) <= 2.0**-6 * nz + 1e-30)
    c = bf16_bits_to_f32(cs)[pos][:, None, :h].astype(np.float64)
    sn = bf16_bits_to_f32(cs)[pos][:, None, h:].astype(np.float64)
    a = rf[..., :h] * c + rf[..., h:] * sn            # rotate back
    assert np.all(np.abs(a - zf[..., :h]) <= 2.0**-5 * nz + 1e-30)


ALL_PINS = [
    pin_golden_midpoints,
    pin_group_scale_fp32,
    pin_ue8m0_packed_golden,
    pin_ue8m0_packed_decodes,
    pin_ue8m0_mx_tiles,
    pin_e4m3_roundtrip,
    pin_op_a_hand_rows,
    pin_scale_layouts,
    pin_rms_inv_chain,
    pin_rms_residual_zero,
    pin_rms_constant_row,
    pin_rms_weight_pow2,
    pin_silu_reduces_to_group_quant,
    pin_silu_zero_gate,
    pin_silu_large_negative_gate,
    pin_op_a_bruteforce,
    pin_quotient_near_midpoints,
    pin_op_a_invariants,
    pin_rms_bruteforce,
    pin_rms_sumsq,
    pin_silu_values,
    pin_silu_bruteforce,
    pin_per_token_bruteforce,
    pin_per_token_row_amax,
    pin_rms_per_token_bruteforce,
    pin_silu_per_token_bruteforce,
    pin_qk_rope_bruteforce,
    pin_qk_rope_position_zero_is_the_norm,
    pin_qk_rope_pairings_are_a_permutation,
    pin_qk_rope_rotation_keeps_pair_norms,
    pin_e4m3_structured_exact,
    pin_ue8m0,
    pin_e4m3_torch_cast,
    pin_e4m3_exhaustive_bf16,
]

__all__ = ["ALL_PINS", "near_midpoint_cases", "near_midpoint_groups", "ordinal",
           "bf16_bits_to_f32", "all_bf16_finite", "load_midpoints"] + [p.__name__ for p in ALL_PINS]
