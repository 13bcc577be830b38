"""Parity of the CUDA library with the CPU oracle, through the C ABI.

per_token_group_fp8_quant is compared bit for bit; the fused ops with the
rules of tolerance.py.  Inputs are the seeded workloads of
fp8_token_group_bf16_b300.inputs; tensors too large for the oracle are
compared on sampled rows (rows are independent, so the oracle run on those
rows alone gives their exact expected values), in the same launch
configuration the benchmark times.
"""

import functools
import os

import numpy as np
import pytest
import torch

import oracle
import pins
from fp8_token_group_bf16_b300 import inputs
from gpu_util import gpu_group_quant, gpu_rms, gpu_silu, require_gpu, sample_rows
from tolerance import assert_exact, check_fused, to_tg

pytestmark = pytest.mark.gpu

VARIANTS = [(u, c) for u in (False, True) for c in (False, True)]
VID = [f"{'ue8m0' if u else 'fp32'}-{'col' if c else 'row'}" for u, c in VARIANTS]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@functools.lru_cache(maxsize=2)
def _heavy_bits(T):
    return inputs.bits(inputs.heavy_tailed_input(T, inputs.SWEEP_H, inputs.sweep_seed(T)))


# ------------------------------------------------------- op A (exact) ----


def _oracle_a(xb, ue8m0):
    q, s, _ = oracle.per_token_group_quant(xb, ue8m0=ue8m0, col_major=False)
    return q, s


@pytest.mark.parametrize("ue8m0,col", VARIANTS, ids=VID)
def test_group_quant_small_case_with_hand_rows(ue8m0, col):
    xb = inputs.bits(inputs.small_group_quant_input())
    q, s = gpu_group_quant(xb, ue8m0, col)
    qr, sr, _ = oracle.per_token_group_quant(xb, ue8m0=ue8m0, col_major=col)
    assert_exact(q, s, qr, to_tg(sr, col), "small case")
    # the hand-derived midpoint codes, straight from the golden file
    golden = [c for _, c in pins.load_midpoints()][:-2]
    assert q[18, : len(golden)].tolist() == golden


@pytest.mark.parametrize("ue8m0,col", VARIANTS, ids=VID)
@pytest.mark.parametrize("T", inputs.SWEEP_T)
def test_group_quant_heavy_tailed_sweep(T, ue8m0, col):
    xb = _heavy_bits(T)
    q, s = gpu_group_quant(xb, ue8m0, col)
    rows = sample_rows(T, 512, seed=T)
    qr, sr = _oracle_a(np.ascontiguousarray(xb[rows]), ue8m0)
    assert_exact(q[rows], s[rows], qr, sr, f"T={T}")


def test_group_quant_near_midpoint_quotients():
    xb = pins.near_midpoint_groups(pins.near_midpoint_cases(n_scales=3000, seed=9))
    for ue8m0 in (False, True):
        q, s = gpu_group_quant(xb, ue8m0)
        qr, sr = _oracle_a(xb, ue8m0)
        assert_exact(q, s, qr, sr, f"near midpoints ue8m0={ue8m0}")


def _quotient_domain_groups(stride: int) -> np.ndarray:
    """Groups [amax, x_1 .. x_127] for every stride-th positive finite bf16
    amax and every bf16 x with |x| <= amax (alternating signs): the whole
    domain of the quotient x / RN32(amax/448) that the op can meet."""
    b = pins.all_bf16_finite()
    pos = b[(b >> 15) == 0]
    vals = pins.bf16_bits_to_f32(pos)
    order = np.argsort(vals, kind="stable")
    pos, vals = pos[order], vals[order]
    groups = []
    for i in range(1, len(pos), stride):
        xs = pos[: i + 1]
        xs = np.where(np.arange(xs.size) % 2 == 1, xs | np.uint16(0x8000), xs).astype(np.uint16)
        n = -(-xs.size // 127)
        padded = np.resize(xs, n * 127).reshape(n, 127)
        g = np.empty((n, 128), np.uint16)
        g[:, 0] = pos[i]
        g[:, 1:] = padded
        groups.append(g)
    allg = np.concatenate(groups)
    pad = (-allg.shape[0]) % 8
    if pad:
        allg = np.concatenate([allg, allg[:pad]])
    return allg.reshape(-1, 8 * 128)


def test_group_quant_quotient_domain():
    """Every positive bf16 amax with every bf16 |x| <= amax (537 M values);
    FP8Q_QUICK=1 takes every 61st amax instead, for quick local runs."""
    stride = 61 if os.environ.get("FP8Q_QUICK") else 1
    xb = _quotient_domain_groups(stride)
    for ue8m0 in (False, True):
        q, s = gpu_group_quant(xb, ue8m0)
        qr, sr = _oracle_a(xb, ue8m0)
        assert_exact(q, s, qr, sr, f"quotient domain ue8m0={ue8m0}")


@pytest.mark.parametrize("T,H", [(1, 128), (2, 256), (3, 384), (5, 640), (37, 7168), (1000, 128),
                                 (7, 1152), (129, 896), (4097, 256)])
@pytest.mark.parametrize("ue8m0,col", VARIANTS, ids=VID)
def test_group_quant_ragged_shapes(T, H, ue8m0, col):
    xb = inputs.bits(inputs.heavy_tailed_input(T, H, seed=77 + T + H))
    q, s = gpu_group_quant(xb, ue8m0, col)
    qr, sr = _oracle_a(xb, ue8m0)
    assert_exact(q, s, qr, sr, f"T={T} H={H}")


# ------------------------------------------- e4m3 conversion on its own --


def test_f32_to_e4m3_conversion():
    import fp8_token_group_bf16_b300 as fq

    rng = np.random.default_rng(1)
    v = np.concatenate([
        pins.bf16_bits_to_f32(pins.all_bf16_finite()),
        pins.structured_f32(),
        rng.integers(0, 2**32, size=1 << 24, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    v = v[~np.isnan(v)]
    got = fq.f32_to_e4m3(torch.from_numpy(v).cuda()).cpu().numpy()
    want = oracle.f32_to_e4m3(v)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (bad.size, v[bad[:4]], got[bad[:4]], want[bad[:4]])


def test_f32_to_e4m3_all_fp32_patterns():
    """Every non-NaN fp32 bit pattern (2^32); FP8Q_QUICK=1 takes every 61st
    pattern instead, for quick local runs."""
    import fp8_token_group_bf16_b300 as fq

    step = 61 if os.environ.get("FP8Q_QUICK") else 1
    chunk = 1 << 26
    for start in range(0, 1 << 32, chunk * step):
        u = np.arange(start, min(start + chunk * step, 1 << 32), step, dtype=np.uint64).astype(np.uint32)
        v = u.view(np.float32)
        v = v[~np.isnan(v)]
        got = fq.f32_to_e4m3(torch.from_numpy(v).cuda()).cpu().numpy()
        want = oracle.f32_to_e4m3(v)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (start, bad.size, v[bad[:4]], got[bad[:4]], want[bad[:4]])


def test_group_scale_every_fp32_significand():
    """The scale from an fp32 group maximum (ops B and C meet any fp32 amax):
    every fp32 significand at binades spread over the range (the division
    scales exactly with the exponent while the quotient is normal), near the
    floor, and both UE8M0 modes, against the oracle's IEEE division."""
    import fp8_token_group_bf16_b300 as fq

    sig = np.arange(1 << 23, dtype=np.uint32) | np.uint32(127 << 23)        # [1, 2)
    for e in (-100, -61, -60, -34, -1, 0, 37, 100):
        a = (sig.view(np.float32) * np.float32(2.0 ** e)).astype(np.float32)
        for ue8m0 in (False, True):
            got = fq.group_scale(torch.from_numpy(a).cuda(), ue8m0=ue8m0).cpu().numpy()
            want = oracle.group_scale(a, ue8m0=ue8m0)
            bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
            assert bad.size == 0, (e, ue8m0, bad.size, a[bad[:3]], got[bad[:3]], want[bad[:3]])
    rng = np.random.default_rng(4)
    a = np.concatenate([rng.random(1 << 16).astype(np.float32) * np.float32(2e-10), np.zeros(4, np.float32),
                        np.array([1e-10, 3.0e38], np.float32)])
    for ue8m0 in (False, True):
        for eps in (1e-10, 1e-30):
            got = fq.group_scale(torch.from_numpy(a).cuda(), eps=eps, ue8m0=ue8m0).cpu().numpy()
            want = oracle.group_scale(a, eps=np.float32(eps), ue8m0=ue8m0)
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (ue8m0, eps)


def _quotient_pairs(rng, n_random=1 << 18, n_hard=20000):
    """(v, s) pairs: scales RN32(amax / 448) over the binades with values up to
    amax; pairs whose quotient lies within about 2^-47 (relative) of a
    midpoint between two fp32 values (for an odd scale significand S and a
    small odd t, N = 2^24 + (t S^-1 mod 2^24) makes S N = V 2^24 + t, so
    v = V, s = S give v/s = N 2^-24 (1 - t / (S N)), scaled); signed zeros
    and values whose quotient underflows."""
    amax = (rng.uniform(1, 2, n_random) * 2.0 ** rng.integers(-60, 60, n_random)).astype(np.float32)
    s = (amax.astype(np.float64) / 448).astype(np.float32)
    v = (amax * rng.uniform(-1, 1, n_random)).astype(np.float32)
    vs, ss = [v], [s]
    hv, hs = [], []
    mod = 1 << 24
    while len(hv) < n_hard:
        S = int(rng.integers(1 << 22, 1 << 23)) * 2 + 1
        t = int(rng.choice([-3, -1, 1, 3]))
        N = mod + (t * pow(S, -1, mod)) % mod
        V = (S * N - t) // mod
        if V >= mod:
            continue
        a = int(rng.integers(-40, 30))
        shift = int(rng.choice([-9, -3, 0, 4, 7]))
        sign = 1.0 if rng.random() < 0.5 else -1.0
        hv.append(sign * float(V) * 2.0 ** (a - 23 + shift))
        hs.append(float(S) * 2.0 ** (a - 23))
    vs.append(np.array(hv, np.float32))
    ss.append(np.array(hs, np.float32))
    z = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-40, -1e-40, 2.0 ** -126, -(2.0 ** -126)], np.float32)
    vs.append(z)
    ss.append(np.full(z.size, 3.0 / 448, np.float32))
    return np.concatenate(vs), np.concatenate(ss)


def test_quotient_of_arbitrary_fp32_values():
    """The quotient every kernel takes for a non-power-of-two scale, on fp32
    values (ops B and C quantise fp32 values, not bf16 ones), bit for bit
    against the oracle's division, next to rounding midpoints included."""
    import fp8_token_group_bf16_b300 as fq

    v, s = _quotient_pairs(np.random.default_rng(15))
    got = fq.quant_pairs(torch.from_numpy(v).cuda(), torch.from_numpy(s).cuda()).cpu().numpy()
    want = oracle.quant_pairs(v, s)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (bad.size, v[bad[:4]], s[bad[:4]], got[bad[:4]], want[bad[:4]])
    assert (want == 0x80).any() and (want == 0x00).any()


# ----------------------------------------------- op B (rms + quant) ----


def _check_rms(xb, wb, rb, ue8m0, col, rows=None, what=""):
    q, s, rout = gpu_rms(xb, wb, rb, ue8m0, col)
    if rows is None:
        rows = np.arange(xb.shape[0])
    xs = np.ascontiguousarray(xb[rows])
    rs = np.ascontiguousarray(rb[rows]) if rb is not None else None
    qr, sr, spr, _, ror, vr = oracle.rms_norm_per_block_quant(xs, wb, rs, ue8m0=ue8m0, want_values=True)
    if rb is not None:
        assert np.array_equal(rout[rows], ror), f"{what}: residual output differs"
    return check_fused(q[rows], s[rows], qr, sr, spr, vr, ue8m0, what)


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
@pytest.mark.parametrize("ue8m0,col", VARIANTS, ids=VID)
def test_rms_4096(residual, ue8m0, col):
    x, w, r = inputs.rms_input(256, 4096)
    _check_rms(inputs.bits(x), inputs.bits(w), inputs.bits(r) if residual else None, ue8m0, col,
               what=f"rms 256x4096 residual={residual}")


@pytest.mark.parametrize("T", inputs.MIX_T)
def test_rms_qwen3_mix(T):
    x = inputs.lognormal_channel_input(T, inputs.MIX_H, inputs.mix_seed(T))
    w = inputs.rms_weight(inputs.MIX_H)
    rows = sample_rows(T, 512, seed=T)
    _check_rms(inputs.bits(x), inputs.bits(w), None, True, False, rows, what=f"rms mix T={T}")


@pytest.mark.parametrize("T,H", [(1, 128), (3, 384), (37, 1152), (2, 8192), (5, 16384),
                                 (3, 24576), (2, 32768), (300, 256), (700, 8192), (1, 8320)])
@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
def test_rms_ragged_shapes(T, H, residual):
    x, w, r = inputs.rms_input(T, H, seeds=(900 + T, 901 + H, 902))
    for ue8m0, col in VARIANTS:
        _check_rms(inputs.bits(x), inputs.bits(w), inputs.bits(r) if residual else None, ue8m0, col,
                   what=f"rms T={T} H={H}")


def test_rms_degenerate_rows():
    """All-zero row (inv = 1/sqrt(eps), every value 0, floor scale) and a
    constant row (every code +-448)."""
    H = 1024
    x = torch.zeros(4, H)
    x[1] = 0.75
    x[2] = -3.0
    x[3, ::2] = 1e-20
    xb = inputs.bits(inputs.bf16(x))
    wb = inputs.bits(inputs.bf16(torch.ones(H)))
    for ue8m0, col in VARIANTS:
        q, s, _ = gpu_rms(xb, wb, None, ue8m0, col)
        qr, sr, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, None, ue8m0=ue8m0)
        assert_exact(q, s, qr, sr, "degenerate rows")


# ---------------------------------------------- op C (silu + quant) ----


def _check_silu(xb, ue8m0, col, rows=None, what=""):
    q, s = gpu_silu(xb, ue8m0, col)
    if rows is None:
        rows = np.arange(xb.shape[0])
    qr, sr, spr, vr = oracle.silu_and_mul_per_block_quant(np.ascontiguousarray(xb[rows]), ue8m0=ue8m0,
                                                          want_values=True)
    return check_fused(q[rows], s[rows], qr, sr, spr, vr, ue8m0, what)


def test_silu_12288_ue8m0_col_major():
    xb = inputs.bits(inputs.silu_input(1024, 12288))
    _check_silu(xb, True, True, what="silu 1024x12288")


@pytest.mark.parametrize("ue8m0,col", VARIANTS, ids=VID)
def test_silu_12288_other_variants(ue8m0, col):
    xb = inputs.bits(inputs.silu_input(64, 12288, seed=inputs.SEED_SILU + 1))
    _check_silu(xb, ue8m0, col, what="silu 64x12288")


@pytest.mark.parametrize("T", inputs.MIX_T)
def test_silu_qwen3_mix(T):
    x = inputs.lognormal_channel_input(T, 2 * inputs.MIX_I, inputs.mix_seed(T) + 50)
    rows = sample_rows(T, 128, seed=T)
    _check_silu(inputs.bits(x), True, False, rows, what=f"silu mix T={T}")


def test_silu_reduces_to_group_quant():
    """gate >= 20 and up = 1: silu(a) * 1 == a exactly, so the result must be
    the per-group quantisation of the gate half, bit for bit."""
    rng = np.random.default_rng(5)
    T, I = 64, 7168
    a = (20.0 + np.abs(rng.standard_normal((T, I))) * 40.0).astype(np.float32)
    ab = inputs.bits(inputs.bf16(torch.from_numpy(a)))
    xb = np.concatenate([ab, inputs.bits(inputs.bf16(torch.ones(T, I)))], axis=1)
    for ue8m0, col in VARIANTS:
        q, s = gpu_silu(xb, ue8m0, col)
        qr, sr = _oracle_a(ab, ue8m0)
        assert_exact(q, s, qr, sr, "silu reduction")


@pytest.mark.parametrize("T,I", [(1, 128), (3, 384), (37, 1152), (5, 640), (1000, 256)])
def test_silu_ragged_shapes(T, I):
    xb = inputs.bits(inputs.silu_input(T, I, seed=700 + T + I))
    for ue8m0, col in VARIANTS:
        _check_silu(xb, ue8m0, col, what=f"silu T={T} I={I}")


def test_silu_extreme_gates():
    """Gates far below -88 (exp overflows, silu -> -0), zeros, and +-0 ups."""
    T, I = 4, 256
    a = torch.randn(T, I, generator=torch.Generator().manual_seed(3)) * 50.0
    a[0] = -200.0
    a[1, ::3] = 0.0
    b = torch.randn(T, I, generator=torch.Generator().manual_seed(4))
    b[2, ::2] = -0.0
    xb = inputs.bits(inputs.bf16(torch.cat([a, b], dim=1)))
    for ue8m0, col in VARIANTS:
        _check_silu(xb, ue8m0, col, what="silu extreme gates")


# ------------------------------------ op B: the exact sum of squares ----


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
@pytest.mark.parametrize("ue8m0,col", VARIANTS, ids=VID)
def test_rms_bit_exact(residual, ue8m0, col):
    """The GPU adds the squares without rounding error and rounds once, so
    away from fp32 underflow op B equals the oracle bit for bit."""
    x, w, r = inputs.rms_input(256, 4096)
    xb, wb, rb = inputs.bits(x), inputs.bits(w), inputs.bits(r) if residual else None
    q, s, rout = gpu_rms(xb, wb, rb, ue8m0, col)
    qr, sr, _, _, ror = oracle.rms_norm_per_block_quant(xb, wb, rb, ue8m0=ue8m0, col_major=col)
    assert_exact(q, s, qr, to_tg(sr, col), f"rms residual={residual}")
    if residual:
        assert np.array_equal(rout, ror)


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
def test_rms_single_wave_grids_alternating_block_sizes(residual):
    """Rows of 4096, 5120 and 8192 values run one kernel with blocks of 128,
    160 and 256 threads.  A grid that fits in one wave is spread evenly by
    padding its CTAs with warps that own no group (T = 512, 300, 444 and
    768 here: 256, 320, 320 and 160 threads), which leave at once and must
    neither hold up the row barrier nor write; T = 256, 1000 and 888 are not
    padded.  Interleaving the sizes checks that each launch takes its own
    block."""
    for T, H in [(256, 4096), (512, 5120), (300, 8192), (256, 4096), (1000, 4096), (888, 5120), (444, 5120),
                 (768, 4096), (512, 5120)]:
        x, w, r = inputs.rms_input(T, H, seeds=(8100 + T, 8101 + H, 8102))
        xb, wb, rb = inputs.bits(x), inputs.bits(w), inputs.bits(r) if residual else None
        q, s, rout = gpu_rms(xb, wb, rb, True, False)
        qr, sr, _, _, ror = oracle.rms_norm_per_block_quant(xb, wb, rb, ue8m0=True)
        assert_exact(q, s, qr, sr, f"rms single wave T={T} H={H} residual={residual}")
        if residual:
            assert np.array_equal(rout, ror)


@pytest.mark.parametrize("H", [4096, 896])
@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32", "ue8m0"])
def test_rms_signed_zeros_and_underflowing_quotients(ue8m0, H):
    """Signed zeros of x and of the weight give v = -0 or +0, whose codes are
    0x80 and 0x00; negative subnormal inputs give quotients that underflow to
    -0.  The quotient steps must keep those signs, per group and per token
    (a CTA per row at H = 4096, a warp per row at H = 896)."""
    import fp8_token_group_bf16_b300 as fq

    T = 8
    xb = inputs.bits(inputs.bf16(torch.randn(T, H, generator=torch.Generator().manual_seed(8800))))
    xb[:, ::7] = 0x8000             # -0
    xb[:, 3::7] = 0x0000            # +0
    xb[1, 5::11] = 0x8001           # the smallest negative subnormal
    xb[2, 6::13] = 0x0001
    wb = inputs.bits(inputs.rms_weight(H))
    wb[::13] |= 0x8000              # negative weights
    wb[::17] = 0x8000               # -0 weights
    q, s, _ = gpu_rms(xb, wb, None, ue8m0, False)
    qr, sr, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, None, ue8m0=ue8m0)
    assert_exact(q, s, qr, sr, f"signed zeros ue8m0={ue8m0}")
    assert (qr == 0x80).any() and (qr == 0x00).any()
    xd, wd = inputs.from_bits(xb).cuda(), inputs.from_bits(wb).cuda()
    qt, st = fq.rms_norm_dynamic_per_token_quant(xd, wd, None, ue8m0=ue8m0)
    torch.cuda.synchronize()
    qtr, str_, _, _, _ = oracle.rms_norm_dynamic_per_token_quant(xb, wb, None, ue8m0=ue8m0)
    assert np.array_equal(st.cpu().numpy().reshape(-1), str_)
    assert np.array_equal(qt.view(torch.uint8).cpu().numpy(), qtr)


@pytest.mark.parametrize("T,H", [(3, 24576), (512, 5120), (37, 1152), (2, 32768),
                                 # wide CTAs (65 to 256 groups), one wave and the prefetching build
                                 (100, 8320), (300, 24576), (150, 32768)])
def test_rms_bit_exact_shapes(T, H):
    x = inputs.lognormal_channel_input(T, H, 6000 + T)
    w = inputs.rms_weight(H)
    xb, wb = inputs.bits(x), inputs.bits(w)
    q, s, _ = gpu_rms(xb, wb, None, True, False)
    qr, sr, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, None, ue8m0=True)
    assert_exact(q, s, qr, sr, f"rms T={T} H={H}")


@pytest.mark.parametrize("T,H,residual", [(1100, 4096, True), (1024, 5120, False), (2048, 8192, True),
                                          (1500, 384, True), (1031, 1152, False), (64, 16384, True),
                                          (33, 12288, False), (9, 32768, True), (17, 20480, False),
                                          (400, 12288, False), (200, 20480, False), (160, 32768, False)])
def test_rms_many_rows_bit_exact(T, H, residual):
    """Larger launches, ragged group counts, rows of 1, 2 and 4 groups per quad,
    and (T > 64 without the residual) their builds that prefetch a later row
    into L2 once the grid outlasts the CTAs resident at once."""
    x, w, r = inputs.rms_input(T, H, seeds=(910 + T, 911 + H, 912))
    xb, wb, rb = inputs.bits(x), inputs.bits(w), inputs.bits(r) if residual else None
    for ue8m0, col in VARIANTS:
        q, s, rout = gpu_rms(xb, wb, rb, ue8m0, col)
        qr, sr, _, _, ror = oracle.rms_norm_per_block_quant(xb, wb, rb, ue8m0=ue8m0, col_major=col)
        assert_exact(q, s, qr, to_tg(sr, col), f"rms T={T} H={H} residual={residual}")
        if residual:
            assert np.array_equal(rout, ror)


# ----------------------------------- the SiLU arithmetic on its own ----


def _ulp_gap(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """Distance in fp32 steps between two fp32 arrays (same sign assumed
    where both are nonzero; a sign change counts through zero)."""
    def ordinal(v):
        i = v.view(np.int32).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)
    return np.abs(ordinal(x) - ordinal(y))


def test_silu_mul_against_oracle_every_bf16_gate():
    """silu(a) * b for every finite bf16 gate a, with b = 1 and with random
    b: the GPU's exponential (2^(x log2 e) with a corrected product) and
    quotient against the oracle's libm expf and IEEE division.  Both sides are
    within a few ulp of the exact value; the gap is bounded here."""
    import fp8_token_group_bf16_b300 as fq

    a = pins.bf16_bits_to_f32(pins.all_bf16_finite())
    rng = np.random.default_rng(3)
    stats = []
    for b in (np.ones_like(a), rng.standard_normal(a.size).astype(np.float32)):
        got = fq.silu_mul(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()).cpu().numpy()
        want = oracle.silu_mul(a, b)
        gap = _ulp_gap(got, want)
        # values below 1e-30 in magnitude (gates below about -64) quantise to a
        # zero code in any group (the smallest nonzero code is 2^-9 s, s >= 2.2e-13);
        # there the GPU's approximate reciprocal may flush, so only the size is checked
        norm = np.abs(want) >= 1e-30
        assert gap[norm].max() <= 4, (gap[norm].max(), a[norm][np.argmax(gap[norm])])
        assert np.all(np.abs(got[~norm]) < 1e-30)
        # most values agree exactly
        assert np.count_nonzero(gap[norm]) <= 0.05 * norm.sum(), np.count_nonzero(gap[norm]) / norm.sum()
        stats.append((int(gap[norm].max()), float(np.count_nonzero(gap[norm]) / norm.sum())))
    print("silu_mul vs oracle: (max ulp gap, fraction differing) per b:", stats)


def test_silu_mul_against_oracle_random_fp32_gates():
    """The same on a million fp32 gates that are not bf16 values (uniform in
    [-90, 90] and N(0, 4)), where the exponential's argument uses all 24 bits."""
    import fp8_token_group_bf16_b300 as fq

    rng = np.random.default_rng(9)
    a = np.concatenate([rng.uniform(-90, 90, 1 << 19), rng.standard_normal(1 << 19) * 4]).astype(np.float32)
    b = rng.standard_normal(a.size).astype(np.float32)
    got = fq.silu_mul(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()).cpu().numpy()
    want = oracle.silu_mul(a, b)
    norm = np.abs(want) >= 1e-30
    gap = _ulp_gap(got, want)
    # off the bf16 grid the exponential's argument carries all 24 bits and
    # ex2.approx's own error shows more: a looser bound than on the op's inputs
    assert gap[norm].max() <= 8, (gap[norm].max(), a[norm][np.argmax(gap[norm])])
    assert np.all(np.abs(got[~norm]) < 1e-30)
    assert np.count_nonzero(gap[norm]) <= 0.25 * norm.sum()
    print("silu_mul vs oracle, fp32 gates: max ulp gap", int(gap[norm].max()),
          "fraction differing", float(np.count_nonzero(gap[norm]) / norm.sum()))
