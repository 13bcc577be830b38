"""Seeded synthetic inputs for the FP8 quantisation epilogues and the fused
QK-norm + rotary embedding.

This module only draws numbers.  It holds none of the arithmetic of the
method (no scale, no rounding to e4m3, no norm, no SiLU), so the CPU oracle
and the CUDA path can both be fed from it without sharing any of the
computation they are compared on.

Every tensor is drawn in fp32 from a ``torch.Generator('cpu')`` seeded with a
fixed integer, in a fixed draw order, and then rounded to bf16 with torch's
round-to-nearest-even cast.  The shapes and value distributions stand in for
the shape sweeps over public model configurations that the RFC "[RFC]: Using
Helion for Selected vLLM CustomOps" measures (section "Standalone Kernel
Performance with Extensive Shape Sweeps on H100 and B200"); the shape lists
themselves are not published, so the recipes below are synthetic.
"""

from __future__ import annotations

import torch

GROUP = 128

# Seeds of the five workload recipes.  A sweep point i of a recipe uses
# ``base + i``; the same seed always yields the same tensor.
SEED_SMALL = 1000
SEED_RMS_X, SEED_RMS_W, SEED_RMS_R = 2000, 2001, 2002
SEED_SILU = 3000
SEED_SWEEP = 4000
SEED_MIX_SIGMA, SEED_MIX_X = 5000, 5001
SEED_QK = 6000

SWEEP_T = (1, 4, 16, 64, 256, 1024, 4096, 16384)
MIX_T = (1, 8, 64, 512, 4096, 16384)
SWEEP_H = 7168
MIX_H = 5120
MIX_I = 25600


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    return g


def normal_f32(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    """fp32 N(0, std^2) tensor, seeded."""
    t = torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def bf16(t: torch.Tensor) -> torch.Tensor:
    """Round an fp32 tensor to bf16 (round to nearest, ties to even)."""
    return t.to(torch.bfloat16).contiguous()


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (a view, no copy)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def from_bits(a) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    import numpy as np

    return torch.from_numpy(np.ascontiguousarray(a).view("int16")).view(torch.bfloat16)


# --------------------------------------------------------------------------
# Small per-token-group case: 16 random rows + 4 hand-set rows, H = 512.
# --------------------------------------------------------------------------

# Values of the rounding-midpoint group (row 18, group 0).  All are exact in
# bf16.  With amax = 448 the group scale is exactly 1, so each value is its
# own quotient; most sit exactly half way between two e4m3 neighbours.
MIDPOINT_VALUES = (
    448.0,
    1.0625,
    1.1875,
    -1.1875,
    17.0,
    19.0,
    248.0,
    432.0,
    1.5 * 2.0**-9,
    2.5 * 2.0**-9,
    2.0**-10,
    7.5 * 2.0**-9,
)


def hand_rows(H: int = 512, seed: int = SEED_SMALL + 1) -> torch.Tensor:
    """The four hand-set rows (bf16 [4, H], H a multiple of 512).

    row 0: group 0 is all zeros (alternating +0.0 / -0.0), the other groups N(0,1).
    row 1: group 0 is N(0,1) with one entry set to +1e4 (bf16 9984), group 1 the
           same with -1e4, further groups N(0,1) with an outlier at another slot.
    row 2: rounding midpoints: group 0 = MIDPOINT_VALUES then +0.0/-0.0,
           group 1 = 2 * group 0, group 2 = -group 0, group 3 = -group 1
           (further groups repeat the pattern).
    row 3: small magnitudes: group 0 = one 448 among U(-0.02, 0.02) values,
           group 1 = bf16 subnormals with mixed signs, group 2 = values of
           order 1e-10 with amax 2e-10 (just above the 1e-10 floor),
           group 3 = N(0,1) * 1e-3.
    """
    assert H % (4 * GROUP) == 0
    g = _gen(seed)
    G = H // GROUP
    out = torch.zeros(4, H, dtype=torch.float32)

    # row 0
    r = torch.randn(H, generator=g)
    z = torch.zeros(GROUP)
    z[1::2] = -0.0
    r[:GROUP] = z
    out[0] = r

    # row 1
    r = torch.randn(H, generator=g)
    base = torch.randn(GROUP, generator=g)
    r[0:GROUP] = base
    r[5] = 1.0e4
    r[GROUP : 2 * GROUP] = base
    r[GROUP + 5] = -1.0e4
    for gi in range(2, G):
        r[gi * GROUP + (17 * gi) % GROUP] = 1.0e4 if gi % 2 == 0 else -1.0e4
    out[1] = r

    # row 2
    mid = torch.zeros(GROUP)
    mid[1::2] = -0.0
    mid[: len(MIDPOINT_VALUES)] = torch.tensor(MIDPOINT_VALUES)
    pattern = [mid, 2.0 * mid, -mid, -(2.0 * mid)]
    for gi in range(G):
        out[2, gi * GROUP : (gi + 1) * GROUP] = pattern[gi % 4]

    # row 3
    r = torch.empty(H)
    u = (torch.rand(GROUP, generator=g) * 2.0 - 1.0) * 0.02
    u[0] = 448.0
    r[0:GROUP] = u
    k = torch.randint(1, 128, (GROUP,), generator=g).to(torch.float32)
    sign = torch.where(torch.rand(GROUP, generator=g) < 0.5, -1.0, 1.0)
    r[GROUP : 2 * GROUP] = sign * k * (2.0**-133)  # exact bf16 subnormals
    t = torch.randn(GROUP, generator=g) * 0.5e-10
    t = t.clamp(-1.9e-10, 1.9e-10)
    t[3] = 2.0e-10
    r[2 * GROUP : 3 * GROUP] = t
    r[3 * GROUP :] = torch.randn(H - 3 * GROUP, generator=g) * 1e-3
    out[3] = r
    return bf16(out)


def small_group_quant_input(seed: int = SEED_SMALL) -> torch.Tensor:
    """bf16 [20, 512]: rows 0-15 N(0,1), rows 16-19 the hand-set rows."""
    x = normal_f32((16, 512), seed)
    return torch.cat([bf16(x), hand_rows(512, seed + 1)], dim=0).contiguous()


# --------------------------------------------------------------------------
# RMSNorm case: x [T, H] N(0,1), weight 1 + 0.1 N(0,1), residual N(0, 0.5^2).
# --------------------------------------------------------------------------


def rms_weight(H: int, seed: int = SEED_RMS_W) -> torch.Tensor:
    return bf16(1.0 + normal_f32((H,), seed, 0.1))


def rms_input(T: int = 256, H: int = 4096, seeds=(SEED_RMS_X, SEED_RMS_W, SEED_RMS_R)):
    """Returns (x, weight, residual), all bf16."""
    sx, sw, sr = seeds
    return (
        bf16(normal_f32((T, H), sx)),
        rms_weight(H, sw),
        bf16(normal_f32((T, H), sr, 0.5)),
    )


# --------------------------------------------------------------------------
# SiLU-and-mul case: x [T, 2I], gate half N(0, 2^2), up half N(0, 1).
# --------------------------------------------------------------------------


def silu_input(T: int = 1024, I: int = 12288, seed: int = SEED_SILU) -> torch.Tensor:
    g = _gen(seed)
    x = torch.empty(T, 2 * I, dtype=torch.float32)
    x[:, :I] = torch.randn(T, I, generator=g) * 2.0
    x[:, I:] = torch.randn(T, I, generator=g)
    return bf16(x)


# --------------------------------------------------------------------------
# Heavy-tailed sweep: H = 7168, N(0,1) with 0.1 % of entries (drawn without
# replacement) multiplied by 100.
# --------------------------------------------------------------------------


def heavy_tailed_input(T: int, H: int = SWEEP_H, seed: int = SEED_SWEEP) -> torch.Tensor:
    g = _gen(seed)
    x = torch.randn(T * H, generator=g)
    n_out = int(round(0.001 * T * H))
    if n_out:
        pos = torch.randperm(T * H, generator=g)[:n_out]
        x[pos] *= 100.0
    return bf16(x.view(T, H))


def sweep_seed(T: int) -> int:
    return SEED_SWEEP + SWEEP_T.index(T) if T in SWEEP_T else SEED_SWEEP + 100 + T


# --------------------------------------------------------------------------
# Qwen3-32B-shaped mix: per-channel std sigma_c = exp(N(0,1)) drawn once per
# column, x[t, c] = sigma_c * N(0,1).
# --------------------------------------------------------------------------


def channel_sigma(C: int, seed: int = SEED_MIX_SIGMA) -> torch.Tensor:
    return torch.exp(normal_f32((C,), seed))


def lognormal_channel_input(T: int, C: int, seed_x: int, seed_sigma: int = SEED_MIX_SIGMA) -> torch.Tensor:
    sigma = channel_sigma(C, seed_sigma)
    x = normal_f32((T, C), seed_x)
    x.mul_(sigma)
    return bf16(x)


def mix_seed(T: int) -> int:
    return SEED_MIX_X + MIX_T.index(T) if T in MIX_T else SEED_MIX_X + 100 + T


# --------------------------------------------------------------------------
# The same two recipes drawn on a CUDA device (for timing at sizes where
# drawing on the host would take longer than the measurement): a seeded
# device generator, the same distributions, bf16 on the device.  The values
# differ from the host draws of the same seed.
# --------------------------------------------------------------------------


def device_heavy_tailed_input(T: int, H: int, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn(T * H, generator=g, device=device)
    n_out = int(round(0.001 * T * H))
    if n_out:
        pos = torch.randperm(T * H, generator=g, device=device)[:n_out]
        x[pos] *= 100.0
    return x.view(T, H).to(torch.bfloat16)


def device_lognormal_channel_input(T: int, C: int, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device).manual_seed(seed)
    sigma = torch.exp(torch.randn(C, generator=g, device=device))
    x = torch.randn(T, C, generator=g, device=device)
    x.mul_(sigma)
    return x.to(torch.bfloat16)


# --------------------------------------------------------------------------
# fused_qk_norm_rope case, Qwen3-32B attention shape: 64 query heads and 8
# key/value heads of 128 values per token; query/key activations with
# per-channel spread (lognormal channel std), value heads N(0,1); norm
# weights 1 + 0.1 N(0,1); positions uniform in [0, P); the rotary table a
# model holds for those positions: row p = (cos(p f_j), sin(p f_j)), j < D/2,
# f_j = base^(-2j/D), base 1e6 (Qwen3), computed in float64 and rounded to
# bf16.  The table is an input of the op, like the weights.
# --------------------------------------------------------------------------

QK_HQ, QK_HKV, QK_D, QK_P = 64, 8, 128, 40960


def rotary_table(P: int, D: int = QK_D, base: float = 1e6) -> torch.Tensor:
    j = torch.arange(D // 2, dtype=torch.float64)
    freq = base ** (-2.0 * j / D)
    ang = torch.arange(P, dtype=torch.float64)[:, None] * freq[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.bfloat16).contiguous()


def qk_norm_rope_input(T: int, Hq: int = QK_HQ, Hkv: int = QK_HKV, D: int = QK_D, P: int = QK_P,
                       seed: int = SEED_QK):
    """Returns (qkv bf16 [T, (Hq + 2 Hkv) D], q_weight bf16 [D], k_weight bf16 [D],
    cos_sin bf16 [P, D], positions int64 [T])."""
    g = _gen(seed)
    nqk = (Hq + Hkv) * D
    sigma = torch.exp(torch.randn(nqk, generator=g) * 0.5)
    qkv = torch.randn(T, (Hq + 2 * Hkv) * D, generator=g)
    qkv[:, :nqk] *= sigma
    qw = 1.0 + 0.1 * torch.randn(D, generator=g)
    kw = 1.0 + 0.1 * torch.randn(D, generator=g)
    pos = torch.randint(0, P, (T,), generator=g, dtype=torch.int64)
    return bf16(qkv), bf16(qw), bf16(kw), rotary_table(P, D), pos


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("annotations", "torch")]
