"""Comparison rules between the CUDA library's outputs and the oracle's.

per_token_group_fp8_quant: codes and scales bit-identical.

rms_norm_per_block_quant and silu_and_mul_per_block_quant (the sum of
squares is reduced in a different order on the GPU, and CUDA's expf is not
libm's), per call:
  * non-UE8M0 scales within 1e-5 relative of the oracle's;
  * UE8M0 scales equal, except a factor-2 flip, allowed only where the
    oracle's scale before the power-of-two rounding lies within 1e-5
    (relative) of a power of two; in such a group the GPU codes are checked
    against the oracle quantising its own values with the GPU's scale, and
    all 128 elements of the group count as mismatches;
  * every code within one e4m3 step (on the monotone ordinal line) of the
    oracle's, and at most 1e-4 of the elements different at all.
"""

from __future__ import annotations

import math

import numpy as np

import oracle

SCALE_RTOL = 1e-5
CODE_FRAC = 1e-4
GROUP = 128


def ordinal(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def to_tg(s: np.ndarray, col_major: bool) -> np.ndarray:
    """Scales in [T, G] order whatever the layout they were stored in."""
    return s.T if col_major else s


def assert_exact(q_gpu, s_gpu, q_ref, s_ref, what=""):
    if not np.array_equal(s_gpu, s_ref):
        bad = np.argwhere(s_gpu != s_ref)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} scales differ, first at {i}: gpu {s_gpu[i]!r} oracle {s_ref[i]!r}")
    if not np.array_equal(q_gpu, q_ref):
        bad = np.argwhere(q_gpu != q_ref)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} codes differ, first at {i}: gpu {q_gpu[i]:#04x} oracle {q_ref[i]:#04x}")


def _near_pow2(x: np.ndarray, rtol: float) -> np.ndarray:
    m, e = np.frexp(x.astype(np.float64))
    lo = np.ldexp(0.5, e)
    hi = np.ldexp(1.0, e)
    return (np.abs(x - lo) <= rtol * x) | (np.abs(hi - x) <= rtol * x)


def check_fused(q_gpu, s_gpu_tg, q_ref, s_ref_tg, s_pre_tg, v_ref, ue8m0: bool, what="",
                group: int = GROUP) -> dict:
    """Scales in [T, G] order (G = 1 with group = the row length for the
    per-token ops).  Returns counts; raises AssertionError on failure."""
    T, C = q_ref.shape
    G = C // group
    assert q_gpu.shape == q_ref.shape and s_gpu_tg.shape == s_ref_tg.shape == (T, G), what
    flipped = np.zeros((T, G), bool)
    if not ue8m0:
        rel = np.abs(s_gpu_tg.astype(np.float64) - s_ref_tg) / s_ref_tg
        if rel.max(initial=0.0) > SCALE_RTOL:
            i = np.unravel_index(np.argmax(rel), rel.shape)
            raise AssertionError(f"{what}: scale rel err {rel[i]:.3g} at {i} (gpu {s_gpu_tg[i]!r}, oracle {s_ref_tg[i]!r})")
    else:
        diff = s_gpu_tg != s_ref_tg
        if diff.any():
            ratio = s_gpu_tg[diff].astype(np.float64) / s_ref_tg[diff]
            ok_ratio = (ratio == 2.0) | (ratio == 0.5)
            ok_pre = _near_pow2(s_pre_tg[diff], SCALE_RTOL)
            if not np.all(ok_ratio & ok_pre):
                k = np.argmin(ok_ratio & ok_pre)
                idx = tuple(np.argwhere(diff)[k])
                raise AssertionError(f"{what}: UE8M0 scale differs at {idx}: gpu {s_gpu_tg[idx]!r} "
                                     f"oracle {s_ref_tg[idx]!r} (pre-rounding {s_pre_tg[idx]!r})")
            flipped = diff

    qg = q_gpu.reshape(T, G, group)
    qr = q_ref.reshape(T, G, group).copy()
    if flipped.any():
        assert v_ref is not None, "a UE8M0 flip needs the oracle's values to re-check codes"
        vr = v_ref.reshape(T, G, group)
        for t, g in np.argwhere(flipped):
            qr[t, g] = oracle.quant_pairs(vr[t, g], np.full(group, s_gpu_tg[t, g], np.float32))
    d = np.abs(ordinal(qg) - ordinal(qr))
    if d.max(initial=0) > 1:
        i = np.unravel_index(np.argmax(d), d.shape)
        raise AssertionError(f"{what}: code off by {d[i]} e4m3 steps at {i}: gpu {qg[i]:#04x} oracle {qr[i]:#04x}")
    n_diff = int(np.count_nonzero(d)) + group * int(flipped.sum())
    budget = math.floor(CODE_FRAC * T * C)
    if n_diff > budget:
        raise AssertionError(f"{what}: {n_diff} codes differ (budget {budget} = 1e-4 of {T * C})")
    return {"codes_off_by_one": int(np.count_nonzero(d)), "ue8m0_flips": int(flipped.sum()),
            "elements": T * C}
