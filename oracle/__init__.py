"""Python access to the CPU oracle (liboracle.so, built from fp8q_oracle.c).

TEST INFRASTRUCTURE ONLY.  Imported by the tests, by the smoke check and by
the benchmark's CPU-baseline / reference leg; never by the product package.
The oracle shares no code with the CUDA library: it is plain single-threaded
C, compiled here with gcc, and every function states the arithmetic it
follows in fp8q_oracle.c.

Arrays are numpy: bf16 as uint16 bit patterns, e4m3 as uint8 codes, scales
as float32.  Scale layout: ``col_major=False`` -> s[t*G + g],
``col_major=True`` -> s[g*T + t].
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8q_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

SCALE_EPS = np.float32(1e-10)
RMS_EPS = np.float32(1e-6)

CFLAGS = [
    "-O2",
    "-std=c11",
    "-fPIC",
    "-shared",
    "-ffp-contract=off",
    "-fno-fast-math",
    "-frounding-math",
    "-fexcess-precision=standard",
    "-Wall",
    "-Wextra",
]


def build(force: bool = False) -> str:
    """Compile liboracle.so in place with gcc (seconds).  Returns its path."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "fp8q_oracle.h")))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (used by the tests that
    plant a mistake in the oracle to show that the pins catch it)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", *CFLAGS, "-w", "-I", _HERE, "-o", out_path, src, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


@contextlib.contextmanager
def use_library(path: str):
    """Route every oracle call to another build of the oracle for a while."""
    global _lib
    old = _lib
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = old


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        _lib = _configure(ctypes.CDLL(_LIB))
    return _lib


def _configure(L: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    F = ctypes.c_float
    I = ctypes.c_int
    L.oracle_per_token_group_quant.argtypes = [P, P, P, P, I64, I64, I64, F, I, I]
    L.oracle_rms_norm_per_block_quant.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, F, I, I]
    L.oracle_silu_and_mul_per_block_quant.argtypes = [P, P, P, P, P, I64, I64, I64, F, I, I]
    for name in ("oracle_per_token_group_quant", "oracle_rms_norm_per_block_quant",
                 "oracle_silu_and_mul_per_block_quant"):
        getattr(L, name).restype = I
    L.oracle_fused_qk_norm_rope.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, F, I]
    L.oracle_fused_qk_norm_rope.restype = I
    L.oracle_pack_ue8m0.argtypes = [P, I64, I64, P]
    L.oracle_pack_ue8m0.restype = I
    L.oracle_pack_ue8m0_mx.argtypes = [P, I64, I64, P]
    L.oracle_pack_ue8m0_mx.restype = I
    L.oracle_group_scale_n.argtypes = [P, P, I64, F, I]
    L.oracle_f32_to_e4m3_n.argtypes = [P, P, I64]
    L.oracle_ue8m0_ceil_n.argtypes = [P, P, I64]
    L.oracle_silu_mul_n.argtypes = [P, P, P, I64]
    L.oracle_quant_pairs.argtypes = [P, P, P, I64]
    L.oracle_row_sumsq.argtypes = [P, I64, I64, P]
    L.oracle_rms_inv.argtypes = [F, I64, F]
    L.oracle_rms_inv.restype = F
    L.oracle_f32_to_bf16.argtypes = [F]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    return L


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, x.dtype
    return x


def _check(rc: int):
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")


def _scale_shape(T, G, col_major):
    return (G, T) if col_major else (T, G)


def per_token_group_quant(x_bits, group=128, eps=SCALE_EPS, ue8m0=False, col_major=False):
    """op A.  x_bits uint16 [T,H].  Returns (q uint8 [T,H], scales, scales_pre)."""
    x = _u16(x_bits)
    T, H = x.shape
    G = H // group
    q = np.empty((T, H), np.uint8)
    s = np.empty(_scale_shape(T, G, col_major), np.float32)
    sp = np.empty_like(s)
    _check(lib().oracle_per_token_group_quant(_p(x), _p(q), _p(s), _p(sp), T, H, group,
                                              float(eps), int(ue8m0), int(col_major)))
    return q, s, sp


def rms_norm_per_block_quant(x_bits, w_bits, residual_bits=None, group=128, eps=RMS_EPS,
                             ue8m0=False, col_major=False, want_values=False):
    """op B.  Returns (q, scales, scales_pre, inv [T], residual_out or None),
    plus the quantised fp32 values [T,H] when want_values."""
    x = _u16(x_bits)
    w = _u16(w_bits)
    T, H = x.shape
    G = H // group
    q = np.empty((T, H), np.uint8)
    s = np.empty(_scale_shape(T, G, col_major), np.float32)
    sp = np.empty_like(s)
    inv = np.empty(T, np.float32)
    v = np.empty((T, H), np.float32) if want_values else None
    r = None
    if residual_bits is not None:
        r = np.array(_u16(residual_bits), copy=True)
    _check(lib().oracle_rms_norm_per_block_quant(
        _p(x), _p(r) if r is not None else None, _p(w), _p(q), _p(s), _p(sp), _p(inv),
        _p(v) if v is not None else None, T, H, group, float(eps), int(ue8m0), int(col_major)))
    if want_values:
        return q, s, sp, inv, r, v
    return q, s, sp, inv, r


def silu_and_mul_per_block_quant(x_bits, group=128, eps=SCALE_EPS, ue8m0=False, col_major=False,
                                 want_values=False):
    """op C.  x_bits uint16 [T, 2I].  Returns (q uint8 [T,I], scales, scales_pre),
    plus the quantised fp32 values [T,I] when want_values."""
    x = _u16(x_bits)
    T, H2 = x.shape
    I = H2 // 2
    G = I // group
    q = np.empty((T, I), np.uint8)
    s = np.empty(_scale_shape(T, G, col_major), np.float32)
    sp = np.empty_like(s)
    v = np.empty((T, I), np.float32) if want_values else None
    _check(lib().oracle_silu_and_mul_per_block_quant(_p(x), _p(q), _p(s), _p(sp),
                                                     _p(v) if v is not None else None, T, I, group,
                                                     float(eps), int(ue8m0), int(col_major)))
    if want_values:
        return q, s, sp, v
    return q, s, sp


# ------------------------------------------------------ per-token ops --
# "Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA", section "Welche Kernel
# wurden in vLLM integriert": dynamic_per_token_scaled_fp8_quant,
# rms_norm_dynamic_per_token_quant, silu_and_mul_dynamic_per_token_quant.
# The same arithmetic as the per-group ops with the group spanning the row,
# so each is the per-group function called with group = the row length; the
# scales come back as [T] (one per token).


def dynamic_per_token_scaled_fp8_quant(x_bits, eps=SCALE_EPS, ue8m0=False):
    """x_bits uint16 [T,H] -> (q uint8 [T,H], scales [T], scales_pre [T])."""
    x = _u16(x_bits)
    q, s, sp = per_token_group_quant(x, group=x.shape[1], eps=eps, ue8m0=ue8m0)
    return q, s[:, 0].copy(), sp[:, 0].copy()


def rms_norm_dynamic_per_token_quant(x_bits, w_bits, residual_bits=None, eps=RMS_EPS, ue8m0=False,
                                     want_values=False):
    """Returns (q, scales [T], scales_pre [T], inv [T], residual_out or None),
    plus the quantised fp32 values [T,H] when want_values."""
    x = _u16(x_bits)
    out = rms_norm_per_block_quant(x, w_bits, residual_bits, group=x.shape[1], eps=eps, ue8m0=ue8m0,
                                   want_values=want_values)
    q, s, sp = out[0], out[1][:, 0].copy(), out[2][:, 0].copy()
    return (q, s, sp) + tuple(out[3:])


def silu_and_mul_dynamic_per_token_quant(x_bits, eps=SCALE_EPS, ue8m0=False, want_values=False):
    """x_bits uint16 [T, 2I] -> (q uint8 [T,I], scales [T], scales_pre [T]),
    plus the quantised fp32 values [T,I] when want_values."""
    x = _u16(x_bits)
    out = silu_and_mul_per_block_quant(x, group=x.shape[1] // 2, eps=eps, ue8m0=ue8m0,
                                       want_values=want_values)
    return (out[0], out[1][:, 0].copy(), out[2][:, 0].copy()) + tuple(out[3:])


def fused_qk_norm_rope(qkv_bits, q_w_bits, k_w_bits, cos_sin_bits, positions, num_q_heads, num_kv_heads,
                       head_dim=128, eps=RMS_EPS, is_neox=True):
    """fused_qk_norm_rope ("Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA", the
    kernel list): per-head RMSNorm of the query and key heads, then the rotary
    embedding (steps in fp8q_oracle.c).  qkv_bits uint16 [T, (Hq + 2 Hkv) * D];
    returns the updated copy (value heads unchanged)."""
    out = np.array(_u16(qkv_bits), copy=True)
    T = out.shape[0]
    cs = _u16(cos_sin_bits)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    assert pos.shape == (T,) and out.shape[1] == (num_q_heads + 2 * num_kv_heads) * head_dim
    _check(lib().oracle_fused_qk_norm_rope(_p(out), _p(_u16(q_w_bits)), _p(_u16(k_w_bits)), _p(cs), _p(pos), T,
                                           num_q_heads, num_kv_heads, head_dim, cs.shape[0], float(eps),
                                           int(is_neox)))
    return out


def pack_ue8m0(scales_tg) -> np.ndarray:
    """Power-of-two scales [T, G] (fp32, row-major) -> the packed UE8M0 bytes
    (layout in fp8q_oracle.c), as a uint8 array [ceil(G/4), round_up(T, 4), 4]."""
    s = np.ascontiguousarray(scales_tg, dtype=np.float32)
    T, G = s.shape
    K, T_pad = -(-G // 4), -(-T // 4) * 4
    out = np.empty((K, T_pad, 4), np.uint8)
    _check(lib().oracle_pack_ue8m0(_p(s), T, G, _p(out)))
    return out


def pack_ue8m0_mx(scales_tg) -> np.ndarray:
    """Power-of-two scales [T, G] -> the MXFP8 scale-factor tile layout
    (fp8q_oracle.c), as uint8 [round_up(T, 128), 4 G]: the flat bytes in
    storage order, shaped like the padded scale matrix they encode."""
    s = np.ascontiguousarray(scales_tg, dtype=np.float32)
    T, G = s.shape
    T_pad = -(-T // 128) * 128
    out = np.empty((T_pad, 4 * G), np.uint8)
    _check(lib().oracle_pack_ue8m0_mx(_p(s), T, G, _p(out)))
    return out


def group_scale(amax, eps=SCALE_EPS, ue8m0=False) -> np.ndarray:
    """The scale of a group with maximum |value| amax: RN32(max(amax, eps) / 448),
    rounded up to a power of two with ue8m0 (elementwise)."""
    a = np.ascontiguousarray(amax, dtype=np.float32)
    out = np.empty_like(a)
    lib().oracle_group_scale_n(_p(a), _p(out), a.size, eps, int(ue8m0))
    return out


def f32_to_e4m3(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_f32_to_e4m3_n(_p(v), _p(out), v.size)
    return out


def ue8m0_ceil(s) -> np.ndarray:
    s = np.ascontiguousarray(s, dtype=np.float32)
    out = np.empty_like(s)
    lib().oracle_ue8m0_ceil_n(_p(s), _p(out), s.size)
    return out


def silu_mul(a, b) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    out = np.empty_like(a)
    lib().oracle_silu_mul_n(_p(a), _p(b), _p(out), a.size)
    return out


def quant_pairs(v, s) -> np.ndarray:
    """e4m3(RN32(v / s)) elementwise."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_quant_pairs(_p(v), _p(s), _p(out), v.size)
    return out


def row_sumsq(z_bits) -> np.ndarray:
    z = _u16(z_bits)
    T, H = z.shape
    out = np.empty(T, np.float32)
    lib().oracle_row_sumsq(_p(z), T, H, _p(out))
    return out


def rms_inv(ss: float, H: int, eps=RMS_EPS) -> np.float32:
    return np.float32(lib().oracle_rms_inv(float(ss), int(H), float(eps)))
