"""fp8_token_group_bf16_b300: fused FP8 per-group quantisation epilogues for B300 (sm_103a).

The compute lives in ``libfp8q.so`` (hand-written CUDA for sm_103a, C ABI in
``include/fp8q.h``).  This package is a thin ctypes binding over it:

* ``fp8q_per_token_group_quant``, ``fp8q_rms_norm_per_block_quant``,
  ``fp8q_silu_and_mul_per_block_quant``, their per-token variants
  ``fp8q_dynamic_per_token_scaled_fp8_quant``,
  ``fp8q_rms_norm_dynamic_per_token_quant``,
  ``fp8q_silu_and_mul_dynamic_per_token_quant``, ``fp8q_fused_qk_norm_rope``,
  and ``fp8q_f32_to_e4m3``,
  ``fp8q_status_string`` -- the C entry points under their own names, taking
  raw device pointers (ints) and sizes, returning the status code;
* ``per_token_group_fp8_quant``, ``rms_norm_per_block_quant``,
  ``silu_and_mul_per_block_quant``, ``dynamic_per_token_scaled_fp8_quant``,
  ``rms_norm_dynamic_per_token_quant``,
  ``silu_and_mul_dynamic_per_token_quant``, ``fused_qk_norm_rope`` -- the
  same calls on torch tensors:
  argument checks, output allocation, the current CUDA stream, and an
  exception on a non-zero status.  Every step of the computation runs in the
  library's kernels; there is no CPU fallback.  If the library is missing or
  no CUDA device is present the calls raise.

The library is built in place by ``python -m fp8_token_group_bf16_b300.build``.
"""

from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libfp8q.so")

FP8Q_OK = 0
FP8Q_ERR_INVALID_ARG = 1
FP8Q_ERR_UNSUPPORTED = 2
FP8Q_ERR_MISALIGNED = 3
FP8Q_ERR_CUDA = 4
FP8Q_SCALES_ROW_MAJOR = 0
FP8Q_SCALES_COL_MAJOR = 1
FP8Q_SCALES_UE8M0_PACKED = 2
FP8Q_SCALES_UE8M0_MX = 3
FP8Q_RMS_MAX_H = 32768
FP8Q_TOKEN_MAX_COLS = 65536
GROUP = 128

EXPORTS = (
    "fp8q_per_token_group_quant",
    "fp8q_rms_norm_per_block_quant",
    "fp8q_silu_and_mul_per_block_quant",
    "fp8q_dynamic_per_token_scaled_fp8_quant",
    "fp8q_rms_norm_dynamic_per_token_quant",
    "fp8q_silu_and_mul_dynamic_per_token_quant",
    "fp8q_fused_qk_norm_rope",
    "fp8q_f32_to_e4m3",
    "fp8q_silu_mul",
    "fp8q_group_scale",
    "fp8q_quant_pairs",
    "fp8q_status_string",
    "fp8q_version",
)

_lib = None


class Fp8qError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fp8q_status_string(status)} (status {status})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfp8q.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libfp8q.so not found at {path}; build it with "
            "`python -m fp8_token_group_bf16_b300.build` (needs nvcc)")
    L = ctypes.CDLL(path)
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    L.fp8q_per_token_group_quant.argtypes = [P, P, P, I64, I64, I32, F, I32, I32, P]
    L.fp8q_rms_norm_per_block_quant.argtypes = [P, P, P, P, P, I64, I64, I32, F, I32, I32, P]
    L.fp8q_silu_and_mul_per_block_quant.argtypes = [P, P, P, I64, I64, I32, F, I32, I32, P]
    L.fp8q_dynamic_per_token_scaled_fp8_quant.argtypes = [P, P, P, I64, I64, F, I32, P]
    L.fp8q_rms_norm_dynamic_per_token_quant.argtypes = [P, P, P, P, P, I64, I64, F, I32, P]
    L.fp8q_silu_and_mul_dynamic_per_token_quant.argtypes = [P, P, P, I64, I64, F, I32, P]
    L.fp8q_fused_qk_norm_rope.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, F, I32, P]
    L.fp8q_f32_to_e4m3.argtypes = [P, P, I64, P]
    L.fp8q_silu_mul.argtypes = [P, P, P, I64, P]
    L.fp8q_group_scale.argtypes = [P, P, I64, F, I32, P]
    L.fp8q_quant_pairs.argtypes = [P, P, P, I64, P]
    for n in EXPORTS[:10]:
        getattr(L, n).restype = ctypes.c_int
    L.fp8q_status_string.argtypes = [ctypes.c_int]
    L.fp8q_status_string.restype = ctypes.c_char_p
    L.fp8q_version.argtypes = []
    L.fp8q_version.restype = ctypes.c_int
    _lib = L
    return L


# ----------------------------------------------- raw C entry points -----


def fp8q_per_token_group_quant(x, q, scales, T, H, group_size, eps, ue8m0, scale_layout, stream):
    return load().fp8q_per_token_group_quant(x, q, scales, T, H, group_size, eps, ue8m0,
                                             scale_layout, stream)


def fp8q_rms_norm_per_block_quant(x, residual, weight, q, scales, T, H, group_size, eps, ue8m0,
                                  scale_layout, stream):
    return load().fp8q_rms_norm_per_block_quant(x, residual, weight, q, scales, T, H, group_size,
                                                eps, ue8m0, scale_layout, stream)


def fp8q_silu_and_mul_per_block_quant(x, q, scales, T, I, group_size, eps, ue8m0, scale_layout,
                                      stream):
    return load().fp8q_silu_and_mul_per_block_quant(x, q, scales, T, I, group_size, eps, ue8m0,
                                                    scale_layout, stream)


def fp8q_dynamic_per_token_scaled_fp8_quant(x, q, scales, T, H, eps, ue8m0, stream):
    return load().fp8q_dynamic_per_token_scaled_fp8_quant(x, q, scales, T, H, eps, ue8m0, stream)


def fp8q_rms_norm_dynamic_per_token_quant(x, residual, weight, q, scales, T, H, eps, ue8m0, stream):
    return load().fp8q_rms_norm_dynamic_per_token_quant(x, residual, weight, q, scales, T, H, eps, ue8m0,
                                                        stream)


def fp8q_silu_and_mul_dynamic_per_token_quant(x, q, scales, T, I, eps, ue8m0, stream):
    return load().fp8q_silu_and_mul_dynamic_per_token_quant(x, q, scales, T, I, eps, ue8m0, stream)


def fp8q_fused_qk_norm_rope(qkv, q_weight, k_weight, cos_sin, positions, T, num_q_heads, num_kv_heads,
                            head_dim, max_position, eps, is_neox, stream):
    return load().fp8q_fused_qk_norm_rope(qkv, q_weight, k_weight, cos_sin, positions, T, num_q_heads,
                                          num_kv_heads, head_dim, max_position, eps, is_neox, stream)


def fp8q_f32_to_e4m3(v, out, n, stream):
    return load().fp8q_f32_to_e4m3(v, out, n, stream)


def fp8q_silu_mul(a, b, out, n, stream):
    return load().fp8q_silu_mul(a, b, out, n, stream)


def fp8q_group_scale(amax, scales, n, eps, ue8m0, stream):
    return load().fp8q_group_scale(amax, scales, n, eps, ue8m0, stream)


def fp8q_quant_pairs(v, s, out, n, stream):
    return load().fp8q_quant_pairs(v, s, out, n, stream)


def fp8q_status_string(status: int) -> str:
    return load().fp8q_status_string(int(status)).decode()


def fp8q_version() -> int:
    return load().fp8q_version()


# ------------------------------------------------ tensor-level calls ----


def _torch():
    import torch

    return torch


def _check(status: int, where: str):
    if status != FP8Q_OK:
        raise Fp8qError(status, where)


def _stream_ptr(t, stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need_cuda_bf16(name, t):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def packed_scale_shape(T: int, G: int):
    """Shape of packed UE8M0 scales as int32 words: [ceil(G/4), T rounded up to 4]."""
    return (-(-G // 4), -(-T // 4) * 4)


def mx_scale_shape(T: int, G: int):
    """Shape of MXFP8 scale-factor tiles as uint8: [T rounded up to 128, 4 G]
    (the padded E8M0 matrix, one byte per 32 values, stored tile by tile)."""
    return (-(-T // 128) * 128, 4 * G)


def _layout(column_major_scales, packed_ue8m0_scales, ue8m0, mx_scales=False):
    if packed_ue8m0_scales or mx_scales:
        if not ue8m0:
            raise ValueError("exponent-byte scale layouts need ue8m0=True")
        if packed_ue8m0_scales and mx_scales:
            raise ValueError("choose one scale layout")
        return FP8Q_SCALES_UE8M0_PACKED if packed_ue8m0_scales else FP8Q_SCALES_UE8M0_MX
    return FP8Q_SCALES_COL_MAJOR if column_major_scales else FP8Q_SCALES_ROW_MAJOR


def _same_device(name, t, x):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device != x.device:
        raise ValueError(f"{name} must be a tensor on {x.device}, the device of x")


def _check_q(q, x, T, cols):
    """A caller's code buffer: one byte per value, [T, cols], contiguous, on x's device."""
    _same_device("q", q, x)
    if tuple(q.shape) != (T, cols) or q.element_size() != 1 or not q.is_contiguous():
        raise ValueError(f"q must be a contiguous 1-byte tensor of shape [{T}, {cols}]")
    return q


def _outputs(x, T, cols, group_size, layout, q, scales):
    torch = _torch()
    G = cols // group_size
    if q is None:
        q = torch.empty((T, cols), dtype=torch.float8_e4m3fn, device=x.device)
    else:
        _check_q(q, x, T, cols)
    if scales is not None:
        _same_device("scales", scales, x)
    if scales is None:
        if layout == FP8Q_SCALES_UE8M0_PACKED:
            scales = torch.empty(packed_scale_shape(T, G), dtype=torch.int32, device=x.device)
        elif layout == FP8Q_SCALES_UE8M0_MX:
            scales = torch.empty(mx_scale_shape(T, G), dtype=torch.uint8, device=x.device)
        elif layout == FP8Q_SCALES_COL_MAJOR:
            scales = torch.empty((G, T), dtype=torch.float32, device=x.device).t()
        else:
            scales = torch.empty((T, G), dtype=torch.float32, device=x.device)
    return q, scales


def _scale_ptr(scales, T, G, layout):
    if layout == FP8Q_SCALES_UE8M0_MX:
        if tuple(scales.shape) != mx_scale_shape(T, G) or scales.element_size() != 1 or \
                not scales.is_contiguous():
            raise ValueError(f"MX scales must be a contiguous 1-byte tensor of shape {mx_scale_shape(T, G)}")
        return scales.data_ptr()
    if layout == FP8Q_SCALES_UE8M0_PACKED:
        if tuple(scales.shape) != packed_scale_shape(T, G) or scales.dtype != _torch().int32 or \
                not scales.is_contiguous():
            raise ValueError(f"packed scales must be a contiguous int32 tensor of shape {packed_scale_shape(T, G)}")
        return scales.data_ptr()
    want = (1, T) if layout == FP8Q_SCALES_COL_MAJOR else (G, 1)
    if scales.dtype != _torch().float32 or tuple(scales.shape) != (T, G) or \
            (T > 1 and G > 1 and tuple(scales.stride()) != want):
        raise ValueError(f"scales must be a [T, G] = [{T}, {G}] fp32 tensor with strides {want}")
    return scales.data_ptr()


def per_token_group_fp8_quant(x, group_size: int = GROUP, eps: float = 1e-10, ue8m0: bool = False,
                              column_major_scales: bool = False, q=None, scales=None, stream=None,
                              packed_ue8m0_scales: bool = False, mx_scales: bool = False):
    """x bf16 [T, H] (CUDA, contiguous) -> (q float8_e4m3fn [T, H], scales fp32 [T, H/g]).

    Column-major scales come back as a [T, G] view of a [G, T] buffer;
    packed UE8M0 scales as int32 words [ceil(G/4), T rounded up to 4]; MX
    scales as uint8 [T rounded up to 128, 4 G] in the block-scaled GEMM's
    tile order (view them as torch.float8_e8m0fnu to hand them to such a GEMM)."""
    _need_cuda_bf16("x", x)
    if x.dim() != 2:
        raise ValueError("x must be 2-D [T, H]")
    T, H = x.shape
    layout = _layout(column_major_scales, packed_ue8m0_scales, ue8m0, mx_scales)
    q, scales = _outputs(x, T, H, group_size, layout, q, scales)
    sp = _scale_ptr(scales, T, H // max(group_size, 1), layout)
    _check(fp8q_per_token_group_quant(
        x.data_ptr(), q.data_ptr(), sp, T, H, group_size, eps, int(ue8m0), layout,
        _stream_ptr(x, stream)), "per_token_group_fp8_quant")
    return q, scales


def rms_norm_per_block_quant(x, weight, residual=None, eps: float = 1e-6, group_size: int = GROUP,
                             ue8m0: bool = False, column_major_scales: bool = False, q=None,
                             scales=None, stream=None, packed_ue8m0_scales: bool = False,
                             mx_scales: bool = False):
    """RMSNorm(x [+ residual]) * weight, then group FP8 quantisation.

    When ``residual`` is given it is updated in place to bf16(x + residual),
    the value that is normalised.  Returns (q, scales)."""
    _need_cuda_bf16("x", x)
    _need_cuda_bf16("weight", weight)
    _same_device("weight", weight, x)
    if residual is not None:
        _need_cuda_bf16("residual", residual)
        _same_device("residual", residual, x)
        if residual.shape != x.shape:
            raise ValueError("residual must have the shape of x")
    if x.dim() != 2 or weight.dim() != 1 or weight.shape[0] != x.shape[1]:
        raise ValueError("x must be [T, H] and weight [H]")
    T, H = x.shape
    layout = _layout(column_major_scales, packed_ue8m0_scales, ue8m0, mx_scales)
    q, scales = _outputs(x, T, H, group_size, layout, q, scales)
    sp = _scale_ptr(scales, T, H // max(group_size, 1), layout)
    _check(fp8q_rms_norm_per_block_quant(
        x.data_ptr(), residual.data_ptr() if residual is not None else None, weight.data_ptr(),
        q.data_ptr(), sp, T, H, group_size, eps, int(ue8m0), layout,
        _stream_ptr(x, stream)), "rms_norm_per_block_quant")
    return q, scales


def silu_and_mul_per_block_quant(x, group_size: int = GROUP, eps: float = 1e-10, ue8m0: bool = False,
                                 column_major_scales: bool = False, q=None, scales=None,
                                 stream=None, packed_ue8m0_scales: bool = False, mx_scales: bool = False):
    """x bf16 [T, 2I] = [gate | up] -> quant(silu(gate) * up): (q [T, I], scales [T, I/g])."""
    _need_cuda_bf16("x", x)
    if x.dim() != 2 or x.shape[1] % 2:
        raise ValueError("x must be [T, 2I]")
    T, I = x.shape[0], x.shape[1] // 2
    layout = _layout(column_major_scales, packed_ue8m0_scales, ue8m0, mx_scales)
    q, scales = _outputs(x, T, I, group_size, layout, q, scales)
    sp = _scale_ptr(scales, T, I // max(group_size, 1), layout)
    _check(fp8q_silu_and_mul_per_block_quant(
        x.data_ptr(), q.data_ptr(), sp, T, I, group_size, eps, int(ue8m0), layout,
        _stream_ptr(x, stream)), "silu_and_mul_per_block_quant")
    return q, scales


# ------------------------------------------------- per-token variants ----


def _token_outputs(x, T, cols, q, scales):
    torch = _torch()
    if q is None:
        q = torch.empty((T, cols), dtype=torch.float8_e4m3fn, device=x.device)
    else:
        _check_q(q, x, T, cols)
    if scales is None:
        scales = torch.empty((T, 1), dtype=torch.float32, device=x.device)
    _same_device("scales", scales, x)
    if scales.numel() != T or scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError(f"per-token scales must be a contiguous fp32 tensor of {T} elements")
    return q, scales


def dynamic_per_token_scaled_fp8_quant(x, eps: float = 1e-10, ue8m0: bool = False, q=None, scales=None,
                                       stream=None):
    """x bf16 [T, H] -> (q float8_e4m3fn [T, H], scales fp32 [T, 1]): one scale per token."""
    _need_cuda_bf16("x", x)
    if x.dim() != 2:
        raise ValueError("x must be 2-D [T, H]")
    T, H = x.shape
    q, scales = _token_outputs(x, T, H, q, scales)
    _check(fp8q_dynamic_per_token_scaled_fp8_quant(x.data_ptr(), q.data_ptr(), scales.data_ptr(), T, H, eps,
                                                   int(ue8m0), _stream_ptr(x, stream)),
           "dynamic_per_token_scaled_fp8_quant")
    return q, scales


def rms_norm_dynamic_per_token_quant(x, weight, residual=None, eps: float = 1e-6, ue8m0: bool = False, q=None,
                                     scales=None, stream=None):
    """RMSNorm(x [+ residual]) * weight, then one FP8 scale per token.

    ``residual`` (optional) is updated in place to bf16(x + residual), as in
    rms_norm_per_block_quant.  Returns (q [T, H], scales [T, 1])."""
    _need_cuda_bf16("x", x)
    _need_cuda_bf16("weight", weight)
    _same_device("weight", weight, x)
    if residual is not None:
        _need_cuda_bf16("residual", residual)
        _same_device("residual", residual, x)
        if residual.shape != x.shape:
            raise ValueError("residual must have the shape of x")
    if x.dim() != 2 or weight.dim() != 1 or weight.shape[0] != x.shape[1]:
        raise ValueError("x must be [T, H] and weight [H]")
    T, H = x.shape
    q, scales = _token_outputs(x, T, H, q, scales)
    _check(fp8q_rms_norm_dynamic_per_token_quant(
        x.data_ptr(), residual.data_ptr() if residual is not None else None, weight.data_ptr(), q.data_ptr(),
        scales.data_ptr(), T, H, eps, int(ue8m0), _stream_ptr(x, stream)), "rms_norm_dynamic_per_token_quant")
    return q, scales


def silu_and_mul_dynamic_per_token_quant(x, eps: float = 1e-10, ue8m0: bool = False, q=None, scales=None,
                                         stream=None):
    """x bf16 [T, 2I] = [gate | up] -> (q [T, I], scales [T, 1]) of silu(gate) * up."""
    _need_cuda_bf16("x", x)
    if x.dim() != 2 or x.shape[1] % 2:
        raise ValueError("x must be [T, 2I]")
    T, I = x.shape[0], x.shape[1] // 2
    q, scales = _token_outputs(x, T, I, q, scales)
    _check(fp8q_silu_and_mul_dynamic_per_token_quant(x.data_ptr(), q.data_ptr(), scales.data_ptr(), T, I, eps,
                                                     int(ue8m0), _stream_ptr(x, stream)),
           "silu_and_mul_dynamic_per_token_quant")
    return q, scales


# ------------------------------------------------- fused_qk_norm_rope ----


def fused_qk_norm_rope(qkv, q_weight, k_weight, cos_sin, positions, num_q_heads: int, num_kv_heads: int,
                       head_dim: int = 128, eps: float = 1e-6, is_neox: bool = True, stream=None):
    """In place on qkv bf16 [T, (Hq + 2 Hkv) * D]: RMSNorm of every query and
    key head (weights q_weight / k_weight, bf16 [D]), then the rotary
    embedding from cos_sin bf16 [max_position, D] at positions int64 [T].
    Value heads are left as they are.  Returns qkv."""
    torch = _torch()
    for name, t in (("qkv", qkv), ("q_weight", q_weight), ("k_weight", k_weight), ("cos_sin", cos_sin)):
        _need_cuda_bf16(name, t)
        _same_device(name, t, qkv)
    if positions.device != qkv.device or positions.dtype != torch.int64 or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous int64 tensor on the device of qkv")
    T = qkv.shape[0]
    if qkv.dim() != 2 or qkv.shape[1] != (num_q_heads + 2 * num_kv_heads) * head_dim:
        raise ValueError("qkv must be [T, (num_q_heads + 2 * num_kv_heads) * head_dim]")
    if positions.numel() != T or q_weight.numel() != head_dim or k_weight.numel() != head_dim or \
            cos_sin.dim() != 2 or cos_sin.shape[1] != head_dim:
        raise ValueError("positions [T], weights [head_dim] and cos_sin [max_position, head_dim] expected")
    _check(fp8q_fused_qk_norm_rope(qkv.data_ptr(), q_weight.data_ptr(), k_weight.data_ptr(), cos_sin.data_ptr(),
                                   positions.data_ptr(), T, num_q_heads, num_kv_heads, head_dim, cos_sin.shape[0],
                                   eps, int(is_neox), _stream_ptr(qkv, stream)), "fused_qk_norm_rope")
    return qkv


def silu_mul(a, b, out=None, stream=None):
    """fp32 CUDA tensors a, b (same shape) -> silu(a) * b as op C computes it."""
    torch = _torch()
    for name, t in (("a", a), ("b", b)):
        if t.device.type != "cuda" or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
    if a.shape != b.shape or a.device != b.device:
        raise ValueError("a and b must have the same shape and device")
    if out is None:
        out = torch.empty_like(a)
    elif out.device != a.device or out.dtype != torch.float32 or out.shape != a.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous fp32 tensor shaped like a, on a's device")
    _check(fp8q_silu_mul(a.data_ptr(), b.data_ptr(), out.data_ptr(), a.numel(), _stream_ptr(a, stream)), "silu_mul")
    return out


def group_scale(amax, eps: float = 1e-10, ue8m0: bool = False, out=None, stream=None):
    """fp32 CUDA tensor of group maxima -> the scales the kernels form from them."""
    torch = _torch()
    if amax.device.type != "cuda" or amax.dtype != torch.float32 or not amax.is_contiguous():
        raise ValueError("amax must be a contiguous fp32 CUDA tensor")
    if out is None:
        out = torch.empty_like(amax)
    elif out.device != amax.device or out.dtype != torch.float32 or out.shape != amax.shape or \
            not out.is_contiguous():
        raise ValueError("out must be a contiguous fp32 tensor shaped like amax, on its device")
    _check(fp8q_group_scale(amax.data_ptr(), out.data_ptr(), amax.numel(), eps, int(ue8m0), _stream_ptr(amax, stream)),
           "group_scale")
    return out


def quant_pairs(v, s, out=None, stream=None):
    """fp32 CUDA tensors of values and positive normal scales -> the
    float8_e4m3fn codes e4m3(RN32(v / s)), by the kernels' quotient."""
    torch = _torch()
    for name, t in (("v", v), ("s", s)):
        if t.device.type != "cuda" or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
    _same_device("s", s, v)
    if s.shape != v.shape:
        raise ValueError("s must have v's shape")
    if out is None:
        out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    elif out.device != v.device or out.element_size() != 1 or out.numel() != v.numel() or not out.is_contiguous():
        raise ValueError("out must be a contiguous 1-byte tensor with v's element count, on v's device")
    _check(fp8q_quant_pairs(v.data_ptr(), s.data_ptr(), out.data_ptr(), v.numel(), _stream_ptr(v, stream)),
           "quant_pairs")
    return out


def f32_to_e4m3(v, out=None, stream=None):
    """fp32 CUDA tensor -> float8_e4m3fn codes (round to nearest even, saturating)."""
    torch = _torch()
    if v.device.type != "cuda" or v.dtype != torch.float32 or not v.is_contiguous():
        raise ValueError("v must be a contiguous fp32 CUDA tensor")
    if out is None:
        out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    elif out.device != v.device or out.element_size() != 1 or out.numel() != v.numel() or not out.is_contiguous():
        raise ValueError("out must be a contiguous 1-byte tensor with v's element count, on v's device")
    _check(fp8q_f32_to_e4m3(v.data_ptr(), out.data_ptr(), v.numel(), _stream_ptr(v, stream)),
           "f32_to_e4m3")
    return out
