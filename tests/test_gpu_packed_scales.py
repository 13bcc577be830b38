"""Packed UE8M0 scales (exponent bytes, four groups per 32-bit word) from
all three ops, against the oracle's packing of its own power-of-two scales.

The packed words are a re-encoding of the UE8M0 scales: byte e of group g,
token t stands for 2^(e - 127).  Op A and op B must match the oracle byte for
byte; op C may differ only where the oracle's fp32 scale sits on a power of
two within the tolerance, exactly as its fp32 UE8M0 scales may.  The buffers
are pre-filled with 0xFF so the zero padding (tokens past T, groups past G)
is checked too."""

import numpy as np
import pytest
import torch

import fp8_token_group_bf16_b300 as fq
import oracle
from fp8_token_group_bf16_b300 import inputs
from gpu_util import dev_bf16, host_codes, require_gpu
from tolerance import check_fused

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _packed_buffer(T, G, device):
    return torch.full(fq.packed_scale_shape(T, G), -1, dtype=torch.int32, device=device)


def _packed_bytes(s: torch.Tensor) -> np.ndarray:
    """int32 words [K, T_pad] -> uint8 [K, T_pad, 4] (byte j = group 4k + j)."""
    K, Tp = s.shape
    return s.cpu().contiguous().view(torch.uint8).numpy().reshape(K, Tp, 4)


def _decode(pk: np.ndarray, T: int, G: int) -> np.ndarray:
    """Packed bytes -> fp32 scales [T, G]."""
    e = pk.transpose(1, 0, 2).reshape(pk.shape[1], -1)[:T, :G].astype(np.int32)
    return np.ldexp(np.float64(1.0), e - 127).astype(np.float32)


def _assert_padding_zero(pk, T, G):
    K, Tp, _ = pk.shape
    flat = pk.transpose(1, 0, 2).reshape(Tp, 4 * K)   # [T_pad, 4K] in (token, group) order
    assert not flat[T:].any(), "bytes of tokens past T must be 0"
    assert not flat[:, G:].any(), "bytes of groups past G must be 0"


@pytest.mark.parametrize("T,H", [(1, 128), (7, 896), (5, 640), (4, 512), (37, 7168), (4096, 7168)])
def test_group_quant_packed(T, H):
    xb = inputs.bits(inputs.heavy_tailed_input(T, H, 4100 + T + H))
    G = H // 128
    x = dev_bf16(xb)
    s = _packed_buffer(T, G, x.device)
    q, s = fq.per_token_group_fp8_quant(x, ue8m0=True, packed_ue8m0_scales=True, scales=s)
    torch.cuda.synchronize()
    pk = _packed_bytes(s)
    qr, sr, _ = oracle.per_token_group_quant(xb, ue8m0=True, col_major=False)
    assert np.array_equal(host_codes(q), qr)
    assert np.array_equal(pk, oracle.pack_ue8m0(sr))
    _assert_padding_zero(pk, T, G)


@pytest.mark.parametrize("T,H,residual", [(1, 128, False), (7, 896, True), (37, 1152, False),
                                          (256, 4096, True), (3, 24576, False), (5, 16384, True)])
def test_rms_packed(T, H, residual):
    x, w, r = inputs.rms_input(T, H, seeds=(4200 + T, 4201 + H, 4202))
    xb, wb = inputs.bits(x), inputs.bits(w)
    rb = inputs.bits(r) if residual else None
    G = H // 128
    xd, wd = dev_bf16(xb), dev_bf16(wb)
    rd = dev_bf16(rb) if residual else None
    s = _packed_buffer(T, G, xd.device)
    q, s = fq.rms_norm_per_block_quant(xd, wd, rd, ue8m0=True, packed_ue8m0_scales=True, scales=s)
    torch.cuda.synchronize()
    pk = _packed_bytes(s)
    qr, sr, _, _, ror = oracle.rms_norm_per_block_quant(xb, wb, rb, ue8m0=True)
    assert np.array_equal(host_codes(q), qr)
    assert np.array_equal(pk, oracle.pack_ue8m0(sr))
    _assert_padding_zero(pk, T, G)
    if residual:
        assert np.array_equal(inputs.bits(rd.cpu()), ror)


@pytest.mark.parametrize("T,I", [(1, 128), (7, 896), (37, 1152), (64, 12288), (5, 640)])
def test_silu_packed(T, I):
    xb = inputs.bits(inputs.silu_input(T, I, seed=4300 + T + I))
    G = I // 128
    x = dev_bf16(xb)
    s = _packed_buffer(T, G, x.device)
    q, s = fq.silu_and_mul_per_block_quant(x, ue8m0=True, packed_ue8m0_scales=True, scales=s)
    torch.cuda.synchronize()
    pk = _packed_bytes(s)
    _assert_padding_zero(pk, T, G)
    qr, sr, spr, vr = oracle.silu_and_mul_per_block_quant(xb, ue8m0=True, want_values=True)
    check_fused(host_codes(q), _decode(pk, T, G), qr, sr, spr, vr, True, f"silu packed T={T} I={I}")
    # the packed bytes re-encode the kernel's own fp32 UE8M0 scales
    _, s32 = fq.silu_and_mul_per_block_quant(x, ue8m0=True)
    assert np.array_equal(pk, oracle.pack_ue8m0(s32.cpu().numpy()))


def test_packed_with_ue8m0_off_is_refused():
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fq.per_token_group_fp8_quant(x, packed_ue8m0_scales=True)


# ----------------------------------- MXFP8 scale-factor tiles (kMxUe8m0) ----


def _mx_buffer(T, G):
    return torch.full(fq.mx_scale_shape(T, G), 0xA5, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("T,H", [(1, 128), (7, 896), (128, 512), (130, 7168), (4096, 7168)])
def test_group_quant_mx_tiles(T, H):
    xb = inputs.bits(inputs.heavy_tailed_input(T, H, 4500 + T + H))
    x = dev_bf16(xb)
    q, s = fq.per_token_group_fp8_quant(x, ue8m0=True, mx_scales=True, scales=_mx_buffer(T, H // 128))
    torch.cuda.synchronize()
    qr, sr, _ = oracle.per_token_group_quant(xb, ue8m0=True, col_major=False)
    assert np.array_equal(host_codes(q), qr)
    assert np.array_equal(s.cpu().numpy(), oracle.pack_ue8m0_mx(sr))   # every byte, padding rows included


@pytest.mark.parametrize("T,H,residual", [(3, 1152, True), (200, 5120, False), (129, 4096, True)])
def test_rms_mx_tiles(T, H, residual):
    x, w, r = inputs.rms_input(T, H, seeds=(4600 + T, 4601 + H, 4602))
    xb, wb = inputs.bits(x), inputs.bits(w)
    rb = inputs.bits(r) if residual else None
    rd = dev_bf16(rb) if residual else None
    q, s = fq.rms_norm_per_block_quant(dev_bf16(xb), dev_bf16(wb), rd, ue8m0=True, mx_scales=True,
                                       scales=_mx_buffer(T, H // 128))
    torch.cuda.synchronize()
    qr, sr, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, rb, ue8m0=True)
    assert np.array_equal(host_codes(q), qr)
    assert np.array_equal(s.cpu().numpy(), oracle.pack_ue8m0_mx(sr))


@pytest.mark.parametrize("T,I", [(5, 640), (131, 1152), (64, 12288)])
def test_silu_mx_tiles(T, I):
    xb = inputs.bits(inputs.silu_input(T, I, seed=4700 + T + I))
    x = dev_bf16(xb)
    G = I // 128
    q, s = fq.silu_and_mul_per_block_quant(x, ue8m0=True, mx_scales=True, scales=_mx_buffer(T, G))
    _, s32 = fq.silu_and_mul_per_block_quant(x, ue8m0=True)
    torch.cuda.synchronize()
    # the tiles re-encode the kernel's own fp32 UE8M0 scales; those are checked against the oracle
    assert np.array_equal(s.cpu().numpy(), oracle.pack_ue8m0_mx(s32.cpu().numpy()))
    qr, sr, spr, vr = oracle.silu_and_mul_per_block_quant(xb, ue8m0=True, want_values=True)
    check_fused(host_codes(q), s32.cpu().numpy(), qr, sr, spr, vr, True, f"silu mx T={T} I={I}")


def test_mx_and_packed_need_ue8m0():
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fq.per_token_group_fp8_quant(x, mx_scales=True)
    with pytest.raises(ValueError):
        fq.per_token_group_fp8_quant(x, ue8m0=True, mx_scales=True, packed_ue8m0_scales=True)
