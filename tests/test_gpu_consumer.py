"""The outputs feed FP8 GEMMs: a consumer check of the layouts, end to end.

Blackwell's block-scaled FP8 GEMM (cuBLASLt through torch's scaled_mm, MXFP8
recipe: e4m3 operands, one E8M0 exponent byte per 32 values along K) reads
the codes and the packed UE8M0 exponent bytes of the per-group ops: a 1x128
group's byte is used for its four 32-value blocks.  The per-token ops feed the
row-wise scaled GEMM (one fp32 scale per row of each operand).  Each product
is compared with the matmul of the dequantised operands in fp32; a wrong
scale byte, a wrong code or a wrong layout gives errors of order one, while
the check allows the bf16 rounding of the output.  The GEMM is the library's;
these tests only check that what the kernels write is what such a GEMM
consumes."""

import pytest
import torch
import torch.nn.functional as F

import fp8_token_group_bf16_b300 as fq
from fp8_token_group_bf16_b300 import inputs
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu

GROUP = 128


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def swizzle_32_4_4(e: torch.Tensor) -> torch.Tensor:
    """uint8 [rows, cols] scale bytes -> the 32_4_4 scale-factor layout:
    tiles of 128 rows x 4 columns (rows and columns zero-padded to whole
    tiles), tiles in row-block-major order, and inside a tile the byte of
    (r, c) at offset (r % 32) * 16 + (r // 32) * 4 + c."""
    rows, cols = e.shape
    R, C = -(-rows // 128) * 128, -(-cols // 4) * 4
    p = torch.zeros(R, C, dtype=torch.uint8, device=e.device)
    p[:rows, :cols] = e
    t = p.view(R // 128, 4, 32, C // 4, 4)             # [row block, r // 32, r % 32, col block, c]
    t = t.permute(0, 3, 2, 1, 4)                        # [row block, col block, r % 32, r // 32, c]
    return t.reshape(-1).contiguous()


def packed_bytes_tg(sp: torch.Tensor, T: int, G: int) -> torch.Tensor:
    """Packed UE8M0 words [ceil(G/4), T_pad] -> exponent bytes [T, G]."""
    b = sp.view(torch.uint8).view(sp.shape[0], sp.shape[1], 4)
    return b.permute(1, 0, 2).reshape(sp.shape[1], -1)[:T, :G]


def weight_blocks(N: int, K: int, seed: int):
    """Weights [N, K] quantised in 128x128 blocks with power-of-two scales:
    (codes, fp32 scales [N/128, K/128], exponent bytes)."""
    g = torch.Generator().manual_seed(seed)
    w = (torch.randn(N, K, generator=g) * 0.05).cuda()
    wb = w.reshape(N // 128, 128, K // 128, 128)
    e = torch.ceil(torch.log2(wb.abs().amax(dim=(1, 3)).clamp_min(1e-30) / 448.0))
    ws = torch.exp2(e)
    wq = (wb / ws[:, None, :, None]).reshape(N, K).to(torch.float8_e4m3fn)
    return wq, ws, (e + 127).to(torch.uint8)


def dequant(q: torch.Tensor, s_rows: torch.Tensor, rep_r: int, rep_c: int) -> torch.Tensor:
    return q.float() * s_rows.repeat_interleave(rep_r, 0).repeat_interleave(rep_c, 1)


def mx_gemm(q, ebytes, wq, wbytes):
    sa = swizzle_32_4_4(ebytes.repeat_interleave(GROUP // 32, dim=1)).view(torch.float8_e8m0fnu)
    sb = swizzle_32_4_4(wbytes.repeat_interleave(128, dim=0).repeat_interleave(GROUP // 32, dim=1))
    return F.scaled_mm(q, wq.t(), sa, F.ScalingType.BlockWise1x32, sb.view(torch.float8_e8m0fnu),
                       F.ScalingType.BlockWise1x32, swizzle_a=F.SwizzleType.SWIZZLE_32_4_4,
                       swizzle_b=F.SwizzleType.SWIZZLE_32_4_4, output_dtype=torch.bfloat16)


def rel_err(out, ref):
    return ((out.float() - ref).abs().max() / ref.abs().max()).item()


BF16_OUT = 2.0**-7   # bf16 output rounding (2^-8 relative) with room for summation order


@pytest.mark.parametrize("op", ["group", "rms", "silu"])
@pytest.mark.parametrize("M,K,N", [(256, 1024, 512), (200, 7168, 384), (4096, 5120, 256)])
def test_packed_ue8m0_feeds_block_scaled_gemm(op, M, K, N):
    if op == "group":
        x = inputs.heavy_tailed_input(M, K, seed=M + K).cuda()
        q, s32 = fq.per_token_group_fp8_quant(x, ue8m0=True)
        _, sp = fq.per_token_group_fp8_quant(x, ue8m0=True, packed_ue8m0_scales=True)
    elif op == "rms":
        x, w, _ = [t.cuda() for t in inputs.rms_input(M, K, seeds=(M, K, 1))]
        q, s32 = fq.rms_norm_per_block_quant(x, w, ue8m0=True)
        _, sp = fq.rms_norm_per_block_quant(x, w, ue8m0=True, packed_ue8m0_scales=True)
    else:
        x = inputs.silu_input(M, K, seed=M + 2 * K).cuda()
        q, s32 = fq.silu_and_mul_per_block_quant(x, ue8m0=True)
        _, sp = fq.silu_and_mul_per_block_quant(x, ue8m0=True, packed_ue8m0_scales=True)
    G = K // GROUP
    eb = packed_bytes_tg(sp, M, G)
    assert torch.equal(eb.int(), (s32.view(torch.int32) >> 23) & 0xFF)   # the bytes are the scales' exponents
    wq, ws, wb = weight_blocks(N, K, seed=N)
    ref = dequant(q, s32, 1, GROUP) @ dequant(wq, ws, 128, 128).t()
    out = mx_gemm(q, eb, wq, wb)
    torch.cuda.synchronize()
    assert rel_err(out, ref) <= BF16_OUT
    # the check is sensitive: one group's scale 8x too large shows in its row
    bad = eb.clone()
    bad[M // 2, G // 2] += 3
    out_bad = mx_gemm(q, bad, wq, wb)
    torch.cuda.synchronize()
    row = M // 2
    assert (out_bad[row].float() - ref[row]).abs().max() > 4 * BF16_OUT * ref.abs().max()


@pytest.mark.parametrize("op", ["group", "rms", "silu"])
def test_mx_tiles_feed_block_scaled_gemm_directly(op):
    """With mx_scales=True the kernels write the scale operand of the
    block-scaled GEMM themselves: codes and scales go in as they are."""
    M, K, N = 300, 7168, 512
    if op == "group":
        x = inputs.heavy_tailed_input(M, K, seed=11).cuda()
        q, smx = fq.per_token_group_fp8_quant(x, ue8m0=True, mx_scales=True)
        _, s32 = fq.per_token_group_fp8_quant(x, ue8m0=True)
    elif op == "rms":
        x, w, _ = [t.cuda() for t in inputs.rms_input(M, K, seeds=(12, 13, 14))]
        q, smx = fq.rms_norm_per_block_quant(x, w, ue8m0=True, mx_scales=True)
        _, s32 = fq.rms_norm_per_block_quant(x, w, ue8m0=True)
    else:
        x = inputs.silu_input(M, K, seed=15).cuda()
        q, smx = fq.silu_and_mul_per_block_quant(x, ue8m0=True, mx_scales=True)
        _, s32 = fq.silu_and_mul_per_block_quant(x, ue8m0=True)
    wq, ws, wb = weight_blocks(N, K, seed=16)
    sb = swizzle_32_4_4(wb.repeat_interleave(128, dim=0).repeat_interleave(GROUP // 32, dim=1))
    out = F.scaled_mm(q, wq.t(), smx.view(torch.float8_e8m0fnu), F.ScalingType.BlockWise1x32,
                      sb.view(torch.float8_e8m0fnu), F.ScalingType.BlockWise1x32,
                      swizzle_a=F.SwizzleType.SWIZZLE_32_4_4, swizzle_b=F.SwizzleType.SWIZZLE_32_4_4,
                      output_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ref = dequant(q, s32, 1, GROUP) @ dequant(wq, ws, 128, 128).t()
    assert rel_err(out, ref) <= BF16_OUT


@pytest.mark.parametrize("op", ["token", "token_silu", "token_rms"])
def test_per_token_feeds_rowwise_gemm(op):
    M, K, N = 512, 5120, 768
    if op == "token":
        x = inputs.heavy_tailed_input(M, K, seed=3).cuda()
        q, s = fq.dynamic_per_token_scaled_fp8_quant(x)
    elif op == "token_silu":
        q, s = fq.silu_and_mul_dynamic_per_token_quant(inputs.silu_input(M, K, seed=4).cuda())
    else:
        x, w, _ = [t.cuda() for t in inputs.rms_input(M, K, seeds=(5, 6, 7))]
        q, s = fq.rms_norm_dynamic_per_token_quant(x, w)
    g = torch.Generator().manual_seed(9)
    w = (torch.randn(N, K, generator=g) * 0.05).cuda()
    wsc = w.abs().amax(dim=1, keepdim=True) / 448.0
    wq = (w / wsc).to(torch.float8_e4m3fn)
    ref = (q.float() * s) @ (wq.float() * wsc).t()
    out = F.scaled_mm(q, wq.t(), s, F.ScalingType.RowWise, wsc.t().contiguous(), F.ScalingType.RowWise,
                      output_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert rel_err(out, ref) <= BF16_OUT
