"""Per-token variants on the GPU against the oracle (one scale per row).

dynamic_per_token_scaled_fp8_quant and rms_norm_dynamic_per_token_quant are
bit-exact (correctly rounded quotient; exact sum of squares), like their
per-group counterparts; silu_and_mul_dynamic_per_token_quant is held to the
same tolerance as silu_and_mul_per_block_quant with the group spanning the
row.  Rows longer than 64 groups are spread over a thread-block cluster, so
the shapes cover 1, 2, 4 and 8 CTAs per row, and a row maximum placed in
each CTA of the cluster in turn."""

import numpy as np
import pytest
import torch

import fp8_token_group_bf16_b300 as fq
import oracle
from fp8_token_group_bf16_b300 import inputs
from gpu_util import dev_bf16, host_codes, require_gpu
from tolerance import check_fused

pytestmark = pytest.mark.gpu

# The last two are longer than one wave of CTAs, which launches the build
# that prefetches a later CTA's input into L2.
A_SHAPES = [(1, 128), (7, 896), (37, 7168), (3, 8192), (5, 8320), (4, 25600), (2, 65536), (1024, 5120),
            (2048, 7168), (256, 25600)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _token_a(xb, ue8m0, misaligned=False):
    T, H = xb.shape
    x = dev_bf16(xb)
    q = s = None
    if misaligned:   # 16-byte but not 32-byte aligned input and codes
        buf = torch.empty(T * H + 8, dtype=torch.bfloat16, device="cuda")
        buf[8:].copy_(x.reshape(-1))
        x = buf[8:].view(T, H)
        qb = torch.empty(T * H + 16, dtype=torch.float8_e4m3fn, device="cuda")
        q = qb[16:].view(T, H)
    q, s = fq.dynamic_per_token_scaled_fp8_quant(x, ue8m0=ue8m0, q=q, scales=s)
    torch.cuda.synchronize()
    return host_codes(q), s.cpu().numpy()


@pytest.mark.parametrize("T,H", A_SHAPES)
@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32", "ue8m0"])
def test_per_token_quant_exact(T, H, ue8m0):
    xb = inputs.bits(inputs.heavy_tailed_input(T, H, 5100 + T + H))
    q, s = _token_a(xb, ue8m0)
    qr, sr, _ = oracle.dynamic_per_token_scaled_fp8_quant(xb, ue8m0=ue8m0)
    assert s.shape == (T, 1) and np.array_equal(s[:, 0], sr)
    assert np.array_equal(q, qr), np.argwhere(q != qr)[:4]


@pytest.mark.parametrize("T,H", [(5, 8320), (3, 896)])
def test_per_token_quant_16_byte_aligned(T, H):
    xb = inputs.bits(inputs.heavy_tailed_input(T, H, 5200 + T))
    q, s = _token_a(xb, False, misaligned=True)
    qr, sr, _ = oracle.dynamic_per_token_scaled_fp8_quant(xb)
    assert np.array_equal(s[:, 0], sr) and np.array_equal(q, qr)


def _ctas_per_row(G):
    """The kernels' split of a row of G groups: C CTAs (fewest idle lanes,
    from ceil(G/64) to 8) of gpc groups each."""
    best = None
    for C in range(-(-G // 64), 9):
        gpc = -(-G // C)
        if (C - 1) * gpc >= G:
            continue
        idle = C * (-(-gpc * 4 // 32) * 32) - 4 * G
        if best is None or idle < best[0]:
            best = (idle, C, gpc)
    return best[1], best[2]


@pytest.mark.parametrize("H", [8320, 25600, 65536])
def test_per_token_row_max_in_every_cluster_rank(H):
    """Row t carries a +-1e4 outlier in the part of the row owned by CTA
    t mod C, so the maximum must cross the cluster from every rank."""
    G = H // 128
    C, gpc = _ctas_per_row(G)
    T = 2 * C
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(H))
    for t in range(T):
        r = t % C
        col = min(r * gpc * 128 + 77 + 128 * (t % 3), H - 1)
        x[t, col] = 1e4 if t % 2 else -1e4
    xb = inputs.bits(inputs.bf16(x))
    for ue8m0 in (False, True):
        q, s = _token_a(xb, ue8m0)
        qr, sr, _ = oracle.dynamic_per_token_scaled_fp8_quant(xb, ue8m0=ue8m0)
        assert np.array_equal(s[:, 0], sr) and np.array_equal(q, qr)


def test_per_token_degenerate_rows():
    """An all-zero row (floor scale, signed zero codes), a constant row (every
    code +-448) and a row of bf16 subnormals."""
    H = 8320
    x = torch.zeros(4, H)
    x[1] = -2.5
    x[2, ::3] = 3.0
    x[3] = 1e-39
    xb = inputs.bits(inputs.bf16(x))
    xb[0, ::2] |= 0x8000   # -0
    for ue8m0 in (False, True):
        q, s = _token_a(xb, ue8m0)
        qr, sr, _ = oracle.dynamic_per_token_scaled_fp8_quant(xb, ue8m0=ue8m0)
        assert np.array_equal(s[:, 0], sr) and np.array_equal(q, qr)


def _token_rms(xb, wb, rb, ue8m0):
    x, w = dev_bf16(xb), dev_bf16(wb)
    r = dev_bf16(rb) if rb is not None else None
    q, s = fq.rms_norm_dynamic_per_token_quant(x, w, r, ue8m0=ue8m0)
    torch.cuda.synchronize()
    return host_codes(q), s.cpu().numpy(), (inputs.bits(r.cpu()) if r is not None else None)


@pytest.mark.parametrize("T,H,residual", [(1, 128, False), (7, 896, True), (256, 4096, False),
                                          (256, 4096, True), (3, 24576, False), (2, 32768, True),
                                          (5, 16384, False), (512, 5120, True), (2048, 5120, False),
                                          # one-wave grids (per-group scales would pad these CTAs)
                                          (512, 5120, False), (300, 8192, False),
                                          # the prefetching builds of the 2- and 4-groups-per-quad rows
                                          (400, 12288, False), (200, 20480, False)])
@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32", "ue8m0"])
def test_rms_per_token_exact(T, H, residual, ue8m0):
    x, w, r = inputs.rms_input(T, H, seeds=(5300 + T, 5301 + H, 5302))
    xb, wb = inputs.bits(x), inputs.bits(w)
    rb = inputs.bits(r) if residual else None
    q, s, rout = _token_rms(xb, wb, rb, ue8m0)
    qr, sr, _, _, ror = oracle.rms_norm_dynamic_per_token_quant(xb, wb, rb, ue8m0=ue8m0)
    assert np.array_equal(s[:, 0], sr), np.argwhere(s[:, 0] != sr)[:4]
    assert np.array_equal(q, qr), np.argwhere(q != qr)[:4]
    if residual:
        assert np.array_equal(rout, ror)


def test_rms_per_token_lognormal_rows():
    T, H = 64, 5120
    x = inputs.lognormal_channel_input(T, H, 5400)
    xb, wb = inputs.bits(x), inputs.bits(inputs.rms_weight(H))
    for ue8m0 in (False, True):
        q, s, _ = _token_rms(xb, wb, None, ue8m0)
        qr, sr, _, _, _ = oracle.rms_norm_dynamic_per_token_quant(xb, wb, None, ue8m0=ue8m0)
        assert np.array_equal(s[:, 0], sr) and np.array_equal(q, qr)


def _check_token_silu(xb, ue8m0, what):
    x = dev_bf16(xb)
    q, s = fq.silu_and_mul_dynamic_per_token_quant(x, ue8m0=ue8m0)
    torch.cuda.synchronize()
    I = xb.shape[1] // 2
    qr, sr, spr, vr = oracle.silu_and_mul_dynamic_per_token_quant(xb, ue8m0=ue8m0, want_values=True)
    return check_fused(host_codes(q), s.cpu().numpy(), qr, sr[:, None], spr[:, None], vr, ue8m0, what,
                       group=I)


@pytest.mark.parametrize("T,I", [(1, 128), (7, 896), (37, 1152), (64, 12288), (5, 8320), (4, 25600),
                                 (2, 65536), (512, 25600)])
@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32", "ue8m0"])
def test_silu_per_token(T, I, ue8m0):
    xb = inputs.bits(inputs.silu_input(T, I, seed=5500 + T + I))
    _check_token_silu(xb, ue8m0, f"silu per-token T={T} I={I}")


def test_silu_per_token_qwen3_rows():
    x = inputs.lognormal_channel_input(32, 2 * inputs.MIX_I, 5600)
    _check_token_silu(inputs.bits(x), True, "silu per-token lognormal")


def test_silu_per_token_reduces_to_per_token_quant():
    """gate >= 20 and up = 1: silu(a) * 1 == a exactly, so the result must be
    the per-token quantisation of the gate half, bit for bit."""
    rng = np.random.default_rng(8)
    T, I = 16, 25600
    a = (20.0 + np.abs(rng.standard_normal((T, I))) * 40.0).astype(np.float32)
    ab = inputs.bits(inputs.bf16(torch.from_numpy(a)))
    xb = np.concatenate([ab, inputs.bits(inputs.bf16(torch.ones(T, I)))], axis=1)
    for ue8m0 in (False, True):
        x = dev_bf16(xb)
        q, s = fq.silu_and_mul_dynamic_per_token_quant(x, ue8m0=ue8m0)
        qr, sr, _ = oracle.dynamic_per_token_scaled_fp8_quant(ab, ue8m0=ue8m0)
        assert np.array_equal(s.cpu().numpy()[:, 0], sr) and np.array_equal(host_codes(q), qr)


def test_per_token_empty_input():
    for f, cols in ((fq.dynamic_per_token_scaled_fp8_quant, 512), (fq.silu_and_mul_dynamic_per_token_quant, 1024)):
        q, s = f(torch.empty(0, cols, dtype=torch.bfloat16, device="cuda"))
        assert q.shape[0] == 0 and s.numel() == 0
