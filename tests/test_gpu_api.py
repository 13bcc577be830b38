"""Behaviour of the C ABI on a GPU: status codes with real device pointers,
no writes outside the outputs, streams, CUDA-graph capture."""

import ctypes

import numpy as np
import pytest
import torch

import fp8_token_group_bf16_b300 as fq
import oracle
from fp8_token_group_bf16_b300 import inputs
from gpu_util import dev_bf16, require_gpu
from tolerance import assert_exact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_real_pointer_misalignment_rejected():
    buf = torch.zeros(4 * 512 + 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(4 * 512 + 64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(64, dtype=torch.float32, device="cuda")
    M = fq.FP8Q_ERR_MISALIGNED
    assert fq.fp8q_per_token_group_quant(buf.data_ptr() + 2, q.data_ptr(), s.data_ptr(), 4, 512,
                                         128, 1e-10, 0, 0, _stream()) == M
    assert fq.fp8q_per_token_group_quant(buf.data_ptr(), q.data_ptr() + 4, s.data_ptr(), 4, 512,
                                         128, 1e-10, 0, 0, _stream()) == M
    torch.cuda.synchronize()
    assert int(q.count_nonzero()) == 0


def test_zero_tokens_writes_nothing():
    q = torch.full((64,), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((8,), 7.0, dtype=torch.float32, device="cuda")
    x = torch.zeros(1, 512, dtype=torch.bfloat16, device="cuda")
    assert fq.fp8q_per_token_group_quant(x.data_ptr(), q.data_ptr(), s.data_ptr(), 0, 512, 128,
                                         1e-10, 0, 0, _stream()) == 0
    assert fq.fp8q_silu_and_mul_per_block_quant(x.data_ptr(), q.data_ptr(), s.data_ptr(), 0, 256,
                                                128, 1e-10, 1, 1, _stream()) == 0
    torch.cuda.synchronize()
    assert bool((q == 0xAB).all()) and bool((s == 7.0).all())


def _guarded(nbytes, dtype=torch.uint8, pad=4096):
    """A buffer with `pad` canary bytes (0xA5) on both sides of the payload."""
    raw = torch.full((nbytes + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda")
    return raw, raw[pad : pad + nbytes].view(dtype)


def _canaries_intact(raw, nbytes, pad=4096):
    h = raw.cpu().numpy()
    return bool((h[:pad] == 0xA5).all() and (h[pad + nbytes :] == 0xA5).all())


@pytest.mark.parametrize("T,H", [(1, 128), (3, 384), (37, 7168), (129, 896)])
@pytest.mark.parametrize("op", ["group", "rms", "silu"])
@pytest.mark.parametrize("col", [False, True])
def test_no_writes_outside_outputs(T, H, op, col):
    out_cols = H
    xb = inputs.bits(inputs.heavy_tailed_input(T, 2 * H if op == "silu" else H, seed=T * 3 + H))
    x = dev_bf16(xb)
    G = out_cols // 128
    qraw, q = _guarded(T * out_cols)
    sraw, s = _guarded(T * G * 4, torch.float32)
    layout = int(col)
    st = _stream()
    if op == "group":
        rc = fq.fp8q_per_token_group_quant(x.data_ptr(), q.data_ptr(), s.data_ptr(), T, H, 128,
                                           1e-10, 0, layout, st)
    elif op == "silu":
        rc = fq.fp8q_silu_and_mul_per_block_quant(x.data_ptr(), q.data_ptr(), s.data_ptr(), T, H,
                                                  128, 1e-10, 1, layout, st)
    else:
        w = dev_bf16(inputs.bits(inputs.rms_weight(H)))
        rraw, r = _guarded(T * H * 2, torch.bfloat16)
        r = r.view(T, H)
        r.copy_(x)
        rc = fq.fp8q_rms_norm_per_block_quant(x.data_ptr(), r.data_ptr(), w.data_ptr(), q.data_ptr(),
                                              s.data_ptr(), T, H, 128, 1e-6, 0, layout, st)
    assert rc == 0
    torch.cuda.synchronize()
    assert _canaries_intact(qraw, T * out_cols)
    assert _canaries_intact(sraw, T * G * 4)
    if op == "rms":
        assert _canaries_intact(rraw, T * H * 2)


def test_side_stream_and_graph_capture():
    x = dev_bf16(inputs.bits(inputs.heavy_tailed_input(256, 7168, seed=5)))
    xs = dev_bf16(inputs.bits(inputs.silu_input(256, 2048, seed=6)))
    xr, w, r = [dev_bf16(inputs.bits(t)) for t in inputs.rms_input(256, 4096, seeds=(7, 8, 9))]
    r0 = r.clone()

    def step(stream):
        rr = r0.clone()
        a = fq.per_token_group_fp8_quant(x, ue8m0=True, column_major_scales=True, stream=stream)
        b = fq.silu_and_mul_per_block_quant(xs, ue8m0=False, stream=stream)
        c = fq.rms_norm_per_block_quant(xr, w, rr, stream=stream)
        return a, b, c, rr

    eager = step(None)
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        side_out = step(side)
    side.synchronize()

    g = torch.cuda.CUDAGraph()
    static_r = r0.clone()
    with torch.cuda.graph(g):
        ga = fq.per_token_group_fp8_quant(x, ue8m0=True, column_major_scales=True)
        gb = fq.silu_and_mul_per_block_quant(xs, ue8m0=False)
        gc = fq.rms_norm_per_block_quant(xr, w, static_r)
    for _ in range(3):
        static_r.copy_(r0)
        g.replay()
    torch.cuda.synchronize()

    def same(u, v):
        return torch.equal(u.view(torch.uint8) if u.dtype == torch.float8_e4m3fn else u,
                           v.view(torch.uint8) if v.dtype == torch.float8_e4m3fn else v)

    for (ea, eb, ec, er), (oa, ob, oc, orr) in [(eager, side_out), (eager, (ga, gb, gc, static_r))]:
        for e, o in zip((*ea, *eb, *ec), (*oa, *ob, *oc)):
            assert same(e, o)
        assert torch.equal(er, orr)


def test_graph_replay_matches_oracle():
    """A captured per_token_group_fp8_quant replayed on new input data."""
    T, H = 512, 7168
    x = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    x.copy_(dev_bf16(inputs.bits(inputs.heavy_tailed_input(T, H, seed=1))))
    with torch.cuda.graph(g):
        q, s = fq.per_token_group_fp8_quant(x)
    for seed in (2, 3):
        xb = inputs.bits(inputs.heavy_tailed_input(T, H, seed=seed))
        x.copy_(dev_bf16(xb))
        g.replay()
        torch.cuda.synchronize()
        qr, sr, _ = oracle.per_token_group_quant(xb)
        assert_exact(q.view(torch.uint8).cpu().numpy(), s.cpu().numpy(), qr, sr, f"graph seed={seed}")


@pytest.mark.parametrize("T,H", [(1, 128), (5, 640), (37, 896), (130, 8320)])
@pytest.mark.parametrize("op", ["group", "rms", "silu"])
@pytest.mark.parametrize("mx", [False, True], ids=["packed", "mx"])
def test_packed_scales_no_writes_outside(T, H, op, mx):
    """Exponent-byte scales (packed words or MXFP8 tiles): exactly their
    bytes are written (padding included), nothing around them."""
    xb = inputs.bits(inputs.heavy_tailed_input(T, 2 * H if op == "silu" else H, seed=T + 7 * H))
    x = dev_bf16(xb)
    G = H // 128
    nbytes = (-(-T // 128) * 128 * 4 * G) if mx else -(-G // 4) * (-(-T // 4) * 4) * 4
    qraw, q = _guarded(T * H)
    sraw, s = _guarded(nbytes, torch.int32)
    P, st = (fq.FP8Q_SCALES_UE8M0_MX if mx else fq.FP8Q_SCALES_UE8M0_PACKED), _stream()
    if op == "group":
        rc = fq.fp8q_per_token_group_quant(x.data_ptr(), q.data_ptr(), s.data_ptr(), T, H, 128, 1e-10, 1, P, st)
    elif op == "silu":
        rc = fq.fp8q_silu_and_mul_per_block_quant(x.data_ptr(), q.data_ptr(), s.data_ptr(), T, H, 128, 1e-10, 1,
                                                  P, st)
    else:
        w = dev_bf16(inputs.bits(inputs.rms_weight(H)))
        rc = fq.fp8q_rms_norm_per_block_quant(x.data_ptr(), None, w.data_ptr(), q.data_ptr(), s.data_ptr(), T, H,
                                              128, 1e-6, 1, P, st)
    assert rc == 0
    torch.cuda.synchronize()
    assert _canaries_intact(qraw, T * H) and _canaries_intact(sraw, nbytes)
    assert not bool((s.view(torch.uint8) == 0xA5).any()), "every packed byte is written"


# (the RMSNorm variant's rows end at FP8Q_RMS_MAX_H = 32768; longer rows are rejected, see test_native_cpu)
@pytest.mark.parametrize("op,T,H", [(op, T, H) for op in ("token", "token_silu", "token_rms")
                                    for T, H in ((1, 128), (3, 896), (7, 8320), (2, 65536), (2, 32768))
                                    if not (op == "token_rms" and H > fq.FP8Q_RMS_MAX_H)])
def test_per_token_no_writes_outside(op, T, H):
    xb = inputs.bits(inputs.heavy_tailed_input(T, 2 * H if op == "token_silu" else H, seed=T + 11 * H))
    x = dev_bf16(xb)
    qraw, q = _guarded(T * H)
    sraw, s = _guarded(T * 4, torch.float32)
    st = _stream()
    if op == "token":
        rc = fq.fp8q_dynamic_per_token_scaled_fp8_quant(x.data_ptr(), q.data_ptr(), s.data_ptr(), T, H, 1e-10, 0, st)
    elif op == "token_silu":
        rc = fq.fp8q_silu_and_mul_dynamic_per_token_quant(x.data_ptr(), q.data_ptr(), s.data_ptr(), T, H, 1e-10, 1,
                                                          st)
    else:
        w = dev_bf16(inputs.bits(inputs.rms_weight(H)))
        rc = fq.fp8q_rms_norm_dynamic_per_token_quant(x.data_ptr(), None, w.data_ptr(), q.data_ptr(), s.data_ptr(),
                                                      T, H, 1e-6, 0, st)
    assert rc == 0
    torch.cuda.synchronize()
    assert _canaries_intact(qraw, T * H) and _canaries_intact(sraw, T * 4)


def test_qk_norm_rope_no_writes_outside():
    T, Hq, Hkv = 9, 8, 2
    qkv, qw, kw, cs, pos = inputs.qk_norm_rope_input(T, Hq, Hkv, P=64, seed=31)
    n = qkv.numel() * 2
    raw, buf = _guarded(n, torch.bfloat16)
    x = buf.view(qkv.shape)
    x.copy_(qkv.cuda())
    fq.fused_qk_norm_rope(x, qw.cuda(), kw.cuda(), cs.cuda(), pos.cuda(), Hq, Hkv)
    torch.cuda.synchronize()
    assert _canaries_intact(raw, n)


def test_widened_ops_in_a_graph():
    """Packed scales, the per-token ops (a clustered launch) and the rotary
    kernel captured in one CUDA graph give the eager results."""
    xa = dev_bf16(inputs.bits(inputs.heavy_tailed_input(64, 25600, seed=41)))
    xs = dev_bf16(inputs.bits(inputs.silu_input(64, 25600, seed=42)))
    qkv, qw, kw, cs, pos = [t.cuda() for t in inputs.qk_norm_rope_input(32, 16, 4, P=256, seed=43)]

    def run(qkv_buf):
        a = fq.per_token_group_fp8_quant(xa, ue8m0=True, packed_ue8m0_scales=True)
        b = fq.dynamic_per_token_scaled_fp8_quant(xa)
        c = fq.silu_and_mul_dynamic_per_token_quant(xs, ue8m0=True)
        fq.fused_qk_norm_rope(qkv_buf, qw, kw, cs, pos, 16, 4)
        return (*a, *b, *c, qkv_buf)

    eager = run(qkv.clone())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    static_qkv = qkv.clone()
    with torch.cuda.graph(g):
        captured = run(static_qkv)
    static_qkv.copy_(qkv)
    g.replay()
    torch.cuda.synchronize()
    for e, o in zip(eager, captured):
        e8 = e.view(torch.uint8) if e.dtype == torch.float8_e4m3fn else e
        o8 = o.view(torch.uint8) if o.dtype == torch.float8_e4m3fn else o
        assert torch.equal(e8, o8)


def test_tensor_api_rejects_wrong_scale_buffers():
    """The tensor-level calls check caller-provided scale buffers against the
    layout before anything is launched."""
    x = torch.zeros(5, 640, dtype=torch.bfloat16, device="cuda")
    G = 5
    with pytest.raises(ValueError):   # packed words need [ceil(G/4), T rounded up to 4]
        fq.per_token_group_fp8_quant(x, ue8m0=True, packed_ue8m0_scales=True,
                                     scales=torch.empty(2, 5, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):   # MXFP8 tiles need [T rounded up to 128, 4 G] bytes
        fq.per_token_group_fp8_quant(x, ue8m0=True, mx_scales=True,
                                     scales=torch.empty(5, 4 * G, dtype=torch.uint8, device="cuda"))
    with pytest.raises(ValueError):   # row-major fp32 [T, G]
        fq.per_token_group_fp8_quant(x, scales=torch.empty(5, G + 1, device="cuda"))
    with pytest.raises(ValueError):   # column-major: a [T, G] view of a [G, T] buffer, not a [T, G] buffer
        fq.per_token_group_fp8_quant(x[:, :512].contiguous(), column_major_scales=True,
                                     scales=torch.empty(5, 4, device="cuda"))
    with pytest.raises(ValueError):   # per-token scales: T values
        fq.dynamic_per_token_scaled_fp8_quant(x, scales=torch.empty(4, device="cuda"))
    # the right shapes go through
    q, s = fq.per_token_group_fp8_quant(x, ue8m0=True, mx_scales=True,
                                        scales=torch.empty(fq.mx_scale_shape(5, G), dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert s.shape == (128, 4 * G)


def test_tensor_api_checks_caller_buffers():
    """Output buffers passed in by the caller are checked before their raw
    pointers reach the kernels: shape, element size, contiguity, dtype of
    fp32 scales, and the device of every tensor."""
    x = torch.zeros(8, 512, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(512, dtype=torch.bfloat16, device="cuda")
    e4 = torch.float8_e4m3fn
    bad_q = [torch.empty(4, 512, dtype=e4, device="cuda"),                   # too few rows
             torch.empty(8, 1024, dtype=e4, device="cuda")[:, ::2],          # strided
             torch.empty(8, 512, dtype=torch.bfloat16, device="cuda"),       # 2-byte elements
             torch.empty(8, 512, dtype=e4)]                                  # on the host
    for q in bad_q:
        with pytest.raises(ValueError, match="q must be"):
            fq.per_token_group_fp8_quant(x, q=q)
        with pytest.raises(ValueError, match="q must be"):
            fq.rms_norm_per_block_quant(x, w, q=q)
        with pytest.raises(ValueError, match="q must be"):
            fq.dynamic_per_token_scaled_fp8_quant(x, q=q)
    with pytest.raises(ValueError, match="q must be"):
        fq.silu_and_mul_per_block_quant(x, q=torch.empty(8, 512, dtype=e4, device="cuda"))   # I = 256
    bad_s = [torch.empty(8, 4, dtype=torch.bfloat16, device="cuda"),          # not fp32
             torch.empty(8, 4, dtype=torch.float32),                          # on the host
             torch.empty(8, 2, dtype=torch.float32, device="cuda")]           # too small
    for s in bad_s:
        with pytest.raises(ValueError, match="scales must be"):
            fq.per_token_group_fp8_quant(x, scales=s)
        with pytest.raises(ValueError, match="scales must be"):
            fq.rms_norm_per_block_quant(x, w, scales=s)
    with pytest.raises(ValueError, match="scales must be"):
        fq.dynamic_per_token_scaled_fp8_quant(x, scales=torch.empty(8, 1, dtype=torch.float32))
    with pytest.raises(ValueError, match="scales must be"):
        fq.per_token_group_fp8_quant(x, ue8m0=True, packed_ue8m0_scales=True,
                                     scales=torch.empty(fq.packed_scale_shape(8, 4), dtype=torch.int32))
    with pytest.raises(ValueError):
        fq.rms_norm_per_block_quant(x, w.cpu())
    with pytest.raises(ValueError):
        fq.rms_norm_per_block_quant(x, w, torch.zeros(8, 512, dtype=torch.bfloat16))
    a = torch.zeros(16, device="cuda")
    with pytest.raises(ValueError, match="out must be"):
        fq.group_scale(a, out=torch.empty(8, device="cuda"))
    with pytest.raises(ValueError, match="out must be"):
        fq.f32_to_e4m3(a, out=torch.empty(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="out must be"):
        fq.silu_mul(a, a, out=torch.empty(16, dtype=torch.float64, device="cuda"))
    # nothing was launched on the rejected buffers; a good call still works
    q, s = fq.per_token_group_fp8_quant(x)
    torch.cuda.synchronize()
    assert q.shape == (8, 512) and s.shape == (8, 4)
