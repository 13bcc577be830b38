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
