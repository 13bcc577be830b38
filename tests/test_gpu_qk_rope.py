"""fused_qk_norm_rope on the GPU against the oracle, bit for bit.

Every step is one correctly rounded fp32 operation in the oracle's order and
the head's sum of squares is exact, so the bf16 outputs must be identical,
value heads included (they must come back untouched).

A grid that fits in one wave with eight lanes a head takes that build (up
to a few hundred tokens of 64 + 8 heads; here T <= 256), larger ones four
lanes a head (T = 600, 1000, 4096 here); both pairings and both load widths
are covered for each."""

import numpy as np
import pytest
import torch

import fp8_token_group_bf16_b300 as fq
import oracle
from fp8_token_group_bf16_b300 import inputs
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(qkv, qw, kw, cs, pos, Hq, Hkv, is_neox, offset_bytes=0):
    """GPU result as uint16 bits; offset_bytes > 0 places qkv 16 (not 32)
    bytes past a 32-byte boundary."""
    if offset_bytes:
        n = qkv.numel()
        buf = torch.empty(n + offset_bytes // 2, dtype=torch.bfloat16, device="cuda")
        x = buf[offset_bytes // 2 :].view(qkv.shape)
        x.copy_(qkv.cuda())
    else:
        x = qkv.cuda()
    fq.fused_qk_norm_rope(x, qw.cuda(), kw.cuda(), cs.cuda(), pos.cuda(), Hq, Hkv, is_neox=is_neox)
    torch.cuda.synchronize()
    return inputs.bits(x.cpu())


def _check(T, Hq, Hkv, is_neox, seed, P=inputs.QK_P, offset_bytes=0, pos=None):
    qkv, qw, kw, cs, p = inputs.qk_norm_rope_input(T, Hq, Hkv, P=P, seed=seed)
    if pos is not None:
        p = pos
    got = _run(qkv, qw, kw, cs, p, Hq, Hkv, is_neox, offset_bytes)
    want = oracle.fused_qk_norm_rope(inputs.bits(qkv), inputs.bits(qw), inputs.bits(kw), inputs.bits(cs),
                                     p.numpy(), Hq, Hkv, is_neox=is_neox)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (len(bad), bad[:4], got[tuple(bad[0])], want[tuple(bad[0])])


@pytest.mark.parametrize("T,Hq,Hkv", [(1, 64, 8), (7, 64, 8), (37, 32, 8), (256, 16, 8), (1000, 64, 8),
                                      (3, 1, 0), (5, 0, 2), (4096, 64, 8)])
@pytest.mark.parametrize("is_neox", [True, False], ids=["neox", "interleaved"])
def test_qk_norm_rope_exact(T, Hq, Hkv, is_neox):
    _check(T, Hq, Hkv, is_neox, seed=6100 + T + Hq)


@pytest.mark.parametrize("T,Hq,Hkv", [(9, 8, 2), (600, 64, 8)])
@pytest.mark.parametrize("is_neox", [True, False], ids=["neox", "interleaved"])
def test_qk_norm_rope_16_byte_aligned(T, Hq, Hkv, is_neox):
    _check(T, Hq, Hkv, is_neox, seed=6200 + T, offset_bytes=16)


def test_qk_norm_rope_table_ends_and_repeats():
    T = 64
    pos = torch.tensor([0, 1, 2, inputs.QK_P - 1] * (T // 4), dtype=torch.int64)
    _check(T, 64, 8, True, seed=6300, pos=pos)


def test_qk_norm_rope_zero_and_constant_heads():
    """An all-zero head (inv = 1/sqrt(eps), every output a signed zero) and a
    constant head."""
    Hq, Hkv, D = 4, 2, 128
    qkv, qw, kw, cs, pos = inputs.qk_norm_rope_input(3, Hq, Hkv, P=64, seed=6400)
    qkv = qkv.float()
    qkv[0, :D] = 0.0
    qkv[1, D : 2 * D] = -0.0
    qkv[2, 2 * D : 3 * D] = 3.0
    qkv = inputs.bf16(qkv)
    for is_neox in (True, False):
        got = _run(qkv, qw, kw, cs, pos, Hq, Hkv, is_neox)
        want = oracle.fused_qk_norm_rope(inputs.bits(qkv), inputs.bits(qw), inputs.bits(kw), inputs.bits(cs),
                                         pos.numpy(), Hq, Hkv, is_neox=is_neox)
        assert np.array_equal(got, want)


def test_qk_norm_rope_empty():
    x = torch.empty(0, 10240, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    cs = torch.ones(4, 128, dtype=torch.bfloat16, device="cuda")
    fq.fused_qk_norm_rope(x, w, w, cs, torch.empty(0, dtype=torch.int64, device="cuda"), 64, 8)
