"""rms_norm_per_block_quant at decode sizes, through the C ABI, bit for bit
against the oracle.

At T <= 64 rows of more than 64 groups run the cluster-split kernel (a row
over up to 8 CTAs exchanging their exact partial sums through distributed
shared memory); shorter rows, and every row at larger T, run one CTA per
row.  Both are covered here at T = 1, 2, 8, 64 (and just past the switch),
with and without the residual, in every scale layout: fp32 row- and
column-major (with and without UE8M0), packed UE8M0 exponent bytes and the
MXFP8 scale tiles.  Group counts that do not divide evenly over the
cluster (65, 97, 255) check the last CTA's share.  Scale buffers are
pre-filled with a canary so the zero padding of the exponent-byte layouts
is checked too.
"""

import numpy as np
import pytest
import torch

import fp8_token_group_bf16_b300 as fq
import oracle
from fp8_token_group_bf16_b300 import inputs
from gpu_util import dev_bf16, host_codes, require_gpu
from tolerance import assert_exact, to_tg

pytestmark = pytest.mark.gpu

T_VALUES = [1, 2, 8, 64, 65]
H_VALUES = [4096, 5120, 8192, 8320, 12288, 12416, 16384, 32640, 32768]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(xb, wb, rb, layout, ue8m0):
    T, H = xb.shape
    G = H // 128
    x, w = dev_bf16(xb), dev_bf16(wb)
    r = dev_bf16(rb) if rb is not None else None
    kw = dict(ue8m0=ue8m0)
    if layout == "packed":
        kw.update(packed_ue8m0_scales=True,
                  scales=torch.full(fq.packed_scale_shape(T, G), -1, dtype=torch.int32, device=x.device))
    elif layout == "mx":
        kw.update(mx_scales=True,
                  scales=torch.full(fq.mx_scale_shape(T, G), 0xEE, dtype=torch.uint8, device=x.device))
    elif layout == "col":
        kw.update(column_major_scales=True)
    q, s = fq.rms_norm_per_block_quant(x, w, r, **kw)
    torch.cuda.synchronize()
    rout = inputs.bits(r.cpu()) if r is not None else None
    return host_codes(q), s, rout


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
@pytest.mark.parametrize("H", H_VALUES)
@pytest.mark.parametrize("T", T_VALUES)
def test_rms_decode_sizes_bit_exact(T, H, residual):
    x, w, r = inputs.rms_input(T, H, seeds=(7100 + T, 7101 + H, 7102 + T))
    xb, wb = inputs.bits(x), inputs.bits(w)
    rb = inputs.bits(r) if residual else None
    G = H // 128
    for layout, ue8m0 in (("row", False), ("col", False), ("row", True), ("col", True), ("packed", True),
                          ("mx", True)):
        what = f"T={T} H={H} residual={residual} {layout} ue8m0={ue8m0}"
        q, s, rout = _run(xb, wb, rb, layout, ue8m0)
        qr, sr, _, _, ror = oracle.rms_norm_per_block_quant(xb, wb, rb, ue8m0=ue8m0, col_major=layout == "col")
        if residual:
            assert np.array_equal(rout, ror), f"{what}: residual output differs"
        if layout in ("row", "col"):
            assert_exact(q, s.cpu().numpy(), qr, to_tg(sr, layout == "col"), what)
        elif layout == "packed":
            assert np.array_equal(q, qr), what
            pk = s.cpu().contiguous().view(torch.uint8).numpy().reshape(s.shape[0], s.shape[1], 4)
            assert np.array_equal(pk, oracle.pack_ue8m0(sr)), what
        else:
            assert np.array_equal(q, qr), what
            assert np.array_equal(s.cpu().numpy(), oracle.pack_ue8m0_mx(sr)), what


@pytest.mark.parametrize("H", [12288, 32768])
def test_rms_decode_degenerate_rows(H):
    """All-zero, constant and tiny rows through the cluster-split kernel."""
    x = torch.zeros(4, H)
    x[1] = 0.75
    x[2] = -3.0
    x[3, ::2] = 1e-20
    xb = inputs.bits(inputs.bf16(x))
    wb = inputs.bits(inputs.bf16(torch.ones(H)))
    for ue8m0 in (False, True):
        q, s, _ = _run(xb, wb, None, "row", ue8m0)
        qr, sr, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, None, ue8m0=ue8m0)
        assert_exact(q, s.cpu().numpy(), qr, sr, f"degenerate rows H={H}")
