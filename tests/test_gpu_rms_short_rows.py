"""rms_norm_per_block_quant (and its per-token variant) on rows of at most 8
groups, through the C ABI, bit for bit against the oracle.

Such a row fits one warp (one quad per group), so the kernel gives each row
a warp of a CTA of several rows (rows of 1, 2 or 4 groups: 8, 4 or 2 rows
to a warp, each on its own segment of lanes) and forms the row's sum from a
butterfly alone, with no shared memory and no barrier.  Covered: T that
leave the last CTA or the last warp partly without rows (1, 3, 5, 127,
1001), a grid long enough for the build that hands later rows to the L2
(6000 rows at H = 1024), rows of 1 to 8 groups, with and without the
residual, in every scale layout.
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

T_VALUES = [1, 3, 5, 127, 1001, 6000]
H_VALUES = [128, 256, 384, 512, 896, 1024]


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
def test_rms_short_rows_bit_exact(T, H, residual):
    x, w, r = inputs.rms_input(T, H, seeds=(9100 + T, 9101 + H, 9102 + T))
    xb, wb = inputs.bits(x), inputs.bits(w)
    rb = inputs.bits(r) if residual else None
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


@pytest.mark.parametrize("T,H,residual", [(1, 128, True), (5, 896, False), (127, 1024, True), (6000, 1024, False),
                                          (1001, 384, False), (77, 256, True), (1001, 512, False), (33, 128, False)])
@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32", "ue8m0"])
def test_rms_per_token_short_rows_bit_exact(T, H, residual, ue8m0):
    x, w, r = inputs.rms_input(T, H, seeds=(9200 + T, 9201 + H, 9202))
    xb, wb = inputs.bits(x), inputs.bits(w)
    rb = inputs.bits(r) if residual else None
    xd, wd = dev_bf16(xb), dev_bf16(wb)
    rd = dev_bf16(rb) if rb is not None else None
    q, s = fq.rms_norm_dynamic_per_token_quant(xd, wd, rd, ue8m0=ue8m0)
    torch.cuda.synchronize()
    qr, sr, _, _, ror = oracle.rms_norm_dynamic_per_token_quant(xb, wb, rb, ue8m0=ue8m0)
    sg = s.cpu().numpy().reshape(-1)
    assert np.array_equal(sg, sr.reshape(-1)), np.argwhere(sg != sr.reshape(-1))[:4]
    qg = host_codes(q)
    assert np.array_equal(qg, qr), np.argwhere(qg != qr)[:4]
    if residual:
        assert np.array_equal(inputs.bits(rd.cpu()), ror)


def test_rms_short_rows_degenerate():
    """All-zero, constant and tiny rows of one group, eight to a warp (six
    rows: the warp's last two segments lie past T)."""
    H = 128
    x = torch.zeros(6, H)
    x[1] = 0.75
    x[2] = -3.0
    x[3, ::2] = 1e-20
    x[4, 5] = 1e4
    xb = inputs.bits(inputs.bf16(x))
    wb = inputs.bits(inputs.bf16(torch.ones(H)))
    for ue8m0 in (False, True):
        q, s, _ = _run(xb, wb, None, "row", ue8m0)
        qr, sr, _, _, _ = oracle.rms_norm_per_block_quant(xb, wb, None, ue8m0=ue8m0)
        assert_exact(q, s.cpu().numpy(), qr, sr, "degenerate short rows")
