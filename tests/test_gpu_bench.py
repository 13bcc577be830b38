"""The end-to-end pipeline that bench.py times computes what the three ops
compute on the whole batch: one pipelined step (uneven token slices, three
streams) against direct calls, bit for bit."""

import os
import sys

import pytest
import torch

import fp8_token_group_bf16_b300 as fq
from gpu_util import require_gpu

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("T,chunks", [(100, 8), (33, 4), (1, 8)])
def test_e2e_pipeline_outputs(T, chunks):
    host = bench.workload_inputs(T)
    pipe = bench.E2EPipeline(host, chunks)
    for _ in range(2):   # a second step overwrites the same buffers
        pipe.step()
    torch.cuda.synchronize()
    xa, (xb, wb), xc = host["per_token_group_fp8_quant"][0], host["rms_norm_per_block_quant"], \
        host["silu_and_mul_per_block_quant"][0]
    qa, sa = fq.per_token_group_fp8_quant(xa.cuda(), ue8m0=True, column_major_scales=True)
    qb, sb = fq.rms_norm_per_block_quant(xb.cuda(), wb.cuda(), ue8m0=True)
    qc, sc = fq.silu_and_mul_per_block_quant(xc.cuda(), ue8m0=True)
    u8 = lambda q: q.view(torch.uint8).cpu()
    for (lo, hi), outs in zip(pipe.bounds, pipe.outs_host):
        pqa, psa, pqb, psb, pqc, psc = outs
        assert torch.equal(pqa.view(torch.uint8), u8(qa)[lo:hi])
        assert torch.equal(psa, sa.cpu()[lo:hi].t())
        assert torch.equal(pqb.view(torch.uint8), u8(qb)[lo:hi])
        assert torch.equal(psb, sb.cpu()[lo:hi])
        assert torch.equal(pqc.view(torch.uint8), u8(qc)[lo:hi])
        assert torch.equal(psc, sc.cpu()[lo:hi])


def test_e2e_record_carries_its_host_link_ceiling():
    """time_e2e reports the step's host bytes and, beside them, the host
    link's own rate for those bytes; the pipelined step cannot beat a plain
    copy of the same bytes by more than timing noise."""
    host = bench.workload_inputs(64)
    rec = bench.time_e2e(host, 3, bench.Dist())
    inputs = (host["per_token_group_fp8_quant"][0], *host["rms_norm_per_block_quant"][:2],
              host["silu_and_mul_per_block_quant"][0])
    assert rec["h2d_bytes_per_step"] == sum(t.numel() * t.element_size() for t in inputs)
    link = rec["host_link"]
    assert min(link["h2d_alone_GBps"], link["d2h_alone_GBps"], link["both_GBps"]) > 0
    assert 0 < link["frac"] < 1.5
