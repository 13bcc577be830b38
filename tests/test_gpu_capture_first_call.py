"""The first call of an entry point in a process may come inside CUDA-graph
capture.  Some launches ask the runtime once per kernel how many CTAs fit a
SM (rms_norm_per_block_quant spreading a one-wave grid by padding its CTAs,
fused_qk_norm_rope choosing four or eight lanes a head); that query is not
a stream operation and must neither fail nor break the capture.  Run in a
fresh process so that nothing is cached yet: capture the first calls,
replay the graph, and compare with the same calls made eagerly afterwards."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch
import fp8_token_group_bf16_b300 as fq
fq.load()
g = torch.Generator(device="cpu").manual_seed(5)
x = torch.randn(512, 5120, generator=g).to(torch.bfloat16).cuda()          # one wave, padded CTAs
w = (1 + 0.1 * torch.randn(5120, generator=g)).to(torch.bfloat16).cuda()
qkv = torch.randn(16, 80 * 128, generator=g).to(torch.bfloat16).cuda()      # eight lanes a head
qw = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16).cuda()
cs = torch.randn(64, 128, generator=g).to(torch.bfloat16).cuda()
pos = torch.randint(0, 64, (16,), generator=g).cuda()
q = torch.empty(512, 5120, dtype=torch.float8_e4m3fn, device="cuda")
s = torch.empty(512, 40, device="cuda")
qkv_g = qkv.clone()
stream = torch.cuda.Stream()
graph = torch.cuda.CUDAGraph()
with torch.cuda.stream(stream):
    with torch.cuda.graph(graph, stream=stream):
        fq.rms_norm_per_block_quant(x, w, None, ue8m0=True, q=q, scales=s)
        fq.fused_qk_norm_rope(qkv_g, qw, qw, cs, pos, 64, 8)
graph.replay()
torch.cuda.synchronize()
q2, s2 = fq.rms_norm_per_block_quant(x, w, None, ue8m0=True)
qkv_e = qkv.clone()
fq.fused_qk_norm_rope(qkv_e, qw, qw, cs, pos, 64, 8)
torch.cuda.synchronize()
assert torch.equal(q.view(torch.uint8), q2.view(torch.uint8)) and torch.equal(s, s2)
assert torch.equal(qkv_g, qkv_e)
print("ok")
"""


def test_first_calls_inside_graph_capture():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
