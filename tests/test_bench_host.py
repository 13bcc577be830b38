"""Host-side logic of bench.py, without a GPU: the byte accounting, the
weak-scaling aggregation over ranks (two gloo processes), and the
reference arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_per_element():
    T, H = 4096, 7168
    assert bench.algorithmic_bytes("per_token_group_fp8_quant", T, H) / (T * H) == 3.03125
    assert bench.algorithmic_bytes("silu_and_mul_per_block_quant", T, 25600) / (T * 25600) == 5.03125
    b = bench.algorithmic_bytes("rms_norm_per_block_quant", T, 5120)
    assert b == T * 5120 * 3 + 4 * T * 40 + 2 * 5120
    assert bench.algorithmic_bytes("rms_norm_per_block_quant", T, 5120, residual=True) == b + 4 * T * 5120
    # the byte counts quoted for the small configurations
    assert bench.algorithmic_bytes("per_token_group_fp8_quant", 20, 512) == 31040
    assert bench.algorithmic_bytes("rms_norm_per_block_quant", 256, 4096) == 3186688
    assert bench.algorithmic_bytes("rms_norm_per_block_quant", 256, 4096, True) == 7380992
    assert bench.algorithmic_bytes("silu_and_mul_per_block_quant", 1024, 12288) == 63307776
    # packed UE8M0: one byte per group, groups padded to 4 and tokens to 4
    assert bench.algorithmic_bytes("per_token_group_fp8_quant", 5, 768, packed=True) == 5 * 768 * 3 + 2 * 8 * 4
    assert bench.algorithmic_bytes("silu_and_mul_per_block_quant", 4096, 25600, packed=True) == \
        4096 * 25600 * 5 + 4096 * 200
    # MXFP8 tiles: four bytes per group (one per 32 values), rows padded to 128
    assert bench.algorithmic_bytes("per_token_group_fp8_quant", 130, 7168, mx=True) == 130 * 7168 * 3 + 256 * 4 * 56
    # per-token variants: one fp32 scale per row
    assert bench.algorithmic_bytes("dynamic_per_token_scaled_fp8_quant", 7, 896) == 7 * 896 * 3 + 4 * 7
    assert bench.algorithmic_bytes("rms_norm_dynamic_per_token_quant", 7, 896, residual=True) == \
        7 * 896 * 3 + 4 * 7 + 2 * 896 + 4 * 7 * 896
    assert bench.algorithmic_bytes("silu_and_mul_dynamic_per_token_quant", 7, 896) == 7 * 896 * 5 + 4 * 7
    # fused_qk_norm_rope: heads read and written, position and table row per token, two weights
    assert bench.qk_rope_bytes(10) == 10 * (72 * 128 * 4 + 8 + 256) + 512
    assert bench.step_bytes(1) == 21728 + 15520 + 10240 + 128800


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    d = bench.Dist(backend="gloo")
    try:
        d.barrier()
        # rank r processed (r+1) GB in (r+1) * 0.5 s
        agg = bench.aggregate(1e9 * (rank + 1), 0.5 * (rank + 1), d, steps=10)
        # the host-link rate of the e2e record is the slowest rank's
        agg["min_link"] = d.min(10.0 * (rank + 1))
        out[rank] = agg
    finally:
        d.close()


def test_weak_scaling_aggregate_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        agg = out[r]
        assert agg["seconds"] == 1.0              # max over ranks
        assert agg["total_bytes"] == 3e9          # every rank's bytes
        assert abs(agg["value"] - 3.0) < 1e-12    # GB/s of the whole job
        assert abs(agg["ms_per_step"] - 100.0) < 1e-9
        assert agg["min_link"] == 10.0            # min over ranks


def test_single_process_aggregate():
    d = bench.Dist()
    agg = bench.aggregate(2e9, 0.25, d, steps=5)
    assert agg["value"] == 8.0 and agg["ms_per_step"] == 50.0


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3", "--reference-budget-s", "5"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_traffic_record_rejects_stale_kernel_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.txt").write_text(
        "kernel_source_sha256 = deadbeef\nsilu_quant_kernel T=4096 I=25600 ue8m0 row = 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("silu_quant_kernel", "T=4096 I=25600 ue8m0 row") is None
