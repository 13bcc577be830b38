#!/usr/bin/env python3
"""Benchmark of the fused FP8 quantisation epilogues on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--sweep]

One *step* is one pass of the whole hot path over one batch of T = 4096
tokens shaped like a Qwen3-32B layer (synthetic, seeded inputs):

  per_token_group_fp8_quant     x bf16 [4096, 7168]   heavy-tailed, UE8M0, column-major scales
  rms_norm_per_block_quant      x bf16 [4096, 5120]   per-channel lognormal std, UE8M0, row-major
  silu_and_mul_per_block_quant  x bf16 [4096, 51200]  per-channel lognormal std, UE8M0, row-major

The metric is achieved HBM bandwidth: algorithmic bytes (every input read
once, every output written once) divided by time.  Rank 0 prints one JSON
line.  ``value`` is device-timed with the inputs already in HBM; ``e2e`` is
the same metric through the package's public calls with the inputs copied
from pinned host memory and the outputs copied back inside the timed
region, with ``e2e.host_link`` the link's own rate for the same bytes
(plain copies, each direction alone and both at once) as its ceiling;
``roofline`` is the dominant kernel's bandwidth (CUDA events around
its launches) against the measured copy bandwidth; ``cpu_baseline`` is the
CPU oracle timed on a bounded sample.  Under torchrun every rank processes
its own batch (weak scaling, no collective on the data path).

``--impl reference`` times the CPU oracle instead (the reference arm: this
method has no published implementation to install).  ``--sweep`` prints
per-op T sweeps with a same-size device-to-device copy for comparison,
including the packed-scale layout, the per-token variants and
fused_qk_norm_rope.  ``--op NAME --tokens T`` times one op alone (for
profiling one kernel).
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GROUP = 128
STEP_T = 4096
A_H, B_H, C_I = 7168, 5120, 25600
METRIC = "achieved HBM GB/s and % of roofline per fused FP8 quant op, vs T sweep"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6400.0
DOMINANT = "silu_and_mul_per_block_quant"
KERNEL_NAMES = {   # the kernel each op launches at the step's T
    "per_token_group_fp8_quant": "group_quant_kernel",
    "rms_norm_per_block_quant": "rms_row_kernel",
    "silu_and_mul_per_block_quant": "silu_quant_kernel",
}


# ------------------------------------------------------------------ bytes --


PER_TOKEN_OPS = {
    "dynamic_per_token_scaled_fp8_quant": "per_token_group_fp8_quant",
    "rms_norm_dynamic_per_token_quant": "rms_norm_per_block_quant",
    "silu_and_mul_dynamic_per_token_quant": "silu_and_mul_per_block_quant",
}


def algorithmic_bytes(op: str, T: int, H: int, residual: bool = False, packed: bool = False,
                      mx: bool = False) -> int:
    """Bytes an op must move: each input read once, each output written once.
    group: x bf16 [T,H] in; e4m3 [T,H] and fp32 [T,H/128] out.
    rms:   the same plus the bf16 weight [H]; with the residual, the
           residual [T,H] is read and written (+4 B per element).
    silu:  H is I; x bf16 [T,2I] in; e4m3 [T,I] and fp32 [T,I/128] out.
    packed: the scales are exponent bytes, [ceil(G/4), T rounded up to 4]
           32-bit words, instead of fp32 [T, G].
    mx:    the scales as MXFP8 GEMM tiles, one byte per 32 values, rows
           padded to 128: round_up(T, 128) * 4 * G bytes.
    The per-token variants move the same bytes with one fp32 scale per row."""
    G = H // GROUP
    sb = -(-G // 4) * (-(-T // 4) * 4) * 4 if packed else 4 * T * G
    if mx:
        sb = -(-T // 128) * 128 * 4 * G
    if op in PER_TOKEN_OPS:
        op, sb = PER_TOKEN_OPS[op], 4 * T
    if op == "per_token_group_fp8_quant":
        return T * H * 3 + sb
    if op == "rms_norm_per_block_quant":
        return T * H * 3 + sb + 2 * H + (4 * T * H if residual else 0)
    if op == "silu_and_mul_per_block_quant":
        return T * H * 5 + sb
    raise ValueError(op)


def qk_rope_bytes(T: int, Hq: int = 64, Hkv: int = 8, D: int = 128) -> int:
    """fused_qk_norm_rope: every query and key head read and written once
    (bf16), each token's position (8 B) and its cos/sin table row (2D bf16),
    and the two norm weights once per launch; value heads are not touched."""
    return T * ((Hq + Hkv) * D * 4 + 8 + 2 * D) + 4 * D


def step_bytes(T: int = STEP_T) -> int:
    return (algorithmic_bytes("per_token_group_fp8_quant", T, A_H)
            + algorithmic_bytes("rms_norm_per_block_quant", T, B_H)
            + algorithmic_bytes("silu_and_mul_per_block_quant", T, C_I))


# ------------------------------------------------------------ distributed --


class Dist:
    """One process per GPU under torchrun; a no-op at N = 1."""

    def __init__(self, backend: str | None = None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist

            if backend is None:
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
                dist.init_process_group(backend, device_id=torch.device("cuda", self.local_rank))
            else:
                dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        return self._reduce(v, "max")

    def sum(self, v: float) -> float:
        return self._reduce(v, "sum")

    def min(self, v: float) -> float:
        return -self._reduce(-v, "max")

    def _reduce(self, v: float, op: str) -> float:
        if self.pg is None:
            return float(v)
        import torch

        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()
            self.pg = None


def aggregate(bytes_per_rank: float, seconds_per_rank: float, dist: Dist, steps: int) -> dict:
    """Whole-job throughput: the bytes every rank processed over the slowest rank's time."""
    t_max = dist.max(seconds_per_rank)
    total = dist.sum(bytes_per_rank)
    return {"value": total / t_max / 1e9, "seconds": t_max, "ms_per_step": t_max / steps * 1e3,
            "total_bytes": total}


# ----------------------------------------------------------------- peaks ---


NOMINAL_HBM_GBS = 7700.0   # B300 HBM3e, nominal


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "fp8_token_group_bf16_b300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(kernel: str, key: str):
    """DRAM bytes per launch of `kernel` on workload `key` from the committed
    ncu summary (profiles/dram_traffic.txt), or None if absent or taken on a
    different kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src_hash, val = None, None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line.startswith("kernel_source_sha256"):
                src_hash = line.split("=", 1)[1].strip()
            elif line.startswith(kernel + " ") and "=" in line:
                _, rest = line.split(" ", 1)
                k, v = rest.rsplit("=", 1)
                if k.strip() == key:
                    val = int(v.strip())
    if val is None or src_hash != kernel_source_hash():
        return None
    return val


# ---------------------------------------------------------------- clocks ---


class ClockSampler:
    """Samples SM clock and clock-event (throttle) reasons while the timed
    region runs: through NVML when the Python bindings are importable, else
    by polling `nvidia-smi` (the same fields).  Samples are kept with their
    wall time; `summary(t0, t1)` reports those inside [t0, t1]."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4,
        "hw_slowdown": 0x8, "sync_boost": 0x10, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80, "display_clock_setting": 0x100,
    }

    def __init__(self, cuda_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples = []  # (wall time, SM MHz, reasons bitmask)
        self.max_mhz = None
        self.mode = None
        self.error = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None
        self.bus = None
        try:
            import torch

            p = torch.cuda.get_device_properties(cuda_index)
            self.bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except Exception:
            self.bus = None
        try:
            import pynvml

            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = (pynvml.nvmlDeviceGetHandleByPciBusId(self.bus.encode()) if self.bus
                      else pynvml.nvmlDeviceGetHandleByIndex(cuda_index))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self._reasons_fn = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.mode = "nvml"
        except Exception as e:
            import shutil

            self.error = f"nvml: {type(e).__name__}"
            if shutil.which("nvidia-smi"):
                self.mode = "nvidia-smi"
                self.target = self.bus or str(cuda_index)

    def _poll_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append((time.perf_counter(), nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM),
                                     int(self._reasons_fn(self.h))))
            except Exception:
                pass
            time.sleep(self.period)

    def _read_smi(self):
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 3:
                continue
            try:
                mhz, mx = float(parts[0]), float(parts[1])
                reasons = int(parts[2], 16)
            except ValueError:
                continue
            self.max_mhz = mx
            self.samples.append((time.perf_counter(), mhz, reasons))

    def start(self):
        if self.mode == "nvml":
            self._t = threading.Thread(target=self._poll_nvml, daemon=True)
            self._t.start()
        elif self.mode == "nvidia-smi":
            import subprocess

            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target,
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read_smi, daemon=True)
            self._t.start()
            t_end = time.perf_counter() + 5.0
            while not self.samples and time.perf_counter() < t_end and self._proc.poll() is None:
                time.sleep(0.01)
        return self

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._t is not None:
            self._t.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        where = "timed region"
        if not inside and self.samples:
            before = [s for s in self.samples if s[0] < t0][-1:]
            after = [s for s in self.samples if s[0] > t1][:1]
            inside, where = before + after, "adjacent to the timed region (shorter than the period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"],
                    "source": self.mode, "error": self.error}
        bits = 0
        for s in inside:
            bits |= s[2]
        names = [n for n, b in self.REASONS.items() if bits & b]
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(inside), "source": self.mode, "window": where}


# -------------------------------------------------------------- workload ---


def workload_inputs(T: int = STEP_T):
    """Seeded host (CPU) bf16 inputs of one step."""
    from fp8_token_group_bf16_b300 import inputs

    return {
        "per_token_group_fp8_quant": (inputs.heavy_tailed_input(T, A_H, inputs.sweep_seed(T)),),
        "rms_norm_per_block_quant": (inputs.lognormal_channel_input(T, B_H, inputs.mix_seed(T)),
                                     inputs.rms_weight(B_H)),
        "silu_and_mul_per_block_quant": (inputs.lognormal_channel_input(T, 2 * C_I, inputs.mix_seed(T) + 50),),
    }


STEP_OPTS = {
    "per_token_group_fp8_quant": dict(ue8m0=True, col=True),
    "rms_norm_per_block_quant": dict(ue8m0=True, col=False),
    "silu_and_mul_per_block_quant": dict(ue8m0=True, col=False),
}


class DeviceStep:
    """Device buffers of one step and the raw C-ABI launches on a stream."""

    def __init__(self, host, stream, T: int = STEP_T):
        import torch

        import fp8_token_group_bf16_b300 as fq

        self.fq, self.T, self.stream = fq, T, stream
        dev = torch.device("cuda", torch.cuda.current_device())
        xa = host["per_token_group_fp8_quant"][0].to(dev)
        xb, wb = (t.to(dev) for t in host["rms_norm_per_block_quant"])
        xc = host["silu_and_mul_per_block_quant"][0].to(dev)
        e4 = torch.float8_e4m3fn
        self.bufs = {
            "per_token_group_fp8_quant": dict(x=xa, q=torch.empty(T, A_H, dtype=e4, device=dev),
                                              s=torch.empty(A_H // GROUP, T, device=dev)),
            "rms_norm_per_block_quant": dict(x=xb, w=wb, q=torch.empty(T, B_H, dtype=e4, device=dev),
                                             s=torch.empty(T, B_H // GROUP, device=dev)),
            "silu_and_mul_per_block_quant": dict(x=xc, q=torch.empty(T, C_I, dtype=e4, device=dev),
                                                 s=torch.empty(T, C_I // GROUP, device=dev)),
        }
        self.bytes = {
            "per_token_group_fp8_quant": algorithmic_bytes("per_token_group_fp8_quant", T, A_H),
            "rms_norm_per_block_quant": algorithmic_bytes("rms_norm_per_block_quant", T, B_H),
            "silu_and_mul_per_block_quant": algorithmic_bytes("silu_and_mul_per_block_quant", T, C_I),
        }
        self.ops = list(self.bufs)

    def launch(self, op: str) -> None:
        fq, b, T, st = self.fq, self.bufs[op], self.T, self.stream.cuda_stream
        o = STEP_OPTS[op]
        if op == "per_token_group_fp8_quant":
            rc = fq.fp8q_per_token_group_quant(b["x"].data_ptr(), b["q"].data_ptr(), b["s"].data_ptr(), T,
                                               A_H, GROUP, 1e-10, int(o["ue8m0"]), int(o["col"]), st)
        elif op == "rms_norm_per_block_quant":
            rc = fq.fp8q_rms_norm_per_block_quant(b["x"].data_ptr(), None, b["w"].data_ptr(),
                                                  b["q"].data_ptr(), b["s"].data_ptr(), T, B_H, GROUP,
                                                  1e-6, int(o["ue8m0"]), int(o["col"]), st)
        else:
            rc = fq.fp8q_silu_and_mul_per_block_quant(b["x"].data_ptr(), b["q"].data_ptr(),
                                                      b["s"].data_ptr(), T, C_I, GROUP, 1e-10,
                                                      int(o["ue8m0"]), int(o["col"]), st)
        if rc != 0:
            raise RuntimeError(f"{op}: {fq.fp8q_status_string(rc)}")


def time_device(step: DeviceStep, steps: int, warmup: int, dist: Dist):
    """K steps of the three launches back to back, bracketed by barrier +
    synchronize, timed with one pair of CUDA events on the launching stream.
    No event sits between two kernels: it would stop the second from being
    scheduled while the first drains (the per-op figures come from
    per_op_records and chain_record instead)."""
    import torch

    st = step.stream
    for _ in range(warmup):
        for op in step.ops:
            step.launch(op)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record(st)
    for _ in range(steps):
        for op in step.ops:
            step.launch(op)
    end.record(st)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    dist.barrier()
    return start.elapsed_time(end) / 1e3, (t0, t1)


class E2EPipeline:
    """One end-to-end step through the public tensor API from pinned host
    memory: copy the three inputs in, run the three ops, copy every output
    (codes and scales) out.

    The host link, not the kernels, bounds this, so a step is pipelined over
    `chunks` token slices on three streams: slice i's inputs go in on the
    copy-in stream while slice i-1 is computed and slice i-2's outputs go out
    on the copy-out stream.  Rows are independent in all three ops, so a slice
    is a complete call of each op on its rows; op A's column-major scales
    come back per slice ([G, rows of the slice] each).  Each step waits for
    the previous step's readers of the buffers it overwrites."""

    def __init__(self, host, chunks: int = 8):
        import torch

        self.torch = torch
        dev = torch.device("cuda", torch.cuda.current_device())
        pinned = {op: tuple(t.pin_memory() for t in ts) for op, ts in host.items()}
        self.xa_h = pinned["per_token_group_fp8_quant"][0]
        self.xb_h, self.wb_h = pinned["rms_norm_per_block_quant"][:2]
        self.xc_h = pinned["silu_and_mul_per_block_quant"][0]
        T = self.T = self.xa_h.shape[0]
        chunks = max(1, min(chunks, T))
        self.bounds = [(T * i // chunks, T * (i + 1) // chunks) for i in range(chunks)]
        self.xa_d, self.xb_d, self.xc_d = (torch.empty_like(t, device=dev) for t in (self.xa_h, self.xb_h, self.xc_h))
        self.wb_d = torch.empty_like(self.wb_h, device=dev)
        self.h2d = sum(t.numel() * t.element_size() for t in (self.xa_h, self.xb_h, self.wb_h, self.xc_h))
        self.streams = [torch.cuda.Stream() for _ in range(3)]
        self.outs_dev, self.outs_host = [], []
        ha, hb, hc = self.xa_h.shape[1], self.xb_h.shape[1], self.xc_h.shape[1] // 2
        for lo, hi in self.bounds:   # per-slice output buffers, device and pinned host
            n = hi - lo
            shapes = [((n, ha), torch.float8_e4m3fn), ((ha // 128, n), torch.float32),
                      ((n, hb), torch.float8_e4m3fn), ((n, hb // 128), torch.float32),
                      ((n, hc), torch.float8_e4m3fn), ((n, hc // 128), torch.float32)]
            self.outs_dev.append([torch.empty(sh, dtype=dt, device=dev) for sh, dt in shapes])
            self.outs_host.append([torch.empty(sh, dtype=dt, pin_memory=True) for sh, dt in shapes])
        self.d2h = sum(o.numel() * o.element_size() for os_ in self.outs_dev for o in os_)
        self.prev_c_done, self.prev_out = None, [None] * len(self.bounds)

    def step(self):
        import fp8_token_group_bf16_b300 as fq

        torch = self.torch
        s_in, s_c, s_out = self.streams
        ev_in = [torch.cuda.Event() for _ in self.bounds]
        ev_c = [torch.cuda.Event() for _ in self.bounds]
        ev_out = [torch.cuda.Event() for _ in self.bounds]
        with torch.cuda.stream(s_in):
            if self.prev_c_done is not None:
                s_in.wait_event(self.prev_c_done)
            self.wb_d.copy_(self.wb_h, non_blocking=True)
            for i, (lo, hi) in enumerate(self.bounds):
                self.xa_d[lo:hi].copy_(self.xa_h[lo:hi], non_blocking=True)
                self.xb_d[lo:hi].copy_(self.xb_h[lo:hi], non_blocking=True)
                self.xc_d[lo:hi].copy_(self.xc_h[lo:hi], non_blocking=True)
                ev_in[i].record(s_in)
        for i, (lo, hi) in enumerate(self.bounds):
            s_c.wait_event(ev_in[i])
            if self.prev_out[i] is not None:
                s_c.wait_event(self.prev_out[i])
            qa, sa, qb, sb, qc, sc = self.outs_dev[i]
            fq.per_token_group_fp8_quant(self.xa_d[lo:hi], ue8m0=True, column_major_scales=True, q=qa,
                                         scales=sa.t(), stream=s_c)
            fq.rms_norm_per_block_quant(self.xb_d[lo:hi], self.wb_d, ue8m0=True, q=qb, scales=sb, stream=s_c)
            fq.silu_and_mul_per_block_quant(self.xc_d[lo:hi], ue8m0=True, q=qc, scales=sc, stream=s_c)
            ev_c[i].record(s_c)
        c_done = torch.cuda.Event()
        c_done.record(s_c)
        with torch.cuda.stream(s_out):
            for i in range(len(self.bounds)):
                s_out.wait_event(ev_c[i])
                for o, h in zip(self.outs_dev[i], self.outs_host[i]):
                    h.copy_(o, non_blocking=True)
                ev_out[i].record(s_out)
        self.prev_c_done, self.prev_out = c_done, ev_out


def host_link_ceiling(h2d_bytes: int, d2h_bytes: int, reps: int = 5) -> dict:
    """The host link's own rate for one step's bytes: plain copies of
    h2d_bytes from pinned host memory and d2h_bytes back, each alone and both
    at once on two streams (median of `reps` after one warm-up, host wall
    clock).  No kernel runs; it is the ceiling the end-to-end number is
    read against."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device())
    hin = torch.empty(h2d_bytes, dtype=torch.uint8, pin_memory=True)
    hout = torch.empty(d2h_bytes, dtype=torch.uint8, pin_memory=True)
    din = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dout = torch.zeros(d2h_bytes, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def once(h2d: bool, d2h: bool) -> float:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if h2d:
            with torch.cuda.stream(s_in):
                din.copy_(hin, non_blocking=True)
        if d2h:
            with torch.cuda.stream(s_out):
                hout.copy_(dout, non_blocking=True)
        torch.cuda.synchronize()
        return time.perf_counter() - t0

    def rate(h2d: bool, d2h: bool) -> float:
        once(h2d, d2h)
        secs = statistics.median(once(h2d, d2h) for _ in range(reps))
        return ((h2d_bytes if h2d else 0) + (d2h_bytes if d2h else 0)) / secs / 1e9

    out = {"h2d_alone_GBps": round(rate(True, False), 1), "d2h_alone_GBps": round(rate(False, True), 1),
           "both_GBps": round(rate(True, True), 1)}
    del hin, hout, din, dout
    return out


def time_e2e(host, steps: int, dist: Dist, chunks: int = 8):
    """The end-to-end metric: `steps` pipelined steps (E2EPipeline) between
    two synchronisations, host wall clock, max over ranks."""
    import torch

    pipe = E2EPipeline(host, chunks)
    pipe.step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        pipe.step()
    torch.cuda.synchronize()
    secs = time.perf_counter() - t0
    dist.barrier()
    agg = aggregate(step_bytes(pipe.T) * steps, secs, dist, steps)
    link = host_link_ceiling(pipe.h2d, pipe.d2h)
    # the slowest rank's link against the slowest rank's step time
    link = {k: round(dist.min(v), 1) for k, v in link.items()}
    link["frac"] = round((pipe.h2d + pipe.d2h) / (agg["ms_per_step"] * 1e-3) / 1e9 / link["both_GBps"], 4)
    link["ranks"] = "each rate is the minimum over ranks"
    return {"value": round(agg["value"], 2), "unit": UNIT, "h2d_bytes_per_step": pipe.h2d,
            "d2h_bytes_per_step": pipe.d2h, "steps": steps, "ms_per_step": round(agg["ms_per_step"], 3),
            "pipeline": f"{len(pipe.bounds)} token slices, copy-in / compute / copy-out streams",
            "host_link": link}


# ------------------------------------------------------------ CPU oracle ---


def oracle_sample_run(host, rows: int) -> tuple[float, int]:
    """Run the CPU oracle on the first `rows` tokens of each op; returns
    (seconds, algorithmic bytes of the sample)."""
    import numpy as np

    import oracle
    from fp8_token_group_bf16_b300 import inputs

    xa = np.ascontiguousarray(inputs.bits(host["per_token_group_fp8_quant"][0])[:rows])
    xb = np.ascontiguousarray(inputs.bits(host["rms_norm_per_block_quant"][0])[:rows])
    wb = inputs.bits(host["rms_norm_per_block_quant"][1])
    xc = np.ascontiguousarray(inputs.bits(host["silu_and_mul_per_block_quant"][0])[:rows])
    t0 = time.perf_counter()
    oracle.per_token_group_quant(xa, ue8m0=True, col_major=True)
    oracle.rms_norm_per_block_quant(xb, wb, None, ue8m0=True)
    oracle.silu_and_mul_per_block_quant(xc, ue8m0=True)
    secs = time.perf_counter() - t0
    return secs, step_bytes(rows)


def cpu_baseline(host, T: int = STEP_T, target_s: float = 10.0) -> dict:
    secs, _ = oracle_sample_run(host, 8)
    rows = max(8, min(T, int(8 * target_s / max(secs, 1e-6))))
    secs, nbytes = oracle_sample_run(host, rows)
    return {"value": round(nbytes / secs / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {rows} of {T} tokens of each of the three ops "
                      f"({nbytes / 1e6:.1f} MB algorithmic, {secs:.1f} s, single-threaded C)"}


def step_config(T: int = STEP_T) -> dict:
    mb = step_bytes(T) / 1e6
    return {
        "workload": f"Qwen3-32B-shaped FP8 quant epilogues, T={T} tokens per step: "
                    f"per_token_group_fp8_quant [{T},{A_H}] heavy-tailed (UE8M0, column-major scales); "
                    f"rms_norm_per_block_quant [{T},{B_H}] lognormal channels (UE8M0, row-major); "
                    f"silu_and_mul_per_block_quant [{T},{2 * C_I}] lognormal channels (UE8M0, row-major); "
                    "group 128",
        "T": T, "H_group_quant": A_H, "H_rms": B_H, "I_silu": C_I, "group": GROUP,
        "l2": (f"inputs larger than L2: a step touches {mb:.0f} MB (> 126 MB L2), so every "
               "buffer is evicted by the other two ops before it is read again") if mb > 2 * 126
              else f"a step touches {mb:.0f} MB, not much more than the 126 MB L2: not a bandwidth figure",
        "parallelism": "one independent batch per GPU (weak scaling, no collective)",
    }


def reference_arm(args):
    """The CPU oracle as the reference arm (run on rank 0 only)."""
    host = workload_inputs(STEP_T)
    t1, _ = oracle_sample_run(host, 2)
    per_step = args.reference_budget_s / (args.steps + args.warmup)
    rows = max(1, min(STEP_T, int(2 * per_step / max(t1, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample_run(host, rows)
    secs, nbytes = 0.0, 0
    for _ in range(args.steps):
        s, b = oracle_sample_run(host, rows)
        secs += s
        nbytes += b
    value = round(nbytes / secs / 1e9, 4)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
        "config": step_config(),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {rows} of {STEP_T} tokens of each op per step "
                                   "(single-threaded C oracle)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------ isolated op timing --

L2_BYTES = 126 << 20
RECORD_T = (512, 4096, 16384)   # the per-op record of the default run
CHAIN_T = 512
STEP_SHAPES = {   # op: (row length H or I, scale layout) as in the step
    "per_token_group_fp8_quant": (A_H, "col"),
    "rms_norm_per_block_quant": (B_H, "row"),
    "silu_and_mul_per_block_quant": (C_I, "row"),
}


def graph_time_us(make, nbytes: int, iters: int, reps: int = 5) -> float:
    """Per-launch device time (us) of `iters` back-to-back calls captured in
    one CUDA graph, cycling over enough independent buffer sets (each from
    make()) that their bytes exceed 3x L2, so no call finds its inputs in L2
    from an earlier one.  Median over `reps` replays, each bracketed by CUDA
    events on the stream the graph is replayed on."""
    import torch

    nsets = min(64, max(2, int(3 * L2_BYTES // max(nbytes, 1)) + 1))
    calls = [make() for _ in range(nsets)]
    for c in calls:
        c()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g):
            for k in range(iters):
                calls[k % nsets]()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / iters)
    del g, calls
    torch.cuda.empty_cache()
    return statistics.median(ts) * 1e3


def copy_maker(nbytes: int):
    """A same-size copy on the SMs (an elementwise x * 1 over fp32 words,
    reading and writing nbytes in total): a plain device-to-device memcpy may
    be handed to a copy engine, which is slower at some sizes."""
    import torch

    def make():
        n = max(1, nbytes // 8)
        a = torch.zeros(n, dtype=torch.float32, device="cuda")
        b = torch.empty(n, dtype=torch.float32, device="cuda")
        return lambda: torch.mul(a, 1.0, out=b)
    return make


def step_op_maker(op: str, T: int, seed: int):
    """make() for one of the step's ops at T tokens, with the step's options
    (UE8M0; op A column-major scales) on fresh device buffers drawn from the
    step's distributions by a seeded device generator."""
    import torch

    import fp8_token_group_bf16_b300 as fq
    from fp8_token_group_bf16_b300 import inputs

    H, lay = STEP_SHAPES[op]
    G = H // GROUP
    counter = [0]

    def make():
        counter[0] += 1
        sd = seed + 7919 * counter[0]
        q = torch.empty(T, H, dtype=torch.float8_e4m3fn, device="cuda")
        if op == "per_token_group_fp8_quant":
            x = inputs.device_heavy_tailed_input(T, H, sd, "cuda")
            s = torch.empty(G, T, device="cuda").t()
            return lambda: fq.per_token_group_fp8_quant(x, ue8m0=True, column_major_scales=True, q=q, scales=s)
        s = torch.empty(T, G, device="cuda")
        if op == "rms_norm_per_block_quant":
            x = inputs.device_lognormal_channel_input(T, H, sd, "cuda")
            w = (1.0 + 0.1 * torch.randn(H, generator=torch.Generator(device="cuda").manual_seed(sd + 1),
                                         device="cuda")).to(torch.bfloat16)
            return lambda: fq.rms_norm_per_block_quant(x, w, None, ue8m0=True, q=q, scales=s)
        x = inputs.device_lognormal_channel_input(T, 2 * H, sd, "cuda")
        return lambda: fq.silu_and_mul_per_block_quant(x, ue8m0=True, q=q, scales=s)
    return make


def _iters(nbytes: int) -> int:
    return 200 if nbytes < 50e6 else 40


def per_op_records(peak: float, T_values=RECORD_T) -> list:
    """The metric itself: each of the step's three ops alone at each T, its
    algorithmic bytes over its per-launch time (graph replay, inputs rotated
    past L2), beside a same-size SM copy timed the same way."""
    rows = []
    for T in T_values:
        for i, op in enumerate(STEP_SHAPES):
            H, lay = STEP_SHAPES[op]
            nbytes = algorithmic_bytes(op, T, H)
            us = graph_time_us(step_op_maker(op, T, 9000 + 10 * T + i), nbytes, _iters(nbytes))
            cus = graph_time_us(copy_maker(nbytes), nbytes, _iters(nbytes))
            gbs, cgbs = nbytes / us / 1e3, nbytes / cus / 1e3
            rows.append({"op": op, "T": T, "H_or_I": H, "scales": f"UE8M0 {lay}-major", "bytes": nbytes,
                         "us": round(us, 3), "GBps": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                         "copy_us": round(cus, 3), "copy_GBps": round(cgbs, 1),
                         "copy_frac_of_peak": round(cgbs / peak, 4)})
    return rows


def chain_record(peak: float, T: int = CHAIN_T) -> dict:
    """The step's three ops back to back at T as dependent launches (no event
    between them), in one graph over rotated buffer sets; ops A and B get
    their marginal cost inside the chain: t(A, B, C) - t(B, C) and
    t(A, B, C) - t(A, C)."""
    ops = list(STEP_SHAPES)
    makers = {op: step_op_maker(op, T, 9500 + i) for i, op in enumerate(ops)}
    nb = {op: algorithmic_bytes(op, T, STEP_SHAPES[op][0]) for op in ops}

    def chain(sel):
        def make():
            calls = [makers[op]() for op in sel]

            def run():
                for c in calls:
                    c()
            return run
        nbytes = sum(nb[op] for op in sel)
        return graph_time_us(make, nbytes, _iters(nbytes))

    t_abc, t_bc, t_ac = chain(ops), chain(ops[1:]), chain([ops[0], ops[2]])
    out = {"T": T, "step_us": round(t_abc, 3), "step_GBps": round(sum(nb.values()) / t_abc / 1e3, 1),
           "method": "graph of back-to-back dependent launches (A, B, C), buffers rotated past 3x L2; "
                     "marginal = t(A,B,C) minus the chain without the op"}
    for op, rest in ((ops[0], t_bc), (ops[1], t_ac)):
        m = t_abc - rest
        out[op] = {"marginal_us": round(m, 3), "GBps": round(nb[op] / m / 1e3, 1) if m > 0 else None,
                   "frac_of_peak": round(nb[op] / m / 1e3 / peak, 4) if m > 0 else None}
    return out


# ------------------------------------------------------------------ sweep --


def sweep(args):
    """Per-op T sweeps; each point: back-to-back launches in a CUDA graph over
    buffer sets rotated past 3x L2, median of 5 replays, and the same-size
    device-to-device copy for comparison."""
    import torch

    import fp8_token_group_bf16_b300 as fq

    fq.load()
    dev = torch.device("cuda")
    peak, peak_kind = load_peaks()
    clocks = ClockSampler(torch.cuda.current_device()).start()
    try:
        t0 = time.perf_counter()
        rows = _sweep_points(fq, dev, peak, peak_kind)
        t1 = time.perf_counter()
    finally:
        clocks.stop()
    # one line for the whole sweep: the SM clock and clock-event reasons over its replays
    print(json.dumps({"sweep_clocks": clocks.summary(t0, t1)}), flush=True)
    return rows


def _sweep_points(fq, dev, peak, peak_kind):
    import torch

    timed = graph_time_us

    e4 = torch.float8_e4m3fn
    points = []   # (op, T, H or I, ue8m0, scale layout, residual)
    for T in (1, 4, 16, 64, 256, 512, 1024, 4096, 16384):
        for ue8m0, lay in ((False, "row"), (True, "col")):
            points.append(("per_token_group_fp8_quant", T, A_H, ue8m0, lay, False))
    for T in (1, 8, 64, 512, 4096, 16384):
        points.append(("rms_norm_per_block_quant", T, B_H, True, "row", False))
        points.append(("silu_and_mul_per_block_quant", T, C_I, True, "row", False))
    points.append(("rms_norm_per_block_quant", 256, 4096, False, "row", True))
    points.append(("rms_norm_per_block_quant", 256, 4096, False, "row", False))
    points.append(("silu_and_mul_per_block_quant", 1024, 12288, True, "col", False))
    for T in (4096, 16384):   # short rows: a warp per row
        points.append(("rms_norm_per_block_quant", T, 1024, True, "row", False))
    points.append(("rms_norm_per_block_quant", 65536, 128, True, "row", False))   # eight rows to a warp
    for H in (16384, 32768):   # long rows: a wide CTA per row
        points.append(("rms_norm_per_block_quant", 4096, H, True, "row", False))
    for T in (512, 4096):   # packed UE8M0 exponent bytes, and the same bytes in MXFP8 GEMM tiles
        for lay in ("packed", "mx"):
            points.append(("per_token_group_fp8_quant", T, A_H, True, lay, False))
            points.append(("rms_norm_per_block_quant", T, B_H, True, lay, False))
            points.append(("silu_and_mul_per_block_quant", T, C_I, True, lay, False))
    for T in (64, 512, 4096, 16384):   # per-token variants, one scale per row
        points.append(("dynamic_per_token_scaled_fp8_quant", T, A_H, False, "token", False))
        points.append(("rms_norm_dynamic_per_token_quant", T, B_H, False, "token", False))
        points.append(("silu_and_mul_dynamic_per_token_quant", T, C_I, False, "token", False))
    rows = []
    for op, T, H, ue8m0, lay, res in points:
        nbytes = algorithmic_bytes(op, T, H, res, packed=lay == "packed", mx=lay == "mx")
        G = H // GROUP

        def make(op=op, T=T, H=H, ue8m0=ue8m0, lay=lay, res=res, G=G):
            xin = torch.randn(T, 2 * H if op.startswith("silu") else H, device=dev).to(torch.bfloat16)
            q = torch.empty(T, H, dtype=e4, device=dev)
            if lay == "token":
                s = torch.empty(T, 1, device=dev)
                if op == "dynamic_per_token_scaled_fp8_quant":
                    return lambda: fq.dynamic_per_token_scaled_fp8_quant(xin, ue8m0=ue8m0, q=q, scales=s)
                if op == "silu_and_mul_dynamic_per_token_quant":
                    return lambda: fq.silu_and_mul_dynamic_per_token_quant(xin, ue8m0=ue8m0, q=q, scales=s)
                w = torch.randn(H, device=dev).to(torch.bfloat16)
                return lambda: fq.rms_norm_dynamic_per_token_quant(xin, w, None, ue8m0=ue8m0, q=q, scales=s)
            if lay == "packed":
                s = torch.empty(fq.packed_scale_shape(T, G), dtype=torch.int32, device=dev)
            elif lay == "mx":
                s = torch.empty(fq.mx_scale_shape(T, G), dtype=torch.uint8, device=dev)
            else:
                s = torch.empty(G, T, device=dev).t() if lay == "col" else torch.empty(T, G, device=dev)
            kw = dict(ue8m0=ue8m0, column_major_scales=lay == "col", packed_ue8m0_scales=lay == "packed",
                      mx_scales=lay == "mx", q=q, scales=s)
            if op == "per_token_group_fp8_quant":
                return lambda: fq.per_token_group_fp8_quant(xin, **kw)
            if op == "silu_and_mul_per_block_quant":
                return lambda: fq.silu_and_mul_per_block_quant(xin, **kw)
            w = torch.randn(H, device=dev).to(torch.bfloat16)
            r = torch.randn(T, H, device=dev).to(torch.bfloat16) if res else None
            return lambda: fq.rms_norm_per_block_quant(xin, w, r, **kw)

        iters = 200 if nbytes < 50e6 else 40
        us = timed(make, nbytes, iters)
        cus = timed(copy_maker(nbytes), nbytes, iters)
        torch.cuda.empty_cache()
        row = {"op": op, "T": T, "H_or_I": H, "ue8m0": ue8m0, "scales": lay, "residual": res,
               "bytes": nbytes, "us": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
               "frac_of_peak": round(nbytes / us / 1e3 / peak, 4),
               "frac_of_nominal": round(nbytes / us / 1e3 / NOMINAL_HBM_GBS, 4), "copy_us": round(cus, 3),
               "copy_GBps": round(nbytes / cus / 1e3, 1), "peak": peak, "peak_kind": peak_kind}
        rows.append(row)
        print(json.dumps(row), flush=True)

    # fused_qk_norm_rope, Qwen3-32B attention shape (64 query, 8 key/value heads of 128)
    from fp8_token_group_bf16_b300 import inputs as _inputs
    table = _inputs.rotary_table(_inputs.QK_P).to(dev)
    qw = (1.0 + 0.1 * torch.randn(128, device=dev)).to(torch.bfloat16)
    kw = (1.0 + 0.1 * torch.randn(128, device=dev)).to(torch.bfloat16)
    for T in (64, 256, 512, 4096, 16384):
        nbytes = qk_rope_bytes(T)

        def make(T=T):
            qkv = torch.randn(T, 80 * 128, device=dev).to(torch.bfloat16)
            pos = torch.randint(0, _inputs.QK_P, (T,), device=dev, dtype=torch.int64)
            return lambda: fq.fused_qk_norm_rope(qkv, qw, kw, table, pos, 64, 8)

        iters = 200 if nbytes < 50e6 else 40
        us = timed(make, nbytes, iters)
        cus = timed(copy_maker(nbytes), nbytes, iters)
        torch.cuda.empty_cache()
        row = {"op": "fused_qk_norm_rope", "T": T, "H_or_I": "64q+8kv x 128", "ue8m0": None, "scales": None,
               "residual": False, "bytes": nbytes, "us": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
               "frac_of_peak": round(nbytes / us / 1e3 / peak, 4),
               "frac_of_nominal": round(nbytes / us / 1e3 / NOMINAL_HBM_GBS, 4), "copy_us": round(cus, 3),
               "copy_GBps": round(nbytes / cus / 1e3, 1), "peak": peak, "peak_kind": peak_kind}
        rows.append(row)
        print(json.dumps(row), flush=True)
    return rows


# ------------------------------------------------------------ one op ------

SINGLE_OPS = {
    # op: (row length, ue8m0, scale layout)
    "per_token_group_fp8_quant": (A_H, True, "col"),
    "rms_norm_per_block_quant": (B_H, True, "row"),
    "silu_and_mul_per_block_quant": (C_I, True, "row"),
    "dynamic_per_token_scaled_fp8_quant": (A_H, False, "token"),
    "rms_norm_dynamic_per_token_quant": (B_H, False, "token"),
    "silu_and_mul_dynamic_per_token_quant": (C_I, False, "token"),
    "fused_qk_norm_rope": (None, None, None),
}


def single_op(args):
    """--op NAME: W warm-up launches, then K launches of one op at T = --tokens
    on one stream, timed with CUDA events; inputs rotated over enough buffer
    sets to exceed 3x L2.  One JSON line (op, T, us per launch, GB/s,
    fraction of the measured copy bandwidth).  Made for profiling one kernel."""
    import torch

    import fp8_token_group_bf16_b300 as fq
    from fp8_token_group_bf16_b300 import inputs as _inputs

    fq.load()
    dev = torch.device("cuda")
    op, T = args.op, args.tokens
    H, ue8m0, lay = SINGLE_OPS[op]
    if op == "fused_qk_norm_rope":
        nbytes = qk_rope_bytes(T)
        table = _inputs.rotary_table(_inputs.QK_P).to(dev)
        w = (1.0 + 0.1 * torch.randn(128, device=dev)).to(torch.bfloat16)
    else:
        nbytes = algorithmic_bytes(op, T, H, packed=args.packed, mx=args.mx)
    nsets = min(16, max(2, int(3 * (126 << 20) // nbytes) + 1))
    calls = []
    for _ in range(nsets):
        if op == "fused_qk_norm_rope":
            qkv = torch.randn(T, 80 * 128, device=dev).to(torch.bfloat16)
            pos = torch.randint(0, _inputs.QK_P, (T,), device=dev, dtype=torch.int64)
            calls.append(lambda qkv=qkv, pos=pos: fq.fused_qk_norm_rope(qkv, w, w, table, pos, 64, 8))
            continue
        x = torch.randn(T, 2 * H if "silu" in op else H, device=dev).to(torch.bfloat16)
        q = torch.empty(T, H, dtype=torch.float8_e4m3fn, device=dev)
        if lay == "token":
            f = getattr(fq, op)
            if op.startswith("rms"):
                wt = torch.randn(H, device=dev).to(torch.bfloat16)
                calls.append(lambda x=x, q=q, wt=wt: fq.rms_norm_dynamic_per_token_quant(x, wt, None, q=q))
            else:
                calls.append(lambda x=x, q=q, f=f: f(x, q=q))
            continue
        kw = dict(ue8m0=ue8m0 or args.packed or args.mx,
                  column_major_scales=lay == "col" and not (args.packed or args.mx),
                  packed_ue8m0_scales=args.packed, mx_scales=args.mx, q=q)
        if op.startswith("rms"):
            wt = torch.randn(H, device=dev).to(torch.bfloat16)
            calls.append(lambda x=x, wt=wt, kw=kw: fq.rms_norm_per_block_quant(x, wt, None, **kw))
        else:
            f = getattr(fq, op)
            calls.append(lambda x=x, f=f, kw=kw: f(x, **kw))
    for k in range(args.warmup):
        calls[k % nsets]()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for k in range(args.steps):
        calls[k % nsets]()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / args.steps
    peak, kind = load_peaks()
    print(json.dumps({"op": op, "T": T, "packed": args.packed, "mx": args.mx, "launches": args.steps, "us": round(us, 3),
                      "GBps": round(nbytes / us / 1e3, 1), "frac_of_peak": round(nbytes / us / 1e3 / peak, 4),
                      "peak": peak, "peak_kind": kind}), flush=True)


# ------------------------------------------------------------------- main --


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--sweep", action="store_true")
    p.add_argument("--op", choices=sorted(SINGLE_OPS), default=None,
                   help="time one op at --tokens (K launches after W warm-ups) instead of the step")
    p.add_argument("--packed", action="store_true", help="with --op: packed UE8M0 scales (per-group ops)")
    p.add_argument("--mx", action="store_true", help="with --op: MXFP8 scale tiles (per-group ops)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-records", action="store_true",
                   help="skip the per-op T records and the chained step (for profiling the step alone)")
    p.add_argument("--tokens", type=int, default=STEP_T,
                   help="tokens per step (default: the T=4096 workload; smaller values are for profiling)")
    p.add_argument("--reference-budget-s", type=float, default=120.0,
                   help="CPU seconds the reference arm spends over all its steps")
    return p.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        # rank 0 alone times the oracle; the other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            reference_arm(args)
        return
    import torch

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    dist = Dist()
    try:
        torch.cuda.set_device(dist.local_rank)
        if args.sweep:
            if dist.rank == 0:
                sweep(args)
            return
        if args.op:
            if dist.rank == 0:
                single_op(args)
            return
        import fp8_token_group_bf16_b300 as fq

        fq.load()
        T = args.tokens
        host = workload_inputs(T)
        stream = torch.cuda.Stream()
        step = DeviceStep(host, stream, T)
        peak, peak_kind = load_peaks()
        clocks = ClockSampler(torch.cuda.current_device()).start()
        try:
            secs, window = time_device(step, args.steps, args.warmup, dist)
            records, chain = None, None
            if not args.no_records:
                # isolated per-op records and the chained step, rank 0 only (one GPU's figures)
                records = per_op_records(peak) if dist.rank == 0 else None
                chain = chain_record(peak) if dist.rank == 0 else None
            t_end = time.perf_counter()
        finally:
            clocks.stop()
        agg = aggregate(step_bytes(T) * args.steps, secs, dist, args.steps)
        # the dominant kernel alone at the step's T, from its isolated record
        # (graph replay on the launching stream, CUDA events around the replay)
        dom = next((r for r in records or [] if r["op"] == DOMINANT and r["T"] == T), None)
        roofline = {"bound": "hbm", "kernel": KERNEL_NAMES[DOMINANT], "unit": "GB/s", "peak": peak,
                    "peak_source": (f"{peak_kind}: MEASURED_PEAKS.json hbm_gbs (device copy bandwidth, burst: "
                                    "the kernel is timed alone)" if peak_kind == "measured"
                                    else "fallback 6.4 TB/s")}
        traffic = recorded_traffic(KERNEL_NAMES[DOMINANT], f"T={T} I={C_I} ue8m0 row")
        if dom is not None:
            roofline.update({"achieved": dom["GBps"], "frac": dom["frac_of_peak"],
                             "algorithmic_bytes_per_launch": dom["bytes"], "us_per_launch": dom["us"],
                             "timing": "isolated launches in a CUDA graph over buffers rotated past 3x L2",
                             "nominal_peak": NOMINAL_HBM_GBS,
                             "frac_of_nominal": round(dom["GBps"] / NOMINAL_HBM_GBS, 4)})
        roofline["traffic"] = traffic
        roofline["traffic_source"] = ("recorded, not measured in this run: DRAM read + write bytes per launch "
                                      "from the committed ncu summary profiles/dram_traffic.txt, taken on the "
                                      "current kernel sources (hash-checked)" if traffic is not None else
                                      "null: no ncu summary of the current kernel sources")
        e2e = time_e2e(host, args.e2e_steps, dist)
        line = {
            "metric": METRIC, "value": round(agg["value"], 2), "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(agg["ms_per_step"], 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded generators; no dataset)", "config": step_config(T),
            "roofline": roofline,
            "e2e": e2e,
            "gpu_launches": len(step.ops) * args.steps,
            "clocks": dict(clocks.summary(window[0], t_end),
                           window_covers="the timed steps, then the per-op records and the chained step"),
        }
        if records is not None:
            line["per_op"] = records
            line["per_op_method"] = ("each op alone at T, graph replay of back-to-back launches over buffer "
                                     "sets rotated past 3x L2, median of 5 replays; copy = a same-size SM copy "
                                     "timed the same way; inputs drawn on the device from the step's "
                                     "distributions")
        if chain is not None:
            line["chain_T512"] = chain
        if dist.rank == 0 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(host, T)
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
