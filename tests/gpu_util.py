"""Helpers for the GPU tests: move seeded inputs to the device, run an op
through the library's C ABI (via the package's ctypes binding) and bring the
outputs back as numpy arrays in the oracle's conventions."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_token_group_bf16_b300 as fq
from fp8_token_group_bf16_b300 import build, inputs


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the tests marked gpu")
    build.build()
    fq.load()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return inputs.from_bits(bits).cuda()


def host_codes(q: torch.Tensor) -> np.ndarray:
    return q.view(torch.uint8).cpu().numpy()


def host_scales_tg(s: torch.Tensor) -> np.ndarray:
    """Scales as a [T, G] numpy array whichever layout they are stored in."""
    return s.cpu().numpy()


def gpu_group_quant(xb, ue8m0=False, col=False):
    x = dev_bf16(xb)
    q, s = fq.per_token_group_fp8_quant(x, ue8m0=ue8m0, column_major_scales=col)
    torch.cuda.synchronize()
    return host_codes(q), host_scales_tg(s)


def gpu_rms(xb, wb, rb=None, ue8m0=False, col=False, eps=1e-6):
    x, w = dev_bf16(xb), dev_bf16(wb)
    r = dev_bf16(rb) if rb is not None else None
    q, s = fq.rms_norm_per_block_quant(x, w, r, eps=eps, ue8m0=ue8m0, column_major_scales=col)
    torch.cuda.synchronize()
    rout = inputs.bits(r.cpu()) if r is not None else None
    return host_codes(q), host_scales_tg(s), rout


def gpu_silu(xb, ue8m0=False, col=False):
    x = dev_bf16(xb)
    q, s = fq.silu_and_mul_per_block_quant(x, ue8m0=ue8m0, column_major_scales=col)
    torch.cuda.synchronize()
    return host_codes(q), host_scales_tg(s)


def sample_rows(T: int, n: int, seed: int = 0) -> np.ndarray:
    """Rows to compare when the oracle cannot afford the whole tensor: the
    first and last rows plus a seeded random subset, sorted."""
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(T, n - 2, replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(rows))
