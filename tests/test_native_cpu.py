"""libfp8q on a machine without a GPU: it builds for sm_103a, loads, exports
exactly the C ABI that include/fp8q.h declares, and rejects bad arguments on
the host before touching CUDA.  No call here reaches a kernel launch."""

import ctypes
import os
import re
import subprocess

import pytest

import fp8_token_group_bf16_b300 as fq
from fp8_token_group_bf16_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fq.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8q_\w+)\s*\(", text)))


def test_header_declares_the_three_ops():
    names = declared_functions()
    for n in ("fp8q_per_token_group_quant", "fp8q_rms_norm_per_block_quant",
              "fp8q_silu_and_mul_per_block_quant", "fp8q_status_string"):
        assert n in names


def test_exports_match_header(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted({l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("fp8q_")})
    assert exported == declared_functions()
    for n in declared_functions():
        assert hasattr(lib, n)
    assert sorted(fq.EXPORTS) == declared_functions()


def test_only_c_abi_symbols_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    text_syms = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert all(s.startswith("fp8q_") for s in text_syms), [s for s in text_syms if not s.startswith("fp8q_")][:5]


def test_built_for_sm103a_only(lib):
    """The build compiles one target, sm_103a machine code (no PTX for a
    driver to recompile): a GPU of another architecture refuses the kernels
    instead of running something else.  The -m gpu tests, which launch every
    kernel on a B300, are the other half of this check."""
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    flags = build.NVCC_FLAGS
    assert flags[: len(build.ARCH)] == build.ARCH
    assert not any("compute_" in f and f not in build.ARCH for f in flags)


def test_status_strings(lib):
    for s in range(5):
        assert fq.fp8q_status_string(s).startswith("FP8Q_")
    assert "unknown" in fq.fp8q_status_string(99)
    assert fq.fp8q_version() >= 100


# Fake, never-dereferenced device addresses: every call below is rejected by
# the host-side checks before any CUDA call.
A = 0x7F0000000000
Q = 0x7F0000100000
S = 0x7F0000200000


def test_rejects_bad_shapes(lib):
    E = fq.FP8Q_ERR_INVALID_ARG
    assert fq.fp8q_per_token_group_quant(A, Q, S, -1, 512, 128, 1e-10, 0, 0, None) == E
    assert fq.fp8q_per_token_group_quant(A, Q, S, 4, 0, 128, 1e-10, 0, 0, None) == E
    assert fq.fp8q_per_token_group_quant(A, Q, S, 4, 500, 128, 1e-10, 0, 0, None) == E
    assert fq.fp8q_per_token_group_quant(A, Q, S, 4, 512, 128, 1e-10, 0, 5, None) == E
    assert fq.fp8q_per_token_group_quant(None, Q, S, 4, 512, 128, 1e-10, 0, 0, None) == E
    assert fq.fp8q_silu_and_mul_per_block_quant(A, Q, S, 4, 100, 128, 1e-10, 0, 0, None) == E
    assert fq.fp8q_rms_norm_per_block_quant(A, None, None, Q, S, 4, 512, 128, 1e-6, 0, 0, None) == E


def test_packed_scales_need_ue8m0(lib):
    """The packed layout holds exponent bytes, so it only takes power-of-two
    scales: without ue8m0 every op refuses it before any CUDA call."""
    E = fq.FP8Q_ERR_INVALID_ARG
    P = fq.FP8Q_SCALES_UE8M0_PACKED
    assert fq.fp8q_per_token_group_quant(A, Q, S, 4, 512, 128, 1e-10, 0, P, None) == E
    assert fq.fp8q_silu_and_mul_per_block_quant(A, Q, S, 4, 512, 128, 1e-10, 0, P, None) == E
    assert fq.fp8q_rms_norm_per_block_quant(A, None, A, Q, S, 4, 512, 128, 1e-6, 0, P, None) == E
    # with ue8m0 it passes the checks: an empty input is then a no-op
    assert fq.fp8q_per_token_group_quant(None, None, None, 0, 512, 128, 1e-10, 1, P, None) == 0
    X = fq.FP8Q_SCALES_UE8M0_MX   # the MXFP8 tile layout likewise
    assert fq.fp8q_per_token_group_quant(A, Q, S, 4, 512, 128, 1e-10, 0, X, None) == E
    assert fq.fp8q_silu_and_mul_per_block_quant(A, Q, S, 4, 512, 128, 1e-10, 0, X, None) == E
    assert fq.fp8q_rms_norm_per_block_quant(A, None, A, Q, S, 4, 512, 128, 1e-6, 0, X, None) == E
    assert fq.fp8q_per_token_group_quant(None, None, None, 0, 512, 128, 1e-10, 1, X, None) == 0
    assert fq.fp8q_per_token_group_quant(A, Q, S, 4, 512, 128, 1e-10, 1, 4, None) == E


def test_packed_scale_shape():
    assert fq.packed_scale_shape(5, 6) == (2, 8)
    assert fq.packed_scale_shape(4096, 56) == (14, 4096)
    assert fq.packed_scale_shape(1, 1) == (1, 4)
    # the header's byte count agrees with the binding's shape
    text = open(HEADER).read()
    assert "#define FP8Q_PACKED_SCALE_BYTES(T, G) ((((G) + 3) / 4) * (((T) + 3) / 4 * 4) * 4)" in text
    for T, G in [(5, 6), (4096, 56), (1, 1), (7, 192)]:
        k, tp = fq.packed_scale_shape(T, G)
        assert k * tp * 4 == (((G) + 3) // 4) * (((T) + 3) // 4 * 4) * 4
    assert "#define FP8Q_MX_SCALE_BYTES(T, G) ((((T) + 127) / 128 * 128) * 4 * (G))" in text
    for T, G in [(5, 6), (4096, 56), (1, 1), (129, 200)]:
        r, c = fq.mx_scale_shape(T, G)
        assert r * c == (((T) + 127) // 128 * 128) * 4 * (G) and r % 128 == 0 and c == 4 * G


def test_per_token_checks(lib):
    E, U, M = fq.FP8Q_ERR_INVALID_ARG, fq.FP8Q_ERR_UNSUPPORTED, fq.FP8Q_ERR_MISALIGNED
    for f in (fq.fp8q_dynamic_per_token_scaled_fp8_quant, fq.fp8q_silu_and_mul_dynamic_per_token_quant):
        assert f(A, Q, S, -1, 512, 1e-10, 0, None) == E
        assert f(A, Q, S, 4, 0, 1e-10, 0, None) == E
        assert f(A, Q, S, 4, 512, 0.0, 0, None) == E
        assert f(A, Q, S, 4, 500, 1e-10, 0, None) == U                    # not a multiple of 128
        assert f(A, Q, S, 4, fq.FP8Q_TOKEN_MAX_COLS + 128, 1e-10, 0, None) == U
        assert f(A + 2, Q, S, 4, 512, 1e-10, 0, None) == M
        assert f(A, Q + 8, S, 4, 512, 1e-10, 0, None) == M
        assert f(A, Q, S + 2, 4, 512, 1e-10, 1, None) == M
        assert f(None, None, None, 0, 512, 1e-10, 1, None) == 0
        assert f(None, Q, S, 4, 512, 1e-10, 0, None) == E
    r = fq.fp8q_rms_norm_dynamic_per_token_quant
    assert r(A, None, A, Q, S, -1, 512, 1e-6, 0, None) == E
    assert r(A, None, A, Q, S, 4, 500, 1e-6, 0, None) == U
    assert r(A, None, A, Q, S, 4, fq.FP8Q_RMS_MAX_H + 128, 1e-6, 0, None) == U
    assert r(A, None, A, Q, S, 4, 512, -1.0, 0, None) == E
    assert r(A, None, None, Q, S, 4, 512, 1e-6, 0, None) == E
    assert r(A, A + 8, A, Q, S, 4, 512, 1e-6, 0, None) == M
    assert r(A, None, A, Q, S + 1, 4, 512, 1e-6, 0, None) == M
    assert r(None, None, None, None, None, 0, 512, 1e-6, 0, None) == 0


def test_qk_norm_rope_checks(lib):
    E, U, M = fq.FP8Q_ERR_INVALID_ARG, fq.FP8Q_ERR_UNSUPPORTED, fq.FP8Q_ERR_MISALIGNED
    f = fq.fp8q_fused_qk_norm_rope
    assert f(A, A, A, A, S, -1, 64, 8, 128, 4096, 1e-6, 1, None) == E
    assert f(A, A, A, A, S, 4, -1, 8, 128, 4096, 1e-6, 1, None) == E
    assert f(A, A, A, A, S, 4, 64, 8, 128, 0, 1e-6, 1, None) == E
    assert f(A, A, A, A, S, 4, 64, 8, 128, 4096, -1.0, 1, None) == E
    assert f(A, A, A, A, S, 4, 64, 8, 0, 4096, 1e-6, 1, None) == E
    assert f(A, A, A, A, S, 4, 64, 8, 64, 4096, 1e-6, 1, None) == U       # only 128-value heads
    assert f(A, A, A, A, S + 4, 4, 64, 8, 128, 4096, 1e-6, 1, None) == M  # positions 8-byte aligned
    assert f(A + 2, A, A, A, S, 4, 64, 8, 128, 4096, 1e-6, 1, None) == M
    assert f(A, A, A, A + 8, S, 4, 64, 8, 128, 4096, 1e-6, 0, None) == M
    assert f(None, A, A, A, S, 4, 64, 8, 128, 4096, 1e-6, 1, None) == E
    assert f(None, None, None, None, None, 0, 64, 8, 128, 4096, 1e-6, 1, None) == 0
    assert f(None, None, None, None, None, 4, 0, 0, 128, 4096, 1e-6, 1, None) == 0


def test_rejects_bad_eps(lib):
    E = fq.FP8Q_ERR_INVALID_ARG
    for eps in (0.0, -1.0, float("inf"), float("nan"), 1e-38):
        assert fq.fp8q_per_token_group_quant(A, Q, S, 4, 512, 128, eps, 0, 0, None) == E
        assert fq.fp8q_silu_and_mul_per_block_quant(A, Q, S, 4, 512, 128, eps, 0, 0, None) == E
    for eps in (-1e-6, float("inf"), float("nan")):
        assert fq.fp8q_rms_norm_per_block_quant(A, None, A, Q, S, 4, 512, 128, eps, 0, 0, None) == E


def test_unsupported(lib):
    U = fq.FP8Q_ERR_UNSUPPORTED
    assert fq.fp8q_per_token_group_quant(A, Q, S, 4, 512, 64, 1e-10, 0, 0, None) == U
    assert fq.fp8q_rms_norm_per_block_quant(A, None, A, Q, S, 4, 512, 256, 1e-6, 0, 0, None) == U
    assert fq.fp8q_rms_norm_per_block_quant(A, None, A, Q, S, 4, fq.FP8Q_RMS_MAX_H + 128, 128, 1e-6,
                                            0, 0, None) == U
    assert fq.fp8q_rms_norm_per_block_quant(A, A + 64, A, Q, S, 4, fq.FP8Q_RMS_MAX_H + 128, 128,
                                            1e-6, 0, 0, None) == U


def test_misaligned(lib):
    M = fq.FP8Q_ERR_MISALIGNED
    assert fq.fp8q_per_token_group_quant(A + 2, Q, S, 4, 512, 128, 1e-10, 0, 0, None) == M
    assert fq.fp8q_per_token_group_quant(A, Q + 8, S, 4, 512, 128, 1e-10, 0, 0, None) == M
    assert fq.fp8q_per_token_group_quant(A, Q, S + 2, 4, 512, 128, 1e-10, 0, 0, None) == M
    assert fq.fp8q_silu_and_mul_per_block_quant(A + 4, Q, S, 4, 512, 128, 1e-10, 0, 0, None) == M
    assert fq.fp8q_rms_norm_per_block_quant(A, A + 8, A, Q, S, 4, 512, 128, 1e-6, 0, 0, None) == M
    assert fq.fp8q_rms_norm_per_block_quant(A, None, A + 2, Q, S, 4, 512, 128, 1e-6, 0, 0, None) == M
    assert fq.fp8q_f32_to_e4m3(A + 4, Q, 16, None) == M
    assert fq.fp8q_silu_mul(A + 4, A, A, 16, None) == M
    assert fq.fp8q_silu_mul(A, A, A, -1, None) == fq.FP8Q_ERR_INVALID_ARG
    assert fq.fp8q_silu_mul(None, None, None, 0, None) == 0
    assert fq.fp8q_group_scale(A + 2, A, 16, 1e-10, 0, None) == M
    assert fq.fp8q_group_scale(A, A, -1, 1e-10, 0, None) == fq.FP8Q_ERR_INVALID_ARG
    assert fq.fp8q_group_scale(A, A, 16, 0.0, 0, None) == fq.FP8Q_ERR_INVALID_ARG
    assert fq.fp8q_group_scale(None, A, 16, 1e-10, 1, None) == fq.FP8Q_ERR_INVALID_ARG
    assert fq.fp8q_group_scale(None, None, 0, 1e-10, 0, None) == 0
    assert fq.fp8q_quant_pairs(A + 2, A, Q, 16, None) == M
    assert fq.fp8q_quant_pairs(A, A + 2, Q, 16, None) == M
    assert fq.fp8q_quant_pairs(A, A, Q, -1, None) == fq.FP8Q_ERR_INVALID_ARG
    assert fq.fp8q_quant_pairs(A, None, Q, 16, None) == fq.FP8Q_ERR_INVALID_ARG
    assert fq.fp8q_quant_pairs(None, None, None, 0, None) == 0


def test_empty_input_is_a_no_op(lib):
    # T == 0 returns before any CUDA call, even with null pointers.
    assert fq.fp8q_per_token_group_quant(None, None, None, 0, 512, 128, 1e-10, 0, 0, None) == 0
    assert fq.fp8q_silu_and_mul_per_block_quant(None, None, None, 0, 512, 128, 1e-10, 1, 1, None) == 0
    assert fq.fp8q_rms_norm_per_block_quant(None, None, None, None, None, 0, 512, 128, 1e-6, 0, 0, None) == 0
    assert fq.fp8q_f32_to_e4m3(None, None, 0, None) == 0


def test_tensor_api_refuses_cpu_tensors(lib):
    import torch

    x = torch.zeros(4, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fq.per_token_group_fp8_quant(x)
    with pytest.raises(ValueError, match="CUDA"):
        fq.silu_and_mul_per_block_quant(x)
    with pytest.raises(ValueError, match="CUDA"):
        fq.rms_norm_per_block_quant(x, torch.ones(512, dtype=torch.bfloat16))


def test_missing_library_fails_loudly(tmp_path):
    import importlib

    saved = fq._lib
    fq._lib = None
    try:
        with pytest.raises(ImportError, match="not found"):
            fq.load(str(tmp_path / "libfp8q.so"))
    finally:
        fq._lib = saved
