// C ABI of libfp8q: argument checks, variant dispatch and launches.
// The contract of every entry point is stated in include/fp8q.h.
#include "fp8q.h"
#include "fp8q_kernels.cuh"

#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

namespace {

using namespace fp8q;

constexpr int kThreads = 256;           // op A / op C CTA size (16 half-warps)
constexpr int kHalfWarpsPerCta = kThreads / kLanesPerGroup;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(const void *x, const void *q, const float *scales, int64_t T, int64_t H,
                 int32_t group_size, int32_t scale_layout)
{
    if (T < 0 || H <= 0 || group_size <= 0 || H % group_size != 0)
        return FP8Q_ERR_INVALID_ARG;
    if (scale_layout != FP8Q_SCALES_ROW_MAJOR && scale_layout != FP8Q_SCALES_COL_MAJOR)
        return FP8Q_ERR_INVALID_ARG;
    if (group_size != kGroup)
        return FP8Q_ERR_UNSUPPORTED;
    if (T == 0)
        return FP8Q_OK;
    if (!x || !q || !scales)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scales, 4))
        return FP8Q_ERR_MISALIGNED;
    return FP8Q_OK;
}

bool valid_scale_eps(float eps) { return std::isfinite(eps) && eps >= 1e-30f; }

int launch_status()
{
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

// Groups per half-warp: more independent loads per thread for large inputs,
// more CTAs (more SMs pulling) for small ones.
int pick_gpt(int64_t n_groups)
{
    const int64_t ctas_at_4 = (n_groups + 4 * kHalfWarpsPerCta - 1) / (4 * kHalfWarpsPerCta);
    if (ctas_at_4 >= 4 * 148)
        return 4;
    const int64_t ctas_at_2 = (n_groups + 2 * kHalfWarpsPerCta - 1) / (2 * kHalfWarpsPerCta);
    if (ctas_at_2 >= 2 * 148)
        return 2;
    return 1;
}

template <bool U, bool C>
void launch_group(int gpt, const uint16_t *x, uint8_t *q, float *s, int64_t n, int64_t G,
                  int64_t T, float eps, cudaStream_t st)
{
    const int64_t per = int64_t(kHalfWarpsPerCta) * gpt;
    const dim3 grid(unsigned((n + per - 1) / per));
    switch (gpt) {
    case 4: group_quant_kernel<U, C, 4><<<grid, kThreads, 0, st>>>(x, q, s, n, G, T, eps); break;
    case 2: group_quant_kernel<U, C, 2><<<grid, kThreads, 0, st>>>(x, q, s, n, G, T, eps); break;
    default: group_quant_kernel<U, C, 1><<<grid, kThreads, 0, st>>>(x, q, s, n, G, T, eps); break;
    }
}

template <bool U, bool C>
void launch_silu(int gpt, const uint16_t *x, uint8_t *q, float *s, int64_t n, int64_t G,
                 int64_t T, int64_t I, float eps, cudaStream_t st)
{
    const int64_t per = int64_t(kHalfWarpsPerCta) * gpt;
    const dim3 grid(unsigned((n + per - 1) / per));
    switch (gpt) {
    case 4: silu_quant_kernel<U, C, 4><<<grid, kThreads, 0, st>>>(x, q, s, n, G, T, I, eps); break;
    case 2: silu_quant_kernel<U, C, 2><<<grid, kThreads, 0, st>>>(x, q, s, n, G, T, I, eps); break;
    default: silu_quant_kernel<U, C, 1><<<grid, kThreads, 0, st>>>(x, q, s, n, G, T, I, eps); break;
    }
}

template <bool U, bool C, bool R>
void launch_rms(int P, const uint16_t *x, uint16_t *res, const uint16_t *w, uint8_t *q,
                float *s, int64_t T, int H, int G, float eps, cudaStream_t st)
{
    const int warps = (G + 2 * P - 1) / (2 * P);
    const dim3 grid{unsigned(T)};
    const dim3 block{unsigned(32 * warps)};
    switch (P) {
    case 1: rms_quant_kernel<U, C, R, 1><<<grid, block, 0, st>>>(x, res, w, q, s, T, H, G, eps); break;
    case 2: rms_quant_kernel<U, C, R, 2><<<grid, block, 0, st>>>(x, res, w, q, s, T, H, G, eps); break;
    case 4: rms_quant_kernel<U, C, R, 4><<<grid, block, 0, st>>>(x, res, w, q, s, T, H, G, eps); break;
    default: rms_quant_kernel<U, C, R, 8><<<grid, block, 0, st>>>(x, res, w, q, s, T, H, G, eps); break;
    }
}

}  // namespace

extern "C" {

int fp8q_per_token_group_quant(const void *x, void *q, float *scales, int64_t T, int64_t H,
                               int32_t group_size, float eps, int32_t ue8m0, int32_t scale_layout,
                               void *stream)
{
    int rc = check_common(x, q, scales, T, H, group_size, scale_layout);
    if (rc != FP8Q_OK)
        return rc;
    if (!valid_scale_eps(eps))
        return FP8Q_ERR_INVALID_ARG;
    if (T == 0)
        return FP8Q_OK;
    const int64_t G = H / kGroup;
    const int64_t n = T * G;
    if (n / T != G || n > (int64_t(1) << 40))
        return FP8Q_ERR_INVALID_ARG;
    auto st = static_cast<cudaStream_t>(stream);
    auto xp = static_cast<const uint16_t *>(x);
    auto qp = static_cast<uint8_t *>(q);
    const int gpt = pick_gpt(n);
    const bool col = scale_layout == FP8Q_SCALES_COL_MAJOR;
    if (ue8m0) {
        if (col) launch_group<true, true>(gpt, xp, qp, scales, n, G, T, eps, st);
        else     launch_group<true, false>(gpt, xp, qp, scales, n, G, T, eps, st);
    } else {
        if (col) launch_group<false, true>(gpt, xp, qp, scales, n, G, T, eps, st);
        else     launch_group<false, false>(gpt, xp, qp, scales, n, G, T, eps, st);
    }
    return launch_status();
}

int fp8q_silu_and_mul_per_block_quant(const void *x, void *q, float *scales, int64_t T, int64_t I,
                                      int32_t group_size, float eps, int32_t ue8m0,
                                      int32_t scale_layout, void *stream)
{
    int rc = check_common(x, q, scales, T, I, group_size, scale_layout);
    if (rc != FP8Q_OK)
        return rc;
    if (!valid_scale_eps(eps))
        return FP8Q_ERR_INVALID_ARG;
    if (T == 0)
        return FP8Q_OK;
    const int64_t G = I / kGroup;
    const int64_t n = T * G;
    if (n / T != G || n > (int64_t(1) << 40))
        return FP8Q_ERR_INVALID_ARG;
    auto st = static_cast<cudaStream_t>(stream);
    auto xp = static_cast<const uint16_t *>(x);
    auto qp = static_cast<uint8_t *>(q);
    const int gpt = pick_gpt(n);
    const bool col = scale_layout == FP8Q_SCALES_COL_MAJOR;
    if (ue8m0) {
        if (col) launch_silu<true, true>(gpt, xp, qp, scales, n, G, T, I, eps, st);
        else     launch_silu<true, false>(gpt, xp, qp, scales, n, G, T, I, eps, st);
    } else {
        if (col) launch_silu<false, true>(gpt, xp, qp, scales, n, G, T, I, eps, st);
        else     launch_silu<false, false>(gpt, xp, qp, scales, n, G, T, I, eps, st);
    }
    return launch_status();
}

int fp8q_rms_norm_per_block_quant(const void *x, void *residual, const void *weight, void *q,
                                  float *scales, int64_t T, int64_t H, int32_t group_size,
                                  float eps, int32_t ue8m0, int32_t scale_layout, void *stream)
{
    int rc = check_common(x, q, scales, T, H, group_size, scale_layout);
    if (rc != FP8Q_OK)
        return rc;
    if (!std::isfinite(eps) || eps < 0.0f)
        return FP8Q_ERR_INVALID_ARG;
    if (H > FP8Q_RMS_MAX_H)
        return FP8Q_ERR_UNSUPPORTED;
    if (T == 0)
        return FP8Q_OK;
    if (!weight)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(weight, 16) || (residual && !aligned(residual, 16)))
        return FP8Q_ERR_MISALIGNED;
    if (T > 0x7FFFFFFF)
        return FP8Q_ERR_INVALID_ARG;
    const int G = int(H / kGroup);
    int P = 8;
    for (int p : {2, 4, 8}) {
        if ((G + 2 * p - 1) / (2 * p) <= 32) {
            P = p;
            break;
        }
    }
    if (G <= 2)
        P = 1;
    auto st = static_cast<cudaStream_t>(stream);
    auto xp = static_cast<const uint16_t *>(x);
    auto rp = static_cast<uint16_t *>(residual);
    auto wp = static_cast<const uint16_t *>(weight);
    auto qp = static_cast<uint8_t *>(q);
    const bool col = scale_layout == FP8Q_SCALES_COL_MAJOR;
    const int h = int(H);
#define FP8Q_RMS(U, C)                                                                           \
    (rp ? launch_rms<U, C, true>(P, xp, rp, wp, qp, scales, T, h, G, eps, st)                    \
        : launch_rms<U, C, false>(P, xp, rp, wp, qp, scales, T, h, G, eps, st))
    if (ue8m0) {
        if (col) FP8Q_RMS(true, true);
        else     FP8Q_RMS(true, false);
    } else {
        if (col) FP8Q_RMS(false, true);
        else     FP8Q_RMS(false, false);
    }
#undef FP8Q_RMS
    return launch_status();
}

int fp8q_f32_to_e4m3(const float *v, void *out, int64_t n, void *stream)
{
    if (n < 0)
        return FP8Q_ERR_INVALID_ARG;
    if (n == 0)
        return FP8Q_OK;
    if (!v || !out)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(v, 16) || !aligned(out, 16))
        return FP8Q_ERR_MISALIGNED;
    const int64_t threads = (n + 3) / 4;
    const dim3 grid(unsigned((threads + 255) / 256));
    if (grid.x == 0 || (threads + 255) / 256 > 0x7FFFFFFF)
        return FP8Q_ERR_INVALID_ARG;
    f32_to_e4m3_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        v, static_cast<uint8_t *>(out), n);
    return launch_status();
}

const char *fp8q_status_string(int status)
{
    switch (status) {
    case FP8Q_OK: return "FP8Q_OK";
    case FP8Q_ERR_INVALID_ARG: return "FP8Q_ERR_INVALID_ARG: invalid argument";
    case FP8Q_ERR_UNSUPPORTED: return "FP8Q_ERR_UNSUPPORTED: unsupported group size or row length";
    case FP8Q_ERR_MISALIGNED: return "FP8Q_ERR_MISALIGNED: pointer not aligned as required";
    case FP8Q_ERR_CUDA: return "FP8Q_ERR_CUDA: CUDA launch failed";
    default: return "unknown fp8q status";
    }
}

int fp8q_version(void) { return 100; }

}  // extern "C"
