// The three quantisation kernels for sm_103a.
//
// All three are HBM-bound streaming kernels: a handful of fp32 operations per
// byte moved, no contraction, so no tensor cores.  Each lane moves its data
// with 16-byte vector loads issued before any arithmetic, so a thread keeps
// several independent loads in flight.
#pragma once

#include "fp8q_device.cuh"

namespace fp8q {

// Index of a group's scale in the chosen layout (row t, group g of G).
template <bool COL>
__device__ __forceinline__ int64_t scale_index(int64_t t, int64_t g, int64_t T, int64_t G)
{
    return COL ? g * T + t : t * G + g;
}

// --------------------------------------------------------------------------
// per_token_group_fp8_quant
//
// A contiguous [T, H] tensor is a flat sequence of T*G groups, so the kernel
// walks groups, not rows: half-warp h of CTA b handles groups
// b*HPB*GPT + j*HPB + h for j < GPT (HPB half-warps per CTA).  The two
// half-warps of a warp take adjacent groups, so every load instruction of a
// warp reads 512 contiguous bytes.  All GPT loads are issued first.
// --------------------------------------------------------------------------
template <bool UE8M0, bool COL, int GPT>
__global__ void __launch_bounds__(256) group_quant_kernel(const uint16_t *__restrict__ x,
                                                          uint8_t *__restrict__ q,
                                                          float *__restrict__ scales,
                                                          int64_t n_groups, int64_t G, int64_t T,
                                                          float eps)
{
    const int lane = threadIdx.x & (kLanesPerGroup - 1);
    const int hpb = blockDim.x / kLanesPerGroup;
    const int64_t first = int64_t(blockIdx.x) * hpb * GPT + (threadIdx.x / kLanesPerGroup);

    uint4 raw[GPT];
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
        const int64_t gi = first + int64_t(j) * hpb;
        raw[j] = gi < n_groups ? ld_stream16(x + gi * kGroup + lane * kValsPerLane)
                               : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
        const int64_t gi = first + int64_t(j) * hpb;
        float v[8];
        unpack8(raw[j], v);
        const float amax = halfwarp_max(absmax8(v));
        const float s = group_scale<UE8M0>(amax, eps);
        const float r = __frcp_rn(s);
        const uint2 codes = quant8<UE8M0>(v, s, r);
        if (gi < n_groups) {
            st8(q + gi * kGroup + lane * kValsPerLane, codes);
            if (lane == 0) {
                if (COL) {
                    const int64_t t = gi / G;
                    scales[scale_index<true>(t, gi - t * G, T, G)] = s;
                } else {
                    scales[gi] = s;
                }
            }
        }
    }
}

// --------------------------------------------------------------------------
// silu_and_mul_per_block_quant
//
// Same group walk over the T*G output groups; output group (t, g) reads the
// gate vector at x[t, g*128 ...] and the up vector at x[t, I + g*128 ...].
// --------------------------------------------------------------------------
__device__ __forceinline__ float silu_mul(float a, float b)
{
    const float d = __fadd_rn(1.0f, expf(-a));
    return __fmul_rn(__fdiv_rn(a, d), b);
}

template <bool UE8M0, bool COL, int GPT>
__global__ void __launch_bounds__(256) silu_quant_kernel(const uint16_t *__restrict__ x,
                                                         uint8_t *__restrict__ q,
                                                         float *__restrict__ scales,
                                                         int64_t n_groups, int64_t G, int64_t T,
                                                         int64_t I, float eps)
{
    const int lane = threadIdx.x & (kLanesPerGroup - 1);
    const int hpb = blockDim.x / kLanesPerGroup;
    const int64_t first = int64_t(blockIdx.x) * hpb * GPT + (threadIdx.x / kLanesPerGroup);

    uint4 ra[GPT], rb[GPT];
    int64_t row[GPT];
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
        const int64_t gi = first + int64_t(j) * hpb;
        const int64_t t = gi / G;
        row[j] = t;
        const int64_t off = t * 2 * I + (gi - t * G) * kGroup + lane * kValsPerLane;
        const bool ok = gi < n_groups;
        ra[j] = ok ? ld_stream16(x + off) : make_uint4(0u, 0u, 0u, 0u);
        rb[j] = ok ? ld_stream16(x + off + I) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
        const int64_t gi = first + int64_t(j) * hpb;
        float a[8], b[8], v[8];
        unpack8(ra[j], a);
        unpack8(rb[j], b);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[k] = silu_mul(a[k], b[k]);
        const float amax = halfwarp_max(absmax8(v));
        const float s = group_scale<UE8M0>(amax, eps);
        const float r = __frcp_rn(s);
        const uint2 codes = quant8<UE8M0>(v, s, r);
        if (gi < n_groups) {
            st8(q + gi * kGroup + lane * kValsPerLane, codes);
            if (lane == 0)
                scales[COL ? scale_index<true>(row[j], gi - row[j] * G, T, G) : gi] = s;
        }
    }
}

// --------------------------------------------------------------------------
// rms_norm_per_block_quant, one CTA per token row.
//
// blockDim = 32 * W threads, W = ceil(G / (2P)); half-warp h holds groups
// h, h + 2W, ..., (P of them), all loaded before any arithmetic.  The row's
// sum of squares is reduced per thread (sequential fma over its values), per
// warp (butterfly), then across warps through shared memory in warp order,
// so every thread ends with the same value.  The optional residual add
// z = bf16(x + r) is written back before the norm.
// --------------------------------------------------------------------------
template <bool UE8M0, bool COL, bool RES, int P>
__global__ void __launch_bounds__(1024) rms_quant_kernel(const uint16_t *__restrict__ x,
                                                         uint16_t *__restrict__ residual,
                                                         const uint16_t *__restrict__ w,
                                                         uint8_t *__restrict__ q,
                                                         float *__restrict__ scales, int64_t T,
                                                         int H, int G, float eps)
{
    __shared__ float part[32];
    const int64_t t = blockIdx.x;
    const int lane = threadIdx.x & (kLanesPerGroup - 1);
    const int hw = threadIdx.x / kLanesPerGroup;
    const int hpb = blockDim.x / kLanesPerGroup;
    const int nwarps = blockDim.x / 32;

    // Short rows load the weight with the row; long rows (P > 2) re-read it
    // from L1/L2 at the end instead of holding it in registers.
    constexpr bool kWeightEarly = P <= 2;
    constexpr int PW = kWeightEarly ? P : 1;
    uint4 rz[P], rw[PW];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        const int g = hw + j * hpb;
        const int64_t off = t * H + int64_t(g) * kGroup + lane * kValsPerLane;
        const bool ok = g < G;
        rz[j] = ok ? ld_stream16(x + off) : make_uint4(0u, 0u, 0u, 0u);
        if (kWeightEarly)
            rw[j % PW] = ok ? ld_keep16(w + g * kGroup + lane * kValsPerLane) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (RES) {
        uint4 rr[P];
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const int g = hw + j * hpb;
            const int64_t off = t * H + int64_t(g) * kGroup + lane * kValsPerLane;
            rr[j] = g < G ? ld_rw16(residual + off) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const int g = hw + j * hpb;
            float a[8], b[8];
            unpack8(rz[j], a);
            unpack8(rr[j], b);
            uint4 z;
            z.x = pack_bf16x2(__fadd_rn(a[0], b[0]), __fadd_rn(a[1], b[1]));
            z.y = pack_bf16x2(__fadd_rn(a[2], b[2]), __fadd_rn(a[3], b[3]));
            z.z = pack_bf16x2(__fadd_rn(a[4], b[4]), __fadd_rn(a[5], b[5]));
            z.w = pack_bf16x2(__fadd_rn(a[6], b[6]), __fadd_rn(a[7], b[7]));
            rz[j] = z;
            if (g < G)
                st16(residual + t * H + int64_t(g) * kGroup + lane * kValsPerLane, z);
        }
    }

    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
        float z[8];
        unpack8(rz[j], z);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            ss = __fmaf_rn(z[k], z[k], ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0)
        part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int i = 0; i < nwarps; ++i)
        tot = __fadd_rn(tot, part[i]);

    const float mean = __fdiv_rn(tot, float(H));
    const float rstd = __fsqrt_rn(__fadd_rn(mean, eps));
    const float inv = __frcp_rn(rstd);

#pragma unroll
    for (int j = 0; j < P; ++j) {
        const int g = hw + j * hpb;
        float z[8], wv[8], v[8];
        unpack8(rz[j], z);
        if (kWeightEarly)
            unpack8(rw[j % PW], wv);
        else
            unpack8(g < G ? ld_keep16(w + g * kGroup + lane * kValsPerLane) : make_uint4(0u, 0u, 0u, 0u), wv);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[k] = __fmul_rn(__fmul_rn(z[k], inv), wv[k]);
        const float amax = halfwarp_max(absmax8(v));
        const float s = group_scale<UE8M0>(amax, kScaleFloor);
        const float r = __frcp_rn(s);
        const uint2 codes = quant8<UE8M0>(v, s, r);
        if (g < G) {
            st8(q + t * H + int64_t(g) * kGroup + lane * kValsPerLane, codes);
            if (lane == 0)
                scales[scale_index<COL>(t, g, T, G)] = s;
        }
    }
}

// --------------------------------------------------------------------------
// Elementwise fp32 -> e4m3 (the conversion on its own, for checking it).
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256) f32_to_e4m3_kernel(const float *__restrict__ v,
                                                          uint8_t *__restrict__ out, int64_t n)
{
    const int64_t i4 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (i4 + 4 <= n) {
        const float4 f = *reinterpret_cast<const float4 *>(v + i4);
        *reinterpret_cast<uint32_t *>(out + i4) = pack4_e4m3(f.x, f.y, f.z, f.w);
    } else if (i4 < n) {
        for (int64_t i = i4; i < n; ++i) {
            const uint32_t c = pack4_e4m3(v[i], 0.f, 0.f, 0.f);
            out[i] = uint8_t(c & 0xFFu);
        }
    }
}

}  // namespace fp8q
