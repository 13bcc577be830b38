// The three quantisation kernels for sm_103a.
//
// All three are HBM-bound streaming kernels: a handful of fp32 operations per
// byte moved, no contraction, so no tensor cores.  A quad of lanes owns a
// group (32 values per lane); every lane issues all of its loads before any
// arithmetic so several 64-byte requests per thread are in flight.
#pragma once

#include "fp8q_device.cuh"

namespace fp8q {

constexpr int kCtaThreads = 256;                               // ops A and C
constexpr int kGroupsPerCta = kCtaThreads / kLanesPerGroup;    // 64
constexpr int kGroupQuantGpt = 2;                              // groups per quad, op A

// Row t and group g of flat group index gi (G groups per row).  The host
// guarantees T*G < 2^31 (2^38 bf16 values would not fit in HBM anyway), so a
// 32-bit division suffices.
__device__ __forceinline__ void split_group(int64_t gi, int64_t G, int64_t &t, int64_t &g)
{
    const uint32_t tt = uint32_t(gi) / uint32_t(G);
    t = tt;
    g = gi - int64_t(tt) * G;
}

// --------------------------------------------------------------------------
// per_token_group_fp8_quant
//
// A contiguous [T, H] tensor is a flat sequence of T*G groups, so the kernel
// walks groups, not rows.  CTA b owns groups [b*64*GPT, (b+1)*64*GPT); quad q
// of the CTA takes groups b*64*GPT + j*64 + q for j < GPT, so the 8 quads of
// a warp read 8 adjacent groups (2 KiB) per pair of load instructions.
// Out-of-range quads load a clamped, valid group and store nothing.
// --------------------------------------------------------------------------
template <bool UE8M0, bool COL, bool V8>
__global__ void __launch_bounds__(kCtaThreads) group_quant_kernel(const uint16_t *__restrict__ x,
                                                                  uint8_t *__restrict__ q,
                                                                  float *__restrict__ scales,
                                                                  int64_t n_groups, int64_t G,
                                                                  int64_t T, float eps)
{
    constexpr int GPT = kGroupQuantGpt;
    const int sub = threadIdx.x & (kLanesPerGroup - 1);
    const int64_t first = int64_t(blockIdx.x) * kGroupsPerCta * GPT + (threadIdx.x / kLanesPerGroup);

    wait_for_producer();
    allow_consumer_launch();
    uint32_t raw[GPT][16];
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
        const int64_t gi = first + int64_t(j) * kGroupsPerCta;
        const int64_t gl = gi < n_groups ? gi : n_groups - 1;
        ld64_stream<V8>(x + gl * kGroup + sub * kValsPerLane, raw[j]);
    }
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
        const int64_t gi = first + int64_t(j) * kGroupsPerCta;
        float v[32];
        unpack32(raw[j], v);
        const float amax = quad_max(absmax32(v));
        const float s = group_scale<UE8M0>(amax, eps);
        const float r = scale_recip<UE8M0>(s);
        uint32_t codes[8];
        quant32<UE8M0>(v, s, r, codes);
        if (gi < n_groups) {
            st32<V8>(q + gi * kGroup + sub * kValsPerLane, codes);
            if (sub == 0) {
                if (COL) {
                    int64_t t, g;
                    split_group(gi, G, t, g);
                    scales[g * T + t] = s;
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
// One output group per quad: output group gi = (t, g) reads the gate values
// x[t, g*128 ...] and the up values x[t, I + g*128 ...] (64 bytes of each per
// lane, both loads issued first).
// --------------------------------------------------------------------------
__device__ __forceinline__ float silu_mul(float a, float b)
{
    const float d = __fadd_rn(1.0f, expf(-a));
    return __fmul_rn(__fdiv_rn(a, d), b);
}

template <bool UE8M0, bool COL, bool V8>
__global__ void __launch_bounds__(kCtaThreads) silu_quant_kernel(const uint16_t *__restrict__ x,
                                                                 uint8_t *__restrict__ q,
                                                                 float *__restrict__ scales,
                                                                 int64_t n_groups, int64_t G,
                                                                 int64_t T, int64_t I, float eps)
{
    const int sub = threadIdx.x & (kLanesPerGroup - 1);
    const int64_t gi = int64_t(blockIdx.x) * kGroupsPerCta + (threadIdx.x / kLanesPerGroup);
    const int64_t gl = gi < n_groups ? gi : n_groups - 1;
    int64_t t, g;
    split_group(gl, G, t, g);
    const uint16_t *pa = x + t * 2 * I + g * kGroup + sub * kValsPerLane;
    wait_for_producer();
    allow_consumer_launch();
    uint32_t ra[16], rb[16];
    ld64_stream<V8>(pa, ra);
    ld64_stream<V8>(pa + I, rb);

    float v[32];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        v[2 * k] = silu_mul(bf_lo(ra[k]), bf_lo(rb[k]));
        v[2 * k + 1] = silu_mul(bf_hi(ra[k]), bf_hi(rb[k]));
    }
    const float amax = quad_max(absmax32(v));
    const float s = group_scale<UE8M0>(amax, eps);
    const float r = scale_recip<UE8M0>(s);
    uint32_t codes[8];
    quant32<UE8M0>(v, s, r, codes);
    if (gi < n_groups) {
        st32<V8>(q + gi * kGroup + sub * kValsPerLane, codes);
        if (sub == 0)
            scales[COL ? g * T + t : gi] = s;
    }
}

// --------------------------------------------------------------------------
// rms_norm_per_block_quant
//
// A CTA of 4*G lanes (rounded up to whole warps) owns whole rows: quad g
// holds group g of the row, 32 values per lane.  The row's sum of squares is
// reduced per lane (two interleaved fma chains), per warp (butterfly) and
// across warps through shared memory in warp order, so every lane gets the
// same value.  Lanes past the end of the row (G not a multiple of 8) hold a
// clamped copy of group G-1 and add nothing.
//
// Rows of up to 8192 values (<= 256 threads, !LONG): the CTA is persistent
// (grid = resident CTAs, rows t = blockIdx.x + k*gridDim.x), keeps its slice
// of the weight in registers across rows, and loads row t + gridDim.x while
// it reduces and quantises row t.  Longer rows (LONG, <= 1024 threads) take
// one row per CTA and read the weight after the reduction.
// --------------------------------------------------------------------------
template <bool RES, bool V8>
__device__ __forceinline__ void load_row(const uint16_t *x, const uint16_t *residual, int64_t off,
                                         uint32_t (&xr)[16], uint32_t (&rr)[16])
{
    ld64_stream<V8>(x + off, xr);
    if (RES)
        ld64_rw<V8>(residual + off, rr);
}

template <bool UE8M0, bool COL, bool RES, bool V8, bool LONG>
__global__ void __launch_bounds__(LONG ? 1024 : 256) rms_quant_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ residual, const uint16_t *__restrict__ w,
    uint8_t *__restrict__ q, float *__restrict__ scales, int64_t T, int H, int G, float eps)
{
    __shared__ float part[2][32];
    const int sub = threadIdx.x & (kLanesPerGroup - 1);
    const int g = threadIdx.x / kLanesPerGroup;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const bool ok = g < G;
    const int col = (ok ? g : G - 1) * kGroup + sub * kValsPerLane;   // clamped into the row

    wait_for_producer();
    allow_consumer_launch();
    uint32_t wr[16];
    if (!LONG)
        ld64_keep<V8>(w + col, wr);

    int64_t t = blockIdx.x;
    uint32_t cx[16], cr[16];
    load_row<RES, V8>(x, residual, t * H + col, cx, cr);

    for (int it = 0; t < T; ++it, t += gridDim.x) {
        uint32_t nx[16], nr[16];
        const int64_t tn = t + gridDim.x;
        if (!LONG && tn < T) {
            load_row<RES, V8>(x, residual, tn * H + col, nx, nr);
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k)
                nx[k] = nr[k] = 0u;
        }

        if (RES) {
            // z = bf16(x + r), written back to the residual, is what is normalised
#pragma unroll
            for (int k = 0; k < 16; ++k)
                cx[k] = pack_bf16x2(__fadd_rn(bf_lo(cx[k]), bf_lo(cr[k])), __fadd_rn(bf_hi(cx[k]), bf_hi(cr[k])));
            if (ok)
                st64<V8>(residual + t * H + col, cx);
        }

        float ss0 = 0.0f, ss1 = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            ss0 = __fmaf_rn(bf_lo(cx[k]), bf_lo(cx[k]), ss0);
            ss1 = __fmaf_rn(bf_hi(cx[k]), bf_hi(cx[k]), ss1);
        }
        const float ssw = warp_sum(ok ? __fadd_rn(ss0, ss1) : 0.0f);
        if ((threadIdx.x & 31) == 0)
            part[it & 1][warp] = ssw;
        __syncthreads();
        float tot = 0.0f;
        for (int i = 0; i < nwarps; ++i)
            tot = __fadd_rn(tot, part[it & 1][i]);

        const float mean = __fdiv_rn(tot, float(H));
        const float rstd = __fsqrt_rn(__fadd_rn(mean, eps));
        const float inv = __frcp_rn(rstd);

        if (LONG)
            ld64_keep<V8>(w + col, wr);
        float v[32];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            v[2 * k] = __fmul_rn(__fmul_rn(bf_lo(cx[k]), inv), bf_lo(wr[k]));
            v[2 * k + 1] = __fmul_rn(__fmul_rn(bf_hi(cx[k]), inv), bf_hi(wr[k]));
        }
        const float amax = quad_max(absmax32(v));
        const float s = group_scale<UE8M0>(amax, kScaleFloor);
        const float r = scale_recip<UE8M0>(s);
        uint32_t codes[8];
        quant32<UE8M0>(v, s, r, codes);
        if (ok) {
            st32<V8>(q + t * H + col, codes);
            if (sub == 0)
                scales[COL ? int64_t(g) * T + t : t * G + g] = s;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            cx[k] = nx[k];
            cr[k] = nr[k];
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
