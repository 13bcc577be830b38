// Device helpers shared by the three quantisation kernels: vector memory
// access, bf16 unpacking, the half-warp group reduction, the group scale,
// the correctly rounded quotient and the packed e4m3 conversion.
//
// A group is 128 consecutive bf16 values of one token row (the Block_FP8
// "1x128 activation scaling" of "Helion：用自动调优改进 vLLM 推理", section
// Scope).  It is held by one half-warp: 16 lanes x 8 values, one 16-byte load
// per lane, so a warp covers two groups = 512 contiguous bytes per load.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp8q {

constexpr int kGroup = 128;
constexpr int kLanesPerGroup = 16;  // half-warp
constexpr int kValsPerLane = 8;     // one 16-byte bf16 vector
constexpr float kFp8Max = 448.0f;   // largest finite float8_e4m3fn
constexpr float kScaleFloor = 1e-10f;

// ------------------------------------------------------------- memory ---

// Loads and stores go through CUDA's intrinsics rather than inline asm so the
// compiler treats them as memory accesses that may fault and never hoists one
// above the bounds check that guards it.

// 16-byte load of data read exactly once (ld.global.cs: evict-first).
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}

// 16-byte load of data every CTA re-reads (the RMSNorm weight): read-only path.
__device__ __forceinline__ uint4 ld_keep16(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// 16-byte load of data this kernel also writes (the residual).
__device__ __forceinline__ uint4 ld_rw16(const void *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ void st16(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

__device__ __forceinline__ void st8(void *p, uint2 v) { *reinterpret_cast<uint2 *>(p) = v; }

// --------------------------------------------------------------- bf16 ---

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);          // lower address
        f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

// Two fp32 -> packed bf16x2 with round to nearest even (lo at the lower address).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------- reductions ---

// Max over the 16 lanes of a half-warp.  Every lane of the warp must call it
// (the shuffles name the full mask); the two half-warps reduce independently.
__device__ __forceinline__ float halfwarp_max(float m)
{
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    return m;
}

__device__ __forceinline__ float warp_sum(float s)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, o));
    return s;
}

// ------------------------------------------------------------ scale -----

// s = RN32(max(amax, eps) / 448); with UE8M0 the smallest power of two >= s.
// eps >= 1e-30 (checked on the host) keeps s a normal number, so the power of
// two is the exponent field bumped by one whenever any mantissa bit is set.
template <bool UE8M0>
__device__ __forceinline__ float group_scale(float amax, float eps)
{
    float s = __fdiv_rn(fmaxf(amax, eps), kFp8Max);
    if (UE8M0) {
        uint32_t u = __float_as_uint(s);
        if (u & 0x007FFFFFu)
            u = (u & 0x7F800000u) + 0x00800000u;
        s = __uint_as_float(u);
    }
    return s;
}

// Correctly rounded |x| / s, given r = RN32(1/s).
//
// Power-of-two s: r is exactly 1/s, so one multiply is the exact quotient
// rounded once.  Otherwise: y0 = RN(x r) is within 1.5 ulp of x/s; one
// residual step y1 = RN(y0 + RN(x - s y0) r) makes it faithful; a second
// step with the exact residual x - s y1 (an FMA) then yields RN32(x/s) by
// Markstein's theorem (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990: a
// faithful quotient corrected with a correctly rounded reciprocal and an
// exact FMA residual is the correctly rounded quotient, barring underflow).
// Underflow only happens for quotients far below 2^-10, whose e4m3 code is
// zero either way.  Working on |x| keeps the sign of zero out of the
// arithmetic; the caller restores it.
template <bool POW2>
__device__ __forceinline__ float quotient_abs(float ax, float s, float r)
{
    float y = __fmul_rn(ax, r);
    if (POW2)
        return y;
    float e = __fmaf_rn(-y, s, ax);
    y = __fmaf_rn(e, r, y);
    e = __fmaf_rn(-y, s, ax);
    return __fmaf_rn(e, r, y);
}

template <bool POW2>
__device__ __forceinline__ float quotient(float x, float s, float r)
{
    return copysignf(quotient_abs<POW2>(fabsf(x), s, r), x);
}

// --------------------------------------------------------------- e4m3 ---

// Four fp32 -> four float8_e4m3fn codes (round to nearest even, saturate to
// +-448) packed little-endian: a0 lands in the lowest byte.  cvt...e4m3x2
// puts its first source in the upper byte of the 16-bit result.
__device__ __forceinline__ uint32_t pack4_e4m3(float a0, float a1, float a2, float a3)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
    return r;
}

// Quantise the 8 values a lane holds with its group's scale; returns 8 codes.
template <bool UE8M0>
__device__ __forceinline__ uint2 quant8(const float (&v)[8], float s, float r)
{
    float p[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        p[k] = quotient<UE8M0>(v[k], s, r);
    uint2 out;
    out.x = pack4_e4m3(p[0], p[1], p[2], p[3]);
    out.y = pack4_e4m3(p[4], p[5], p[6], p[7]);
    return out;
}

__device__ __forceinline__ float absmax8(const float (&v)[8])
{
    float m = fabsf(v[0]);
#pragma unroll
    for (int k = 1; k < 8; ++k)
        m = fmaxf(m, fabsf(v[k]));
    return m;
}

}  // namespace fp8q
