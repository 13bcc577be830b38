// The per-group quantisation kernels of ops A and C for sm_103a, the SiLU
// arithmetic they share with the per-token kernels, and two small kernels
// that expose single steps for checking (the e4m3 rounding, the SiLU value).
//
// They are HBM-bound streaming kernels: a handful of fp32 operations per
// byte moved, no contraction, so no tensor cores.  A quad of lanes owns a
// group (32 values per lane); every lane issues all of its loads (64 bytes,
// or 2 x 64 bytes of gate and up) before any arithmetic.
#pragma once

#include "fp8q_device.cuh"

namespace fp8q {

constexpr int kCtaThreads = 256;                               // largest CTA of the per-token kernels
constexpr int kGroupsPerCta = kCtaThreads / kLanesPerGroup;    // 64 groups
// Op A in CTAs of four warps, one group per quad (32 groups per CTA).
// Measured (UE8M0 column-major / fp32 row-major scales, H = 7168): T = 4096
// 15.45 / 15.01 us, T = 16384 54.3 / 53.4 us, T = 512 3.28 / 3.89 us;
// 256-thread CTAs with two groups per quad: 15.6 / 15.6, 54.6 / 54.1,
// 3.48 / 4.18 us; four groups per quad: 16.3 us at T = 4096.  64-thread CTAs
// match at T = 4096 but reach 59.3 us at T = 16384 (57,344 CTAs of 4 KiB: the
// CTA launch rate, not HBM, limits).
constexpr int kGroupCtaThreads = 128;
// Op A walks token-major tiles only for UE8M0 column-major scales (group_of).
template <bool UE8M0, int LAYOUT>
constexpr bool kGroupTokenMajor = UE8M0 && LAYOUT == kColMajor;
constexpr int kGroupQuantGroupsPerCta = kGroupCtaThreads / kLanesPerGroup;   // 32
// Op C in CTAs of two warps (16 groups): 64 registers a thread allow 16 such
// CTAs per SM.  Measured at T = 4096, I = 25600 (with CUDA's expf then):
// 82.8 us, against 83.4 us with 128-thread and 85.9 us with 256-thread CTAs
// (the same 32 warps per SM in all three; smaller CTAs retire and refill
// independently), and 106 us with one-warp CTAs (102,400 CTAs at about 970
// per us: the CTA launch rate limits).
constexpr int kSiluCtaThreads = 64;
constexpr int kSiluGroupsPerCta = kSiluCtaThreads / kLanesPerGroup;   // 16

// Row t and group g of flat group index gi (G groups per row).  The host
// guarantees T*G < 2^31 (2^38 bf16 values would not fit in HBM anyway), so a
// 32-bit division suffices.
__device__ __forceinline__ void split_group(int64_t gi, int64_t G, int64_t &t, int64_t &g)
{
    const uint32_t tt = uint32_t(gi) / uint32_t(G);
    t = tt;
    g = gi - int64_t(tt) * G;
}

// The group that quad `quad` of CTA `b` owns, Q quads per CTA; false (and a
// valid group to load) when the quad is past the end.  Flat order
// (TOKEN_MAJOR false): consecutive quads on consecutive groups of a row.
// Token-major tiles (TOKEN_MAJOR true): CTA b takes group g = b mod G of
// tokens [tile Q, tile Q + Q), tile = b / G, so the eight quads of a warp
// write the scales of eight consecutive tokens of one group, one 32-byte
// sector of column-major scales instead of eight; the CTAs that follow read
// the same Q rows' next groups.  Grid: ceil(T G / Q) CTAs flat,
// ceil(T / Q) G token-major.  Measured, op A at T = 4096, H = 7168: UE8M0
// column-major scales 15.62 us flat, 14.95 us token-major (used there); fp32
// column-major 15.5 flat, 15.8 token-major; op C with exponent-byte scales
// 80.9-81.6 flat, 85.9-86.1 token-major (flat kept): reading eight rows per
// warp instead of one contiguous run costs the heavier kernels more than the
// scattered scale stores.
template <bool TOKEN_MAJOR, int Q>
__device__ __forceinline__ bool group_of(uint32_t b, int quad, int64_t G, int64_t T, int64_t &t, int64_t &g)
{
    if (!TOKEN_MAJOR) {
        const int64_t n = T * G, gi = int64_t(b) * Q + quad;
        split_group(gi < n ? gi : n - 1, G, t, g);
        return gi < n;
    }
    const uint32_t tile = b / uint32_t(G);
    g = int64_t(b) - int64_t(tile) * G;
    t = int64_t(tile) * Q + quad;
    const bool ok = t < T;
    if (!ok)
        t = T - 1;
    return ok;
}

// --------------------------------------------------------------------------
// per_token_group_fp8_quant
//
// A contiguous [T, H] tensor is a flat sequence of T*G groups, so the kernel
// walks groups, not rows (group_of: the flat order, or token-major tiles for
// UE8M0 column-major scales).  One group per quad, 32 per CTA; every
// lane issues its 64-byte load before any arithmetic.  Out-of-range quads
// load a valid group and store nothing.
// --------------------------------------------------------------------------
template <bool UE8M0, int LAYOUT, bool V8>
__global__ void __launch_bounds__(kGroupCtaThreads) group_quant_kernel(const uint16_t *__restrict__ x,
                                                                  uint8_t *__restrict__ q,
                                                                  float *__restrict__ scales,
                                                                  int64_t G, int64_t T, float eps)
{
    const int sub = threadIdx.x & (kLanesPerGroup - 1);
    int64_t t, g;
    const bool ok = group_of<kGroupTokenMajor<UE8M0, LAYOUT>, kGroupQuantGroupsPerCta>(
        blockIdx.x, threadIdx.x / kLanesPerGroup, G, T, t, g);
    const int64_t off = (t * G + g) * kGroup + sub * kValsPerLane;

    wait_for_producer();
    allow_consumer_launch();
    uint32_t raw[16];
    ld64_stream<V8>(x + off, raw);
    uint64_t v[16];
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        v[k] = f2_from_bf16x2_neg<!UE8M0>(raw[k]);   // v, or -v for quant8
        m = absmax3(m, bf_lo(raw[k]), bf_hi(raw[k]));
    }
    const float amax = quad_max(m);
    const float s = group_scale<UE8M0>(amax, eps);
    const ScaleRecip r = scale_recip<UE8M0>(s);
    uint32_t codes[8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        quant8<UE8M0>(*reinterpret_cast<const uint64_t(*)[4]>(&v[4 * i]), s, r, codes[2 * i], codes[2 * i + 1]);
    if (ok) {
        st32<V8>(q + off, codes);
        if (sub == 0)
            store_scale<LAYOUT>(scales, s, t, g, T, G);
    }
}

// --------------------------------------------------------------------------
// silu_and_mul_per_block_quant
//
// One output group per quad: output group gi = (t, g) reads the gate values
// x[t, g*128 ...] and the up values x[t, I + g*128 ...] (64 bytes of each per
// lane, both loads issued first).
//
// v = RN32(RN32(a / d) * b) with d = RN32(1 + e^-a).  The quotient is
// formed from r = rcp.approx(d) with one residual correction,
// q = q0 + RN32(a - q0 d) r, q0 = RN32(a r) (Newton-Raphson on the quotient;
// the residual is exact by FMA), which is the correctly rounded a / d except
// in rare cases where it is one ulp off, and is cheaper than IEEE division.
// The exponential's argument is capped at 88 (e^88 < FLT_MAX) so that d
// stays finite: for a below -88 the exact result is a negative number below
// 1e-36 (or -0), whose code is a zero of the same sign either way.  Below
// -104 it is floored (e^-104 rounds to 0 in fp32 either way).  Pairs of
// values go through packed fp32x2 instructions.
// --------------------------------------------------------------------------
__device__ __forceinline__ float rcp_approx(float d)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

__device__ __forceinline__ float ex2_approx(float t)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// e^x for a pair of x in [-104, 88], as 2^(x log2 e).  The product x log2 e is
// carried as th + tl: th = RN32(x L) with L = RN32(log2 e), tl its exact
// rounding error (one FMA, the TwoProduct of Ogita, Rump and Oishi) plus
// x (log2 e - L); then e^x = 2^th 2^tl ~ 2^th (1 + tl ln 2), with 2^th from
// the PTX ex2.approx instruction (|tl| < 2^-17 here, so the dropped
// second-order term is below 2^-35 relative).  The error is that of
// ex2.approx plus two roundings; the tests measure it against the libm
// expf of the oracle over every bf16 argument.  It replaces a call of expf,
// whose extra instructions cost 5 % of the whole op in this issue-bound
// kernel.
__device__ __forceinline__ uint64_t exp_f2(uint64_t x)
{
    constexpr float kLog2e = 1.44269502f;       // RN32(log2 e)
    constexpr float kLog2eLo = 1.925963e-08f;   // log2 e - kLog2e
    constexpr float kLn2 = 0.693147182f;        // RN32(ln 2)
    const uint64_t nth = f2_mul(x, f2_pack(-kLog2e, -kLog2e));           // -th
    uint64_t tl = f2_fma(x, f2_pack(kLog2e, kLog2e), nth);               // x L - th, exact
    tl = f2_fma(x, f2_pack(kLog2eLo, kLog2eLo), tl);
    float n0, n1;
    f2_unpack(nth, n0, n1);
    const uint64_t p = f2_pack(ex2_approx(-n0), ex2_approx(-n1));
    return f2_fma(p, f2_mul(tl, f2_pack(kLn2, kLn2)), p);
}

// silu(a) * b for a pair of fp32 values a, b.
__device__ __forceinline__ uint64_t silu_mul_f2(uint64_t a, uint64_t b)
{
    float a0, a1;
    f2_unpack(a, a0, a1);
    // -a clamped to [-104, 88]: e^-104 is below the smallest fp32 subnormal,
    // and the bound keeps x log2 e finite for any finite a
    const uint64_t e = exp_f2(f2_pack(fminf(fmaxf(-a0, -104.0f), 88.0f), fminf(fmaxf(-a1, -104.0f), 88.0f)));
    const uint64_t d = f2_add(f2_pack(1.0f, 1.0f), e);
    const uint64_t nd = f2_sub(f2_pack(-1.0f, -1.0f), e);   // exactly -d
    float d0, d1;
    f2_unpack(d, d0, d1);
    const uint64_t r = f2_pack(rcp_approx(d0), rcp_approx(d1));
    const uint64_t q0 = f2_mul(a, r);
    const uint64_t res = f2_fma(q0, nd, a);
    const uint64_t q = f2_fma(res, r, q0);
    return f2_mul(q, b);
}

// SiLU(a) * b from bf16x2 words; with NEG, SiLU(a) * (-b), the negated
// product (exactly: RN is symmetric).
template <bool NEG = false>
__device__ __forceinline__ uint64_t silu_mul2(uint32_t aw, uint32_t bw)
{
    return silu_mul_f2(f2_from_bf16x2(aw), f2_from_bf16x2_neg<NEG>(bw));
}

template <bool UE8M0, int LAYOUT, bool V8>
__global__ void __launch_bounds__(kSiluCtaThreads, 16) silu_quant_kernel(const uint16_t *__restrict__ x,
                                                                 uint8_t *__restrict__ q,
                                                                 float *__restrict__ scales,
                                                                 int64_t G, int64_t T, int64_t I, float eps)
{
    const int sub = threadIdx.x & (kLanesPerGroup - 1);
    int64_t t, g;
    const bool ok = group_of<false, kSiluGroupsPerCta>(blockIdx.x, threadIdx.x / kLanesPerGroup, G, T, t, g);
    const int64_t gi = t * G + g;
    const uint16_t *pa = x + t * 2 * I + g * kGroup + sub * kValsPerLane;
    wait_for_producer();
    allow_consumer_launch();
    uint32_t ra[16], rb[16];
    ld64_stream<V8>(pa, ra);
    ld64_stream<V8>(pa + I, rb);

    uint64_t v[16];
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        v[k] = silu_mul2<!UE8M0>(ra[k], rb[k]);   // v, or -v for quant8
        float v0, v1;
        f2_unpack(v[k], v0, v1);
        m = absmax3(m, v0, v1);
    }
    const float amax = quad_max(m);
    const float s = group_scale<UE8M0>(amax, eps);
    const ScaleRecip r = scale_recip<UE8M0>(s);
    uint32_t codes[8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        quant8<UE8M0>(*reinterpret_cast<const uint64_t(*)[4]>(&v[4 * i]), s, r, codes[2 * i], codes[2 * i + 1]);
    if constexpr (LAYOUT == kPackedUe8m0) {
        // a CTA starts at a multiple of 16 groups, so each half warp's four
        // quads own four 4-aligned consecutive groups
        const PackedQuads pw = packed_quads_gather(s, ok, t, g, T, G);
        if (ok)
            st32<V8>(q + gi * kGroup + sub * kValsPerLane, codes);
        packed_quads_store(scales, pw, s, ok, sub, t, g, T, G);
    } else if (ok) {
        st32<V8>(q + gi * kGroup + sub * kValsPerLane, codes);
        if (sub == 0)
            store_scale<LAYOUT>(scales, s, t, g, T, G);
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

// --------------------------------------------------------------------------
// Elementwise silu(a) * b in fp32, the value op C quantises (for checking
// the arithmetic on its own).  Thread i takes elements 2i and 2i + 1 (the
// second only if it exists); a, b, out 8-byte aligned.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256) silu_mul_kernel(const float *__restrict__ a, const float *__restrict__ b,
                                                       float *__restrict__ out, int64_t n)
{
    const int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 2;
    if (i + 1 < n) {
        const float2 av = *reinterpret_cast<const float2 *>(a + i), bv = *reinterpret_cast<const float2 *>(b + i);
        float o0, o1;
        f2_unpack(silu_mul_f2(f2_pack(av.x, av.y), f2_pack(bv.x, bv.y)), o0, o1);
        *reinterpret_cast<float2 *>(out + i) = make_float2(o0, o1);
    } else if (i < n) {
        float o0, o1;
        f2_unpack(silu_mul_f2(f2_pack(a[i], 0.0f), f2_pack(b[i], 0.0f)), o0, o1);
        out[i] = o0;
    }
}

// --------------------------------------------------------------------------
// Elementwise group scale from amax, as every kernel forms it (for checking
// the division on its own).
// --------------------------------------------------------------------------
template <bool UE8M0>
__global__ void __launch_bounds__(256) group_scale_kernel(const float *__restrict__ amax, float *__restrict__ out,
                                                          int64_t n, float eps)
{
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n)
        out[i] = group_scale<UE8M0>(amax[i], eps);
}

// --------------------------------------------------------------------------
// Elementwise e4m3(RN32(v / s)) for any positive normal fp32 scale s, by the
// quotient every kernel takes for a non-power-of-two scale (for checking it
// on its own over arbitrary fp32 values and scales).
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_pairs_kernel(const float *__restrict__ v, const float *__restrict__ s,
                                                          uint8_t *__restrict__ out, int64_t n)
{
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) {
        const float si = s[i], w = -v[i];   // quant8 takes -v
        const uint64_t w2 = f2_pack(w, w);
        const uint64_t w8[4] = {w2, w2, w2, w2};
        uint32_t c0, c1;
        quant8<false>(w8, si, scale_recip<false>(si), c0, c1);
        out[i] = uint8_t(c0 & 0xFFu);
    }
}

}  // namespace fp8q
