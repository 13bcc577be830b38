// Device helpers shared by the quantisation kernels: dependent-launch
// control, bf16 unpacking, the quad reduction, the group scale, packed fp32x2
// arithmetic, the correctly rounded quotient and the packed e4m3 conversion.
//
// A group is 128 consecutive values of one token row (the Block_FP8 "1x128
// activation scaling" of "Helion：用自动调优改进 vLLM 推理", section Scope).
// It is held by a quad of 4 consecutive lanes, 32 values per lane, so a warp
// covers 8 groups.  The per-group work (two shuffles, the scale, its
// reciprocal) is then spread over 32 values per lane.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fp8q_rounding.cuh"

namespace fp8q {

constexpr int kGroup = 128;
constexpr int kLanesPerGroup = 4;   // a quad
constexpr int kValsPerLane = 32;    // 64 bytes of bf16, 32 bytes of e4m3
constexpr float kFp8Max = 448.0f;   // largest finite float8_e4m3fn
constexpr float kScaleFloor = 1e-10f;

// ------------------------------------------------------------- memory ---
//
// All loads are volatile inline PTX with a "memory" clobber, issued only on
// addresses the caller has clamped into its buffer, so no access can leave
// the buffer whatever the compiler schedules.  V8 selects 256-bit accesses
// (32-byte aligned buffers) over 128-bit ones.

#define FP8Q_LD4(QUAL, p, a, b, c, d)                                                        \
    asm volatile("ld.global" QUAL ".v4.b32 {%0,%1,%2,%3}, [%4];"                              \
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)                                         \
                 : "l"(p)                                                                     \
                 : "memory")
#define FP8Q_LD8(QUAL, p, w, o)                                                              \
    asm volatile("ld.global" QUAL ".v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"                  \
                 : "=r"(w[o + 0]), "=r"(w[o + 1]), "=r"(w[o + 2]), "=r"(w[o + 3]),             \
                   "=r"(w[o + 4]), "=r"(w[o + 5]), "=r"(w[o + 6]), "=r"(w[o + 7])              \
                 : "l"(p)                                                                     \
                 : "memory")

// 64 bytes read once (streamed input): read-only path, L2 evict-first (the
// eviction hint exists for 256-bit loads only).
template <bool V8>
__device__ __forceinline__ void ld64_stream(const void *p, uint32_t (&w)[16])
{
    const char *c = static_cast<const char *>(p);
    if (V8) {
        FP8Q_LD8(".nc.L1::no_allocate.L2::evict_first", c, w, 0);
        FP8Q_LD8(".nc.L1::no_allocate.L2::evict_first", c + 32, w, 8);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            FP8Q_LD4(".nc.L1::no_allocate", c + 16 * k, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
}

// 64 bytes that will be read again soon (from L2): read-only path, no L1
// allocation, default L2 policy.
template <bool V8>
__device__ __forceinline__ void ld64_keep(const void *p, uint32_t (&w)[16])
{
    const char *c = static_cast<const char *>(p);
    if (V8) {
        FP8Q_LD8(".nc.L1::no_allocate", c, w, 0);
        FP8Q_LD8(".nc.L1::no_allocate", c + 32, w, 8);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            FP8Q_LD4(".nc.L1::no_allocate", c + 16 * k, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
}

// 64 bytes every CTA of a SM reads (the RMSNorm weight): read-only path,
// cached in L1.
template <bool V8>
__device__ __forceinline__ void ld64_keep_l1(const void *p, uint32_t (&w)[16])
{
    const char *c = static_cast<const char *>(p);
    if (V8) {
        FP8Q_LD8(".nc.L2::evict_last", c, w, 0);
        FP8Q_LD8(".nc.L2::evict_last", c + 32, w, 8);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            FP8Q_LD4(".nc", c + 16 * k, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
}

// 64 bytes this kernel also writes (the residual): coherent path.
template <bool V8>
__device__ __forceinline__ void ld64_rw(const void *p, uint32_t (&w)[16])
{
    const char *c = static_cast<const char *>(p);
    if (V8) {
        FP8Q_LD8(".L1::no_allocate", c, w, 0);
        FP8Q_LD8(".L1::no_allocate", c + 32, w, 8);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            FP8Q_LD4(".L1::no_allocate", c + 16 * k, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
}

// 64 bytes (32 bf16 values) to global memory.
template <bool V8>
__device__ __forceinline__ void st64(void *p, const uint32_t (&w)[16])
{
    char *c = static_cast<char *>(p);
    if (V8) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
            asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(c + 32 * h),
                         "r"(w[8 * h]), "r"(w[8 * h + 1]), "r"(w[8 * h + 2]), "r"(w[8 * h + 3]),
                         "r"(w[8 * h + 4]), "r"(w[8 * h + 5]), "r"(w[8 * h + 6]), "r"(w[8 * h + 7])
                         : "memory");
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(c + 16 * k), "r"(w[4 * k]),
                         "r"(w[4 * k + 1]), "r"(w[4 * k + 2]), "r"(w[4 * k + 3])
                         : "memory");
    }
}

// 32 bytes (32 codes) to global memory.
template <bool V8>
__device__ __forceinline__ void st32(void *p, const uint32_t (&w)[8])
{
    char *c = static_cast<char *>(p);
    if (V8) {
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(c), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    } else {
#pragma unroll
        for (int k = 0; k < 2; ++k)
            asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(c + 16 * k), "r"(w[4 * k]),
                         "r"(w[4 * k + 1]), "r"(w[4 * k + 2]), "r"(w[4 * k + 3])
                         : "memory");
    }
}

// ------------------------------------------------ dependent launches ---
//
// Every kernel is launched with programmatic stream serialization allowed,
// so on a stream (or in a CUDA graph) it may start while the kernel before it
// drains.  It therefore waits for that kernel's completion and memory flush
// (griddepcontrol.wait) before its first global load or store, and lets the
// kernel after it begin launching once all of its own CTAs are running.
// Without the launch attribute both instructions are no-ops.

__device__ __forceinline__ void wait_for_producer()
{
#ifndef FP8Q_NO_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

__device__ __forceinline__ void allow_consumer_launch()
{
#ifndef FP8Q_NO_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Ask the L2 to fetch `bytes` (a multiple of 16) starting at the 16-byte
// aligned global address p, in bulk requests of at most 8 KiB.  A hint: it
// returns at once, holds no registers and changes no result.  Kernels whose
// CTAs wait on a barrier use it to fetch the input of a CTA that starts
// later, so that HBM keeps streaming while the resident CTAs wait.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    constexpr uint32_t kChunk = 8192;
    const char *c = static_cast<const char *>(p);
    for (uint32_t o = 0; o < bytes; o += kChunk) {
        const uint32_t n = bytes - o < kChunk ? bytes - o : kChunk;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + o), "r"(n) : "memory");
    }
}

// --------------------------------------------------------------- bf16 ---

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
// Word k holds values 2k (low half, lower address) and 2k+1.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2 with round to nearest even (lo at the lower address).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------- reductions ---

// Max over the 4 lanes of a quad.  Every lane of the warp calls it (the
// shuffles name the full mask); the 8 quads reduce independently.
__device__ __forceinline__ float quad_max(float m)
{
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    return m;
}

// ------------------------------------------------------ scale layouts ---
//
// Where the scale of group g of token t goes (T tokens, G groups per row):
//   kRowMajor     fp32 s[t*G + g]
//   kColMajor     fp32 s[g*T + t]
//   kPackedUe8m0  one byte per scale, its E8M0 exponent e (the scale is
//                 2^(e - 127), UE8M0 only), four groups per 32-bit word:
//                 word (g/4, t) at word index (g/4)*T_pad + t, byte g%4 of
//                 it, T_pad = T rounded up to a multiple of 4.  The bytes of
//                 groups past G and of tokens past T are written as 0 by the
//                 threads of the last group and of the last token.
//   kMxUe8m0      the same exponent bytes in the scale-factor layout of
//                 Blackwell's block-scaled (MXFP8) GEMM operands: one byte
//                 per 32 values along the row, so the group's byte fills a
//                 32-bit word (its four 32-value blocks); the [T_pad, 4G]
//                 byte matrix (T_pad = T rounded up to 128) is stored as
//                 128 x 4 tiles, tile (t / 128, g) at word ((t/128)*G + g)*128,
//                 row r = t % 128 of a tile at word (r % 32) * 4 + r / 32.
//                 The words of tokens past T are written as 0 by the thread
//                 of the last token.
//   kPerToken     one fp32 scale per token, s[t]; the kernels that use it
//                 take the maximum over the whole row and store it
//                 themselves, not through store_scale.
constexpr int kRowMajor = 0, kColMajor = 1, kPackedUe8m0 = 2, kMxUe8m0 = 3, kPerToken = 4;

template <int LAYOUT>
__device__ __forceinline__ void store_scale(float *scales, float s, int64_t t, int64_t g, int64_t T, int64_t G)
{
    if (LAYOUT == kRowMajor) {
        scales[t * G + g] = s;
    } else if (LAYOUT == kColMajor) {
        scales[g * T + t] = s;
    } else if (LAYOUT == kMxUe8m0) {
        uint32_t *w = reinterpret_cast<uint32_t *>(scales);
        const int64_t T_pad = (T + 127) & ~int64_t(127);
        auto word = [&](int64_t tt) { return ((tt >> 7) * G + g) * 128 + (tt & 31) * 4 + ((tt >> 5) & 3); };
        w[word(t)] = (__float_as_uint(s) >> 23) * 0x01010101u;
        if (t == T - 1)
            for (int64_t tp = T; tp < T_pad; ++tp)
                w[word(tp)] = 0;
    } else {
        uint8_t *b = reinterpret_cast<uint8_t *>(scales);
        const int64_t T_pad = (T + 3) & ~int64_t(3), G_pad = (G + 3) & ~int64_t(3);
        auto at = [&](int64_t gg, int64_t tt) -> uint8_t & { return b[((gg >> 2) * T_pad + tt) * 4 + (gg & 3)]; };
        // a UE8M0 scale is a normal power of two: its exponent field is the byte
        at(g, t) = uint8_t(__float_as_uint(s) >> 23);
        if (t == T - 1)
            for (int64_t tp = T; tp < T_pad; ++tp)
                at(g, tp) = 0;
        if (g == G - 1)
            for (int64_t gp = G; gp < G_pad; ++gp) {
                at(gp, t) = 0;
                if (t == T - 1)
                    for (int64_t tp = T; tp < T_pad; ++tp)
                        at(gp, tp) = 0;
            }
    }
}

// kPackedUe8m0 a word at a time.  Four consecutive groups g0 .. g0 + 3 of one
// token (g0 a multiple of 4), owned by the quads at lanes 0, 4, 8, 12 (or 16,
// 20, 24, 28) of a warp, share one word of exponent bytes: when G % 4 == 0
// and none of the four is invalid or writes padding, the lane at 0 (or 16)
// stores the gathered word; otherwise every valid group takes store_scale.
// packed_quads_gather shuffles (every lane of the warp calls it; valid, t and
// g are the calling lane's); packed_quads_store stores.  Op C gathers before
// storing its codes and stores the scales after: 81.3 us at T = 4096 that
// way, 87.6 us both with a byte per group and with the gather after the code
// store.
struct PackedQuads {
    uint32_t word;
    bool whole;
};

__device__ __forceinline__ PackedQuads packed_quads_gather(float s, bool valid, int64_t t, int64_t g, int64_t T,
                                                           int64_t G)
{
    const uint32_t byte = __float_as_uint(s) >> 23;
    PackedQuads p;
    p.word = byte | (__shfl_down_sync(0xFFFFFFFFu, byte, 4) << 8) | (__shfl_down_sync(0xFFFFFFFFu, byte, 8) << 16) |
             (__shfl_down_sync(0xFFFFFFFFu, byte, 12) << 24);
    const int bad = (!valid || t == T - 1 || g == G - 1) ? 1 : 0;
    const int anybad = bad | __shfl_down_sync(0xFFFFFFFFu, bad, 4) | __shfl_down_sync(0xFFFFFFFFu, bad, 8) |
                       __shfl_down_sync(0xFFFFFFFFu, bad, 12);
    p.whole = (G & 3) == 0 && __shfl_sync(0xFFFFFFFFu, anybad, int(threadIdx.x & 31u) & ~15) == 0;
    return p;
}

__device__ __forceinline__ void packed_quads_store(float *scales, const PackedQuads &p, float s, bool valid, int sub,
                                                   int64_t t, int64_t g, int64_t T, int64_t G)
{
    if (p.whole) {
        if ((threadIdx.x & 15u) == 0) {
            const int64_t T_pad = (T + 3) & ~int64_t(3);
            reinterpret_cast<uint32_t *>(scales)[(g >> 2) * T_pad + t] = p.word;
        }
    } else if (valid && sub == 0) {
        store_scale<kPackedUe8m0>(scales, s, t, g, T, G);
    }
}

// ------------------------------------------------------------ scale -----

// s = RN32(max(amax, eps) / 448); with UE8M0 the smallest power of two >= s.
// eps >= 1e-30 (checked on the host) keeps a = max(amax, eps) and s normal.
//
// Without UE8M0 the division is div448_rn (two instructions, correctly
// rounded): it sits on the path from a group's last value to its first code.
//
// With UE8M0 no division is needed.  Write a = m 2^e, m in [1, 2).  The
// power of two 2^j bounds RN32(a / 448) exactly when a <= 448 2^j
// = 1.75 2^(j + 8): above that, the next fp32 value after 448 2^j already
// exceeds 448 2^j (1 + 2^-24), past which a / 448 rounds above 2^j.  So
// j = e - 8, plus one when m > 1.75, i.e. when a's mantissa field exceeds
// 0x600000: three integer instructions on a's bits.  (Forming RN32(a/448)
// first and rounding it up made op C with packed exponent-byte scales 7 %
// slower, 87.7 against 81.5 us at T = 4096.)
template <bool UE8M0>
__device__ __forceinline__ float group_scale(float amax, float eps)
{
    const float a = fmaxf(amax, eps);
    if (UE8M0) {
        const uint32_t u = __float_as_uint(a);
        const uint32_t e = (u >> 23) - 8u + ((u & 0x007FFFFFu) > 0x00600000u ? 1u : 0u);
        return __uint_as_float(e << 23);
    }
    return div448_rn(a);
}

// What quant8 needs of 1/s.  r: exact for a power of two (2^k has biased
// exponent k+127, 2^-k has 127-k = 254 - that; s lies in [2^-108, 2^120] for
// finite inputs, so both are normal), otherwise the correctly rounded
// reciprocal.  For a non-power-of-two s also a split of 1/s into rd <= 1/s,
// within one ulp, and rl = RN(1/s - rd) >= 0, so that rd + rl is 1/s to
// within 2^-46 relative: with r = RN(1/s), the remainder 1 - s r is exact
// (the residual of a faithful reciprocal is representable), so its sign says
// whether r or its predecessor lies below 1/s; 1 - s rd >= 0 is exact for the
// same reason, and rl = RN((1 - s rd) r).
struct ScaleRecip {
    float r, rd, rl;
};

template <bool UE8M0>
__device__ __forceinline__ ScaleRecip scale_recip(float s)
{
    ScaleRecip q;
    if (UE8M0) {
        q.r = __uint_as_float(0x7F000000u - (__float_as_uint(s) & 0x7F800000u));
        q.rd = q.r;
        q.rl = 0.0f;
        return q;
    }
    q.r = __frcp_rn(s);
    q.rd = __fmaf_rn(-s, q.r, 1.0f) < 0.0f ? __uint_as_float(__float_as_uint(q.r) - 1u) : q.r;
    q.rl = __fmul_rn(__fmaf_rn(-s, q.rd, 1.0f), q.r);
    return q;
}

// --------------------------------------------------------- packed fp32x2 ---
//
// add/sub/mul/fma .rn.f32x2 round each half exactly like the scalar
// instruction; one packed instruction takes one issue slot for two values.
// A packed multiply whose product feeds a packed add or subtract can be
// fused into one multiply-add by the code generator (measured: the rotation
// of the fused QK-norm + RoPE kernel); the kernels use that pattern only
// where the product is exact (squares of bf16 values), and the scalar
// __fmul_rn / __fadd_rn intrinsics, which are never fused, elsewhere.

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// A bf16x2 word (value 2k in the low half) as packed fp32x2 (exact).
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w)
{
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// The same, each half negated when NEG (a sign-bit flip, exact).
template <bool NEG>
__device__ __forceinline__ uint64_t f2_from_bf16x2_neg(uint32_t w)
{
    constexpr uint32_t f = NEG ? 0x80000000u : 0u;
    return f2_pack(__uint_as_float((w << 16) ^ f), __uint_as_float((w & 0xFFFF0000u) ^ f));
}

// max(|a|, |b|, |c|) in one three-input instruction.
__device__ __forceinline__ float absmax3(float m, float a, float b)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
    return r;
}

// Running magnitude maximum of bf16x2 words, one instruction per word: each
// half of the result has the larger magnitude of the two halves in that
// position (its sign bit is the xor of the operands' sign bits, which the
// caller clears once at the end).  bf16 max keeps subnormals.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t m, uint32_t w)
{
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w));
    return r;
}

// The largest |value| of NW bf16x2 words, as fp32 (exact).
template <int NW>
__device__ __forceinline__ float bf16x2_words_absmax(const uint32_t (&w)[NW])
{
    uint32_t m0 = 0, m1 = 0;
#pragma unroll
    for (int k = 0; k < NW; k += 2) {
        m0 = bf16x2_absmax(m0, w[k]);
        if (k + 1 < NW)
            m1 = bf16x2_absmax(m1, w[k + 1]);
    }
    const uint32_t m = bf16x2_absmax(m0, m1) & 0x7FFF7FFFu;
    return fmaxf(bf_lo(m), bf_hi(m));
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

// Quantise 8 values (four packed pairs) with their group's scale s and
// rc = scale_recip(s) into 8 codes (c0: values 0-3, c1: values 4-7): each
// code is e4m3(RN32(v / s)), the quotient correctly rounded.  The caller
// passes w = v for a power-of-two scale (UE8M0) and w = -v otherwise (a sign
// flip it gets for free or nearly: a negated factor, or bf16 inputs converted
// with their sign bits flipped, f2_from_bf16x2_neg).
//
// Power-of-two s: r is exactly 1/s, so one multiply is the exact quotient
// rounded once (its sign, zero included, is the sign of v).
// Otherwise: y0 = RN(v rd + RN(v rl)) (two instructions, w (-rl) then
// w (-rd) + that) is v/s (1 + d) rounded once with |d| < 2^-45, so it is
// within 1/2 + 2^-21 ulp of v/s: faithful.  One step with the exact residual
// v - s y0 (an FMA) and r = RN(1/s) then yields RN32(v/s) by Markstein's
// theorem (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990: a faithful
// quotient corrected with a correctly rounded reciprocal and an exact FMA
// residual is the correctly rounded quotient, barring underflow).  Underflow
// only happens for quotients far below 2^-10, whose e4m3 code is zero either
// way.  The step is taken as e = RN(s y0 + w) = -RN(v - s y0) and
// y1 = RN(y0 + e (-r)), the same values (RN is symmetric), in an order that
// keeps the sign of a zero quotient: for v = -0 (w = +0), w (-rl) = -0
// (rl >= 0), y0 = -0, e = RN(s (-0) + 0) = +0 and y1 = RN(+0 (-r) + (-0)) =
// -0; for v = +0 every step gives +0; a quotient that underflows keeps the
// sign of v.
template <bool UE8M0>
__device__ __forceinline__ void quant8(const uint64_t (&w)[4], float s, const ScaleRecip &rc, uint32_t &c0,
                                       uint32_t &c1)
{
    float q[8];
    if (UE8M0) {
        const uint64_t r2 = f2_pack(rc.r, rc.r);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            f2_unpack(f2_mul(w[k], r2), q[2 * k], q[2 * k + 1]);
    } else {
        const uint64_t nr2 = f2_pack(-rc.r, -rc.r), nrd2 = f2_pack(-rc.rd, -rc.rd);
        const uint64_t nrl2 = f2_pack(-rc.rl, -rc.rl), s2 = f2_pack(s, s);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint64_t y = f2_fma(w[k], nrd2, f2_mul(w[k], nrl2));
            const uint64_t e = f2_fma(s2, y, w[k]);
            y = f2_fma(e, nr2, y);
            f2_unpack(y, q[2 * k], q[2 * k + 1]);
        }
    }
    c0 = pack4_e4m3(q[0], q[1], q[2], q[3]);
    c1 = pack4_e4m3(q[4], q[5], q[6], q[7]);
}

}  // namespace fp8q
