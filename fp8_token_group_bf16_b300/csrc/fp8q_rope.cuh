// fused_qk_norm_rope for sm_103a: per-head RMSNorm of the query and key heads
// followed by the rotary position embedding, in place on the packed qkv
// projection ("Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA", section
// "Welche Kernel wurden in vLLM integriert").
//
// A head of 128 values is owned by a quad, as a quantisation group is: 32
// values per lane, the exact sum of squares of fp8q_rms.cuh per lane and
// TwoSum across the quad, so 1/rms is bit-identical to a sequential
// evaluation with the sum carried in double.  The lanes take the values so
// that every rotation pair stays inside one lane:
//   neox pairing (j, j + 64):      lane s holds dims 16s..16s+15 and
//                                  64+16s..64+16s+15 (two 32-byte pieces);
//   interleaved pairing (2j, 2j+1): lane s holds dims 32s..32s+31.
// Either way lane s uses cos/sin entries j = 16s..16s+15 of the position's
// table row.  Every step is one correctly rounded fp32 operation, in the
// order y = (z * inv) * w, a' = a c - b s, b' = b c + a s, then bf16
// round-to-nearest-even, so the result is bit-exact.
#pragma once

#include "fp8q_device.cuh"
#include "fp8q_exact.cuh"
#include "fp8q_rms.cuh"

namespace fp8q {

constexpr int kHeadDim = 128;
// Two warps (16 heads) per CTA: at 72 registers a thread (the launch bounds
// ask for 14 such CTAs per SM; the weights are loaded only after the head's
// sum of squares, so they do not add to the registers live while it is
// formed), 14 CTAs fit a SM.  Measured at T = 4096 with 64 + 8 heads, neox:
// 26.8 us, against 28.0 us at 80 registers (12 CTAs per SM, weights loaded
// with the head) and 29.8 us at 86; 72 registers with the weights loaded
// with the head spill 56 bytes (28.6 us).  CTA size at 80 registers: 28.0 us
// with 64-thread, 28.9 us with 128-thread, 30.1 us with 256-thread CTAs.
constexpr int kRopeCtaThreads = 64;
constexpr int kRopeMinCtas = 14;

// 32 bytes (16 bf16) that this kernel also writes: coherent path.
template <bool V8>
__device__ __forceinline__ void ld32_rw(const void *p, uint32_t *w)
{
    const char *c = static_cast<const char *>(p);
    if (V8) {
        FP8Q_LD8(".L1::no_allocate", c, w, 0);
    } else {
        FP8Q_LD4(".L1::no_allocate", c, w[0], w[1], w[2], w[3]);
        FP8Q_LD4(".L1::no_allocate", c + 16, w[4], w[5], w[6], w[7]);
    }
}

// 32 bytes of a small table every CTA reads (weights, cos/sin rows): L1.
template <bool V8>
__device__ __forceinline__ void ld32_table(const void *p, uint32_t *w)
{
    const char *c = static_cast<const char *>(p);
    if (V8) {
        FP8Q_LD8(".nc.L2::evict_last", c, w, 0);
    } else {
        FP8Q_LD4(".nc", c, w[0], w[1], w[2], w[3]);
        FP8Q_LD4(".nc", c + 16, w[4], w[5], w[6], w[7]);
    }
}

template <bool V8>
__device__ __forceinline__ void st32_words(void *p, const uint32_t *w)
{
    char *c = static_cast<char *>(p);
    if (V8) {
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(c), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    } else {
#pragma unroll
        for (int k = 0; k < 2; ++k)
            asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(c + 16 * k), "r"(w[4 * k]),
                         "r"(w[4 * k + 1]), "r"(w[4 * k + 2]), "r"(w[4 * k + 3])
                         : "memory");
    }
}

// Two fp32 values -> bf16x2 (low half = lo), round to nearest even.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// `piece` bf16 values (16 or 8) that this kernel also writes: coherent path.
template <int NWP, bool V8>
__device__ __forceinline__ void ld_piece_rw(const uint16_t *p, uint32_t *w)
{
    if (NWP == 8)
        ld32_rw<V8>(p, w);
    else
        FP8Q_LD4(".L1::no_allocate", p, w[0], w[1], w[2], w[3]);
}

template <int NWP, bool V8>
__device__ __forceinline__ void ld_piece_table(const uint16_t *p, uint32_t *w)
{
    if (NWP == 8)
        ld32_table<V8>(p, w);
    else
        FP8Q_LD4(".nc", p, w[0], w[1], w[2], w[3]);
}

template <int NWP, bool V8>
__device__ __forceinline__ void st_piece(uint16_t *p, const uint32_t *w)
{
    if (NWP == 8)
        st32_words<V8>(p, w);
    else
        asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
}

// Grid: LPH lanes (4 or 8) per (token, head) unit over the T * (Hq + Hkv)
// query and key heads, flat (unit u: token u / nh, head u % nh,
// nh = Hq + Hkv); kRopeCtaThreads / LPH units per CTA.  A lane holds
// 128 / LPH values as two pieces of 64 / LPH: neox, dims piece*s.. and
// 64 + piece*s..; interleaved, dims 2*piece*s.. and the next piece.  Either
// way it uses cos/sin entries j = piece*s .. piece*s + piece - 1.
// Positions outside [0, P) are clamped into the table (the result for such
// a token is unspecified, the access stays in bounds).
template <int LPH, bool NEOX, bool V8>
__global__ void __launch_bounds__(kRopeCtaThreads, kRopeMinCtas) qk_norm_rope_kernel(uint16_t *__restrict__ qkv,
                                                           const uint16_t *__restrict__ q_w,
                                                           const uint16_t *__restrict__ k_w,
                                                           const uint16_t *__restrict__ cos_sin,
                                                           const int64_t *__restrict__ positions, int64_t n_units,
                                                           int nh, int Hq, int64_t row, int64_t P, float eps)
{
    constexpr int VPL = kHeadDim / LPH;   // values per lane
    constexpr int NW = VPL / 2;            // bf16x2 words per lane
    constexpr int NWP = NW / 2;            // words per piece
    constexpr int PIECE = VPL / 2;         // values per piece
    const int sub = threadIdx.x & (LPH - 1);
    const int64_t u = int64_t(blockIdx.x) * (kRopeCtaThreads / LPH) + (threadIdx.x / LPH);
    const int64_t ul = u < n_units ? u : n_units - 1;
    const uint32_t t = uint32_t(ul) / uint32_t(nh), h = uint32_t(ul) - t * uint32_t(nh);
    uint16_t *xh = qkv + int64_t(t) * row + int64_t(h) * kHeadDim;
    const uint16_t *w = h < uint32_t(Hq) ? q_w : k_w;
    const int o0 = NEOX ? PIECE * sub : VPL * sub;
    const int o1 = NEOX ? kHeadDim / 2 + PIECE * sub : VPL * sub + PIECE;

    wait_for_producer();
    allow_consumer_launch();

    uint32_t z[NW], wr[NW], cs[NW];
    ld_piece_rw<NWP, V8>(xh + o0, z);
    ld_piece_rw<NWP, V8>(xh + o1, z + NWP);
    int64_t pos = positions[t];
    pos = pos < 0 ? 0 : (pos >= P ? P - 1 : pos);
    const uint16_t *crow = cos_sin + pos * kHeadDim;
    ld_piece_table<NWP, V8>(crow + PIECE * sub, cs);                   // cos_j
    ld_piece_table<NWP, V8>(crow + kHeadDim / 2 + PIECE * sub, cs + NWP);   // sin_j

    // ---- 1/rms of the head: exact lane sums, TwoSum across the head's lanes
    float hi, lo;
    lane_sumsq(z, hi, lo);
    // the weights (an L1 hit for all but the first heads of a SM), now that
    // the sum's registers are free
    ld_piece_table<NWP, V8>(w + o0, wr);
    ld_piece_table<NWP, V8>(w + o1, wr + NWP);
#pragma unroll
    for (int o = 1; o < LPH; o <<= 1)
        pair_add(hi, lo, __shfl_xor_sync(0xFFFFFFFFu, hi, o), __shfl_xor_sync(0xFFFFFFFFu, lo, o));
    const float inv = rms_inv(hi, lo, kHeadDim, eps);
    const uint64_t inv2 = f2_pack(inv, inv);
    // -0, formed at run time (eps is finite, so eps * 0 is +0): the addend of
    // the rotation's products below
    const float nzf = -__fmul_rn(eps, 0.0f);
    const uint64_t nz2 = f2_pack(nzf, nzf);

    // ---- y = (z * inv) * w, then the rotation of each (a, b) pair
    uint32_t out[NW];
#pragma unroll
    for (int k = 0; k < NWP; ++k) {
        // table word k holds cos (or sin) of j = PIECE sub + 2k and 2k + 1
        const uint64_t c = f2_from_bf16x2(cs[k]), s = f2_from_bf16x2(cs[NWP + k]);
        uint64_t a, b;
        if (NEOX) {
            // z word k: dims PIECE sub + 2k, +1 (first half); word NWP + k: the partners
            a = f2_mul(f2_mul(f2_from_bf16x2(z[k]), inv2), f2_from_bf16x2(wr[k]));
            b = f2_mul(f2_mul(f2_from_bf16x2(z[NWP + k]), inv2), f2_from_bf16x2(wr[NWP + k]));
        } else {
            // z word m holds dims VPL sub + 2m, +1: the pair j = PIECE sub + m; words
            // 2k, 2k+1 are the pairs j = PIECE sub + 2k and j + 1, (a0, b0), (a1, b1)
            const int k0 = 2 * k;
            const uint64_t y0 = f2_mul(f2_mul(f2_from_bf16x2(z[k0]), inv2), f2_from_bf16x2(wr[k0]));
            const uint64_t y1 = f2_mul(f2_mul(f2_from_bf16x2(z[k0 + 1]), inv2), f2_from_bf16x2(wr[k0 + 1]));
            float a0, b0, a1, b1;
            f2_unpack(y0, a0, b0);
            f2_unpack(y1, a1, b1);
            a = f2_pack(a0, a1);
            b = f2_pack(b0, b1);
        }
        float a0, a1, b0, b1;
        if (NEOX) {
            // The rotation in packed instructions, each product an FMA with a
            // -0 addend that the code generator cannot see: RN(x y + (-0)) =
            // RN(x y), signed zeros included, and an FMA's result is never
            // fused into the add or subtract that follows.  (A packed multiply
            // was: one rounding instead of two.)
            const uint64_t ac = f2_fma(a, c, nz2), bs = f2_fma(b, s, nz2);
            const uint64_t bc = f2_fma(b, c, nz2), as = f2_fma(a, s, nz2);
            f2_unpack(f2_sub(ac, bs), a0, a1);
            f2_unpack(f2_add(bc, as), b0, b1);
        } else {
            // Interleaved pairs (repacked above; the packed form spills
            // here): scalar IEEE intrinsics, which are never fused.
            float ya0, ya1, yb0, yb1, c0, c1, s0, s1;
            f2_unpack(a, ya0, ya1);
            f2_unpack(b, yb0, yb1);
            f2_unpack(c, c0, c1);
            f2_unpack(s, s0, s1);
            a0 = __fsub_rn(__fmul_rn(ya0, c0), __fmul_rn(yb0, s0));
            a1 = __fsub_rn(__fmul_rn(ya1, c1), __fmul_rn(yb1, s1));
            b0 = __fadd_rn(__fmul_rn(yb0, c0), __fmul_rn(ya0, s0));
            b1 = __fadd_rn(__fmul_rn(yb1, c1), __fmul_rn(ya1, s1));
        }
        if (NEOX) {
            out[k] = bf16x2_rn(a0, a1);
            out[NWP + k] = bf16x2_rn(b0, b1);
        } else {
            out[2 * k] = bf16x2_rn(a0, b0);
            out[2 * k + 1] = bf16x2_rn(a1, b1);
        }
    }
    if (u < n_units) {
        st_piece<NWP, V8>(xh + o0, out);
        st_piece<NWP, V8>(xh + o1, out + NWP);
    }
}

}  // namespace fp8q
