// rms_norm_per_block_quant for sm_103a: one CTA per token row with the row
// held in registers, an error-free row sum of squares, then the group
// quantisation of the normalised row.
//
// Sum of squares.  A lane seeds two accumulators (one packed pair) with
// pm = the largest square among its 32 values and adds the squares (each
// exact in fp32: a bf16 value has 8 significant bits) in the manner of
// Dekker's Fast2Sum, whose precondition |accumulator| >= |addend| the seed
// guarantees: t = RN(s + z^2) is one multiply-add, s - t is exact, and the
// rounding error z^2 + (s - t) is representable, so a second multiply-add
// yields it exactly.  The errors are summed separately.  Taking the seed
// back out is exact (pm is a multiple of the accumulator's ulp), and every
// later combination, across groups, lanes and warps, uses Knuth's TwoSum.
// The fp32 result is therefore the exact sum rounded once, like a sum
// carried in wider precision, except when squares underflow fp32 (|z| below
// about 1e-19).
#pragma once

#include "fp8q_device.cuh"
#include "fp8q_exact.cuh"

namespace fp8q {

// Threads that own groups with 2 or 4 groups per quad (the per-token
// scale's rows of more than 64 groups): at most 64 quads.
constexpr int kRmsMaxThreads = 256;
// CTAs of kRmsMaxThreads per SM that the register cap allows: NG groups per
// quad hold 32 NG values and as many weights in registers (64, 128 and 255
// registers a thread).
template <int NG>
constexpr int kRmsMinCtas = NG == 1 ? 4 : (NG == 2 ? 2 : 1);
// The largest block the host may launch: with one group per quad, a row of
// up to 256 groups, or a CTA padded with warps that own no group so that
// fewer CTAs fit a SM (the launch bounds keep the same register cap).
template <int NG>
constexpr int kRmsBlockMax = NG == 1 ? 2 * kRmsMaxThreads : kRmsMaxThreads;
// The shapes of a row's work: a CTA per row (up to 64 groups, or 2 or 4
// groups per quad); a warp per row, several rows per CTA (up to 8 groups);
// a wide CTA per row, one group per quad (65 to 256 groups: up to 1024
// threads, 32 warps, whose partial sums meet in a butterfly).
// Rows of 1, 2 or 4 groups: several to a warp (kRmsSubWarpRow), 4 G lanes each.
constexpr int kRmsCtaRow = 0, kRmsWarpRow = 1, kRmsWideRow = 2, kRmsSubWarpRow = 3;
constexpr int kRmsWideBlockMax = 1024;
// Rows of at most this many groups take a warp each, this many rows per CTA.
constexpr int kRmsWarpRowGroups = 8;
constexpr int kRmsWarpRowsPerCta = 4;

// bar.sync on barrier 1 for the first n threads of the CTA (n a multiple of
// 32); the same memory ordering among them as __syncthreads().
__device__ __forceinline__ void bar_sync_first(int n)
{
    asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory");
}

// Squares of one lane's 2*NW values (NW bf16x2 words, NW even), summed
// exactly: returns (hi, lo) with hi + lo equal to the sum up to lo's own
// rounding.  The two halves of the packed pair accumulate the even and the
// odd values.
template <int NW>
__device__ __forceinline__ void lane_sumsq(const uint32_t (&w)[NW], float &hi, float &lo)
{
    const float m = bf16x2_words_absmax(w);
    const float pm = __fmul_rn(m, m);
    uint64_t s = f2_pack(pm, pm);
    uint64_t c = f2_pack(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        const uint64_t z = f2_from_bf16x2(w[k]);
        const uint64_t t = f2_fma(z, z, s);                // RN(s + z^2), z^2 exact
        c = f2_add(c, f2_fma(z, z, f2_sub(s, t)));         // its error, exact as |s| >= z^2
        s = t;
    }
    float sv[2], cv[2];
    f2_unpack(s, sv[0], sv[1]);
    f2_unpack(c, cv[0], cv[1]);
    const float inf = __int_as_float(0x7F800000);
    if (!(sv[0] < inf && sv[1] < inf)) {
        hi = inf;
        lo = 0.0f;
        return;
    }
    float e;
    two_sum(__fsub_rn(sv[0], pm), __fsub_rn(sv[1], pm), hi, e);
    lo = __fadd_rn(__fadd_rn(cv[0], cv[1]), e);
}

// inv = RN32(1 / RN32(sqrt(RN32(RN32(ss / H) + eps)))) with ss = RN32(hi + lo).
// A sum that overflowed fp32 has hi = +inf (the low part may then be NaN).
__device__ __forceinline__ float rms_inv(float hi, float lo, int H, float eps)
{
    const float ss = hi < __int_as_float(0x7F800000) ? __fadd_rn(hi, lo) : hi;
    return __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, float(H)), eps)));
}

// ------------------------------------------------------------- kernel ---
//
// One CTA per row (grid = T), one quad per group (NG = 2 or 4 groups per
// quad for the per-token scale's rows of more than 64 groups; with per-group
// scales a row of up to 256 groups takes a CTA of up to 1024 threads, whose
// warps' partial sums meet in a butterfly above 8 warps): every lane loads its 32 * NG values and its
// 32 * NG weights straight into registers with 256-bit loads (128-bit when
// the buffers are only 16-byte aligned), so the row is read from HBM once and
// stays in registers between the sum of squares and the quantisation.  Each
// warp reduces its lanes' exact partial sums with a butterfly; one barrier
// joins the warps.  The weight is read through L1 (every CTA of a SM reads
// the same bytes).  Short-lived CTAs at ~64 registers leave room for six per
// SM, whose loads overlap the others' arithmetic.  A row of at most 8 groups
// fits one warp: it then takes a warp of a CTA of several rows and needs
// neither shared memory nor a barrier (one CTA per such short row would make
// the CTA launch rate the limit).
//
// While a CTA waits on its barrier, its loads are done and it asks nothing of
// HBM.  When the grid is longer than the CTAs resident at once, the PF
// variant therefore has thread 0 hand row + pf to the L2 once its own loads
// are issued (pf = 1.5 x the SM count, set by the host): 14.3 us against
// 15.05 us at T = 4096, H = 5120, 48.1 against 52.1 us at T = 16384; per
// token 69.9 against 71.4 us at T = 16384.  The other launches run a build
// without that code, whose mere presence cost 2-5 % in single-wave grids
// (T <= 512), and which measured slower with the residual (24.7 against
// 23.95 us at T = 4096, the residual row prefetched too).
//
// LAYOUT == kPerToken is rms_norm_dynamic_per_token_quant: one scale for the
// whole row.  The normalised values v are formed once, into the registers
// that z and w free (32 a group either way), their row maximum is joined
// across warps by a second barrier, and the codes are taken from v: 18.5 us
// against 20.0 us at T = 4096, H = 5120 for forming v a second time from z
// and w after the barrier.

template <int NG, bool UE8M0, int LAYOUT, bool RES, bool V8, bool PF, int ROWS = kRmsCtaRow>
__global__ void __launch_bounds__(ROWS == kRmsWideRow ? kRmsWideBlockMax : kRmsBlockMax<NG>,
                                  ROWS == kRmsWideRow ? 1 : kRmsMinCtas<NG> * kRmsMaxThreads / kRmsBlockMax<NG>)
    rms_row_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ residual, const uint16_t *__restrict__ w,
                   uint8_t *__restrict__ q, float *__restrict__ scales, int T, int H, int G, float eps, int pf)
{
    constexpr int kWarps = ROWS == kRmsWideRow ? kRmsWideBlockMax / 32 : kRmsMaxThreads / 32;
    __shared__ float2 red[kWarps];
    __shared__ float redm[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, sub = tid & 3, warp = tid >> 5;
    // kRmsWarpRow (rows of at most kRmsWarpRowGroups groups): a warp per
    // row, blockDim.x / 32 rows per CTA.  kRmsSubWarpRow (rows of 1, 2 or 4
    // groups): 32 / (4 G) rows per warp, each on a segment of 4 G lanes whose
    // reductions stay inside it; a lane whose row lies past T works on a copy
    // of row T - 1 (its segment still takes part in the shuffles) and stores
    // nothing.  Otherwise a CTA per row, whose threads that own groups are
    // ceil(G / NG) quads in whole warps; warps beyond them only pad the CTA
    // and leave at once.
    static_assert(ROWS == kRmsCtaRow || NG == 1, "warp and wide rows hold one group per quad");
    static_assert(!(PF && ROWS == kRmsSubWarpRow), "no prefetching build for rows several to a warp");
    constexpr bool subw = ROWS == kRmsSubWarpRow;
    constexpr bool wpr = ROWS == kRmsWarpRow || subw;
    const int lpr = subw ? 4 * G : 32;   // lanes of a row's reductions (a power of two)
    const int nthr = wpr ? 32 : (((G + NG - 1) / NG * 4 + 31) >> 5) << 5;
    const int wrow = int(blockIdx.x) * int(blockDim.x >> 5) + warp;   // the CTA-wide warp index
    const int row = subw ? wrow * (32 / lpr) + lane / lpr : (wpr ? wrow : int(blockIdx.x));
    if (subw ? wrow * (32 / lpr) >= T : ((!wpr && tid >= nthr) || row >= T))
        return;
    const bool live = row < T;
    const int quad = (wpr ? (subw ? lane & (lpr - 1) : lane) : tid) >> 2;
    const int nq = subw ? G : nthr >> 2, nwarps = nthr >> 5;
    const int64_t rbase = int64_t(live ? row : T - 1) * H;

    wait_for_producer();
    allow_consumer_launch();

    uint32_t z[NG][16], wr[NG][16];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
        const int g = quad + nq * j;
        const int off = (g < G ? g : G - 1) * kGroup + sub * kValsPerLane;   // clamped into the row
        ld64_stream<V8>(x + rbase + off, z[j]);
        if (RES) {
            uint32_t r[16];
            ld64_rw<V8>(residual + rbase + off, r);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                // x + r for both halves in one packed add (no product near it to fuse)
                float lo, hi;
                f2_unpack(f2_add(f2_from_bf16x2(z[j][e]), f2_from_bf16x2(r[e])), lo, hi);
                z[j][e] = pack_bf16x2(lo, hi);
            }
        }
        ld64_keep_l1<V8>(w + off, wr[j]);
    }
    // With this CTA's loads issued, row row + pf into L2 for the CTA that
    // will take it.
    if constexpr (PF) {
        static_assert(!RES, "no prefetch with the residual");
        if ((wpr ? lane : tid) == 0 && row + pf < T)
            prefetch_l2_bulk(x + rbase + int64_t(pf) * H, uint32_t(H) * 2);
    }
    if (RES) {
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int g = quad + nq * j;
            if (g < G && live)
                st64<V8>(residual + rbase + g * kGroup + sub * kValsPerLane, z[j]);
        }
    }

    // ---- pass 1: exact sum of squares
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int j = 0; j < NG; ++j) {
        float h, l;
        lane_sumsq(z[j], h, l);
        const bool act = quad + nq * j < G;
        pair_add(hi, lo, act ? h : 0.0f, act ? l : 0.0f);
    }
#pragma unroll
    for (int o = 1; o <= 16; o <<= 1)
        if (o < lpr)
            pair_add(hi, lo, __shfl_xor_sync(0xFFFFFFFFu, hi, o), __shfl_xor_sync(0xFFFFFFFFu, lo, o));
    // One warp: every lane holds the same pair (pair_add is symmetric, so both
    // partners of each butterfly step form the same sum).  Several: one
    // barrier, then every thread adds the warps' pairs in the same order.
    float2 a = make_float2(hi, lo);
    if (nwarps > 1) {
        if (lane == 0)
            red[warp] = a;
        bar_sync_first(nthr);
        if constexpr (ROWS == kRmsWideRow) {
            // up to 32 warps: each warp reads the pairs one a lane and forms
            // the same total with a butterfly (every lane of every warp ends
            // with the same pair, as above)
            a = lane < nwarps ? red[lane] : make_float2(0.0f, 0.0f);
#pragma unroll
            for (int o = 1; o <= 16; o <<= 1)
                pair_add(a.x, a.y, __shfl_xor_sync(0xFFFFFFFFu, a.x, o), __shfl_xor_sync(0xFFFFFFFFu, a.y, o));
        } else {
            a = red[0];
            for (int i = 1; i < nwarps; ++i)
                pair_add(a.x, a.y, red[i].x, red[i].y);
        }
    }
    const float inv = rms_inv(a.x, a.y, H, eps);
    // With an fp32 scale the normalised values are formed negated (exactly:
    // RN is symmetric), as quant8 takes them; the maxima take |v| either way.
    const uint64_t inv2 = UE8M0 ? f2_pack(inv, inv) : f2_pack(-inv, -inv);

    if constexpr (LAYOUT == kPerToken) {
        // ---- pass 2: v = (z * inv) * w, in the registers z and w free, and its row maximum
        uint64_t v[NG][16];
        float mm[2] = {0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const bool act = quad + nq * j < G;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                v[j][k] = f2_mul(f2_mul(f2_from_bf16x2(z[j][k]), inv2), f2_from_bf16x2(wr[j][k]));
                float va, vb;
                f2_unpack(v[j][k], va, vb);
                if (act)
                    mm[k & 1] = absmax3(mm[k & 1], va, vb);
            }
        }
        float m = fmaxf(mm[0], mm[1]);
#pragma unroll
        for (int o = 1; o <= 16; o <<= 1)
            if (o < lpr)
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        float amax = m;
        if (nwarps > 1) {
            if (lane == 0)
                redm[warp] = m;
            bar_sync_first(nthr);
            amax = redm[0];
            for (int i = 1; i < nwarps; ++i)
                amax = fmaxf(amax, redm[i]);
        }
        const float sc = group_scale<UE8M0>(amax, kScaleFloor);
        const ScaleRecip rc = scale_recip<UE8M0>(sc);

        // ---- pass 3: codes
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int g = quad + nq * j;
            uint32_t codes[8];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                quant8<UE8M0>(*reinterpret_cast<const uint64_t(*)[4]>(&v[j][4 * i]), sc, rc, codes[2 * i],
                              codes[2 * i + 1]);
            if (g < G && live)
                st32<V8>(q + rbase + g * kGroup + sub * kValsPerLane, codes);
        }
        if ((wpr ? lane & (lpr - 1) : tid) == 0 && live)
            scales[row] = sc;
    } else {
        // ---- pass 2: v = (z * inv) * w, group scale, codes
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int g = quad + nq * j;
            uint64_t v[4][4];
            float mm[2] = {0.0f, 0.0f};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = 4 * i + e;
                    v[i][e] = f2_mul(f2_mul(f2_from_bf16x2(z[j][k]), inv2), f2_from_bf16x2(wr[j][k]));
                    float va, vb;
                    f2_unpack(v[i][e], va, vb);
                    mm[e & 1] = absmax3(mm[e & 1], va, vb);
                }
            const float amax = quad_max(fmaxf(mm[0], mm[1]));
            const float sc = group_scale<UE8M0>(amax, kScaleFloor);
            const ScaleRecip rc = scale_recip<UE8M0>(sc);
            uint32_t codes[8];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                quant8<UE8M0>(v[i], sc, rc, codes[2 * i], codes[2 * i + 1]);
            // (packed exponent bytes a byte per group: gathering each word of
            // four from the quads, as op C does, measured slower here, 14.93
            // against 14.44 us at T = 4096, H = 5120)
            if (g < G && live) {
                st32<V8>(q + rbase + g * kGroup + sub * kValsPerLane, codes);
                if (sub == 0)
                    store_scale<LAYOUT>(scales, sc, row, g, T, G);
            }
        }
    }
}

}  // namespace fp8q
