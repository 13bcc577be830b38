// rms_norm_per_block_quant for sm_103a: token rows staged in shared memory by
// bulk asynchronous copies (TMA), an error-free row sum of squares, then the
// group quantisation of the normalised row.
//
// Two kernels share the per-row arithmetic below:
//
//  * rms_warp_kernel (many rows of up to 8192 values): a warp owns whole
//    rows; one row stage per warp, refilled segment by segment with the next
//    row while the warp quantises the current one (details at the kernel).
//  * rms_cta_kernel (few rows, decode sizes, and longer rows): a CTA of one
//    quad per group owns a row, so a row's work is spread over up to 64
//    quads; the row is staged in shared memory by bulk asynchronous copies
//    (TMA), the quads' partial sums meet in shared memory, and thread 0 keeps
//    S - 1 rows in flight.
//
// Per row:
//   pass 1  every quad of lanes takes a 128-value group (32 values a lane)
//           from its stage; with a residual, z = bf16(x + r) is written back
//           to the stage and to the residual tensor; each lane sums its
//           squares without rounding error (below) and the partial sums are
//           combined, still without error, and rounded once: ss;
//           inv = 1 / sqrt(ss / H + eps);
//   pass 2  every quad reads its group again with the weight, v = (z inv) w,
//           group amax, scale, codes, stores.
// Reads of a lane's 64 bytes are rotated by (lane >> 1) & 3 sixteen-byte
// pieces, so the 32 lanes of a warp hit all 32 banks evenly (four wavefronts
// per 512 bytes); codes are stored in the same rotated order, eight bytes at
// a time, to their own places.  The weight is converted to fp32 once per CTA
// into a table whose 16-byte units are XOR-swizzled so that the same rotated
// reads of it are conflict-free as well.
//
// Sum of squares.  A lane seeds two accumulators with pm = the largest square
// among its 32 values and adds the squares (each exact in fp32: a bf16 value
// has 8 significant bits) with Dekker's Fast2Sum, whose precondition
// |accumulator| >= |addend| the seed guarantees; the rounding errors are
// collected exactly and summed separately.  Subtracting the seed again is
// exact (pm is a multiple of the accumulator's ulp), and every later
// combination uses TwoSum.  The fp32 result is therefore the exact sum
// rounded once, like a sum carried in wider precision, except when squares
// underflow fp32 (|z| below about 1e-19).
#pragma once

#include "fp8q_device.cuh"
#include "fp8q_pipe.cuh"

namespace fp8q {

constexpr int kRmsMaxThreads = 256;
constexpr int kRmsMaxStages = 8;

// Squares of one lane's 32 values (16 bf16x2 words), summed exactly:
// returns (hi, lo) with hi + lo equal to the sum up to lo's own rounding.
// Four accumulators (two packed pairs: even and odd words) shorten the
// dependency chains.
__device__ __forceinline__ void lane_sumsq(const uint32_t (&w)[16], float &hi, float &lo)
{
    float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
        m0 = absmax3(m0, bf_lo(w[k]), bf_hi(w[k]));
        m1 = absmax3(m1, bf_lo(w[k + 1]), bf_hi(w[k + 1]));
    }
    const float m = fmaxf(m0, m1);
    const float pm = __fmul_rn(m, m);
    uint64_t s[2] = {f2_pack(pm, pm), f2_pack(pm, pm)};
    uint64_t c[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int a = k & 1;
        const uint64_t z = f2_from_bf16x2(w[k]);
        const uint64_t p = f2_mul(z, z);
        const uint64_t t = f2_add(s[a], p);
        c[a] = f2_add(c[a], f2_sub(p, f2_sub(t, s[a])));   // Fast2Sum error, |s| >= |p|
        s[a] = t;
    }
    float sv[4], cv[4];
    f2_unpack(s[0], sv[0], sv[1]);
    f2_unpack(s[1], sv[2], sv[3]);
    f2_unpack(c[0], cv[0], cv[1]);
    f2_unpack(c[1], cv[2], cv[3]);
    const float inf = __int_as_float(0x7F800000);
    if (!(sv[0] < inf && sv[1] < inf && sv[2] < inf && sv[3] < inf)) {   // the squares overflow fp32:
        hi = inf;                                                         // so does the row sum
        lo = 0.0f;
        return;
    }
    // each accumulator minus its seed is exact; combine the four without error
    float h01, e01, h23, e23;
    two_sum(__fsub_rn(sv[0], pm), __fsub_rn(sv[1], pm), h01, e01);
    two_sum(__fsub_rn(sv[2], pm), __fsub_rn(sv[3], pm), h23, e23);
    float e;
    two_sum(h01, h23, hi, e);
    lo = __fadd_rn(__fadd_rn(__fadd_rn(cv[0], cv[1]), __fadd_rn(cv[2], cv[3])), __fadd_rn(__fadd_rn(e01, e23), e));
}

__device__ __forceinline__ float rms_inv(float hi, float lo, int H, float eps)
{
    const float ss = __fadd_rn(hi, lo);
    return __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, float(H)), eps)));
}

// ------------------------------------------------------- fp32 weight table ---
//
// Value v of the weight lives in line v / 32 (128 bytes: the 32 values one
// lane of one quad handles), 16-byte unit (2k + h) ^ swz(line) with
// k = (v % 32) / 8 (the lane's rotated piece) and h = (v % 8) / 4.

__device__ __forceinline__ uint32_t w_swizzle(uint32_t line) { return (((line >> 3) & 3u) << 1) | (line & 1u); }

// All threads of the CTA; the caller synchronises before the first read.
// Each thread issues four 16-byte loads before it converts and stores any,
// so the table costs about one L2 round trip per four chunks of a thread.
__device__ __forceinline__ void fill_weight_table(const uint16_t *__restrict__ w, int H, uint32_t wsm)
{
    const int n = H / 8;   // 16-byte chunks of 8 values
    for (int c0 = threadIdx.x; c0 < n; c0 += 4 * blockDim.x) {
        uint32_t p[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * int(blockDim.x);
            const int cc = c < n ? c : n - 1;   // clamped into the weight
            FP8Q_LD4(".nc", w + 8 * cc, p[u][0], p[u][1], p[u][2], p[u][3]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * int(blockDim.x);
            if (c < n) {
                const uint32_t line = uint32_t(c) >> 2, k = uint32_t(c) & 3u, swz = w_swizzle(line);
                const uint32_t lo[4] = {p[u][0] << 16, p[u][0] & 0xFFFF0000u, p[u][1] << 16, p[u][1] & 0xFFFF0000u};
                const uint32_t hi[4] = {p[u][2] << 16, p[u][2] & 0xFFFF0000u, p[u][3] << 16, p[u][3] & 0xFFFF0000u};
                sts128(wsm + line * 128u + ((2u * k) ^ swz) * 16u, lo);
                sts128(wsm + line * 128u + ((2u * k + 1u) ^ swz) * 16u, hi);
            }
        }
    }
}

// ------------------------------------------------------- per-group work ---

// Pass 1 for one lane and one group: `base` is the lane's 64 bytes of the row
// in the stage, `res_delta` the offset from there to its residual bytes.
// With RES, z = bf16(x + r) replaces x in the stage and, when `act`, is
// written to the residual tensor at `res_lane` (the lane's 32 values).
template <bool RES>
__device__ __forceinline__ void pass1_group(uint32_t base, uint32_t res_delta, int rot, bool act,
                                            uint16_t *res_lane, float &h, float &l)
{
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = (i + rot) & 3;
        const uint32_t a = base + uint32_t(k) * 16u;
        uint32_t p[4];
        lds128(a, p);
        if (RES) {
            uint32_t r[4];
            lds128(a + res_delta, r);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                p[e] = pack_bf16x2(__fadd_rn(bf_lo(p[e]), bf_lo(r[e])), __fadd_rn(bf_hi(p[e]), bf_hi(r[e])));
            if (act) {
                sts128(a, p);
                stg128(res_lane + k * 8, p);
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
            z[4 * i + e] = p[e];
    }
    lane_sumsq(z, h, l);
}

// Pass 2 for one lane and one group: v = (z inv) w for the lane's 32 values
// (z at `base` in the stage, w in weight-table line `wline`), the group scale
// (every lane of the warp must call this: the quad shuffles name the full
// mask) and the codes, eight per rotated piece: codes[i] belongs to piece
// (i + rot) & 3.
template <bool UE8M0>
__device__ __forceinline__ float pass2_group(uint32_t base, uint32_t wline, uint32_t swz, int rot, uint64_t inv2,
                                             uint32_t (&codes)[4][2])
{
    uint64_t v[4][4];
    float mm[2] = {0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t k = uint32_t((i + rot) & 3);
        uint32_t zp[4], w0[4], w1[4];
        lds128(base + k * 16u, zp);
        lds128(wline + ((2u * k) ^ swz) * 16u, w0);
        lds128(wline + ((2u * k + 1u) ^ swz) * 16u, w1);
        const uint64_t wv[4] = {(uint64_t(w0[1]) << 32) | w0[0], (uint64_t(w0[3]) << 32) | w0[2],
                                (uint64_t(w1[1]) << 32) | w1[0], (uint64_t(w1[3]) << 32) | w1[2]};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[i][e] = f2_mul(f2_mul(f2_from_bf16x2(zp[e]), inv2), wv[e]);
            float a, b;
            f2_unpack(v[i][e], a, b);
            mm[e & 1] = absmax3(mm[e & 1], a, b);
        }
    }
    const float amax = quad_max(fmaxf(mm[0], mm[1]));
    const float sc = group_scale<UE8M0>(amax, kScaleFloor);
    const float rc = scale_recip<UE8M0>(sc);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        quant8<UE8M0>(v[i], sc, rc, codes[i][0], codes[i][1]);
    return sc;
}

// ----------------------------------------- warp-per-row, rolling stage ---
//
// For launches of many rows with up to 16 * kWarpMaxSegs groups per row: a
// warp owns whole rows (rows first, first + NW, ...), each lane its groups
// 8 j + quad.  The warp has one row stage in shared memory, cut into
// segments of 16 groups (4 KiB of bf16), each with its own mbarrier.  Pass 1
// waits for the segments in order; pass 2 reads them again and, as soon as
// the warp is done with segment j, lane 0 starts the copy of segment j of the
// warp's next row into it.  The next row therefore streams in while pass 2
// runs, with one stage per warp instead of two, which doubles the warps a
// SM can hold (shared memory, not registers, bounds them otherwise).
// Segments are 4 KiB because bulk copies of 2 KiB do not keep HBM busy on
// B300 (measured: 3.9 TB/s of reads with 2 KiB copies, 6.7-6.9 TB/s with 4
// and 8 KiB).

constexpr int kWarpMaxSegs = 4;             // rows of up to 64 groups (8192 values)
constexpr int kSegGroups = 16;
constexpr uint32_t kSegBytes = kSegGroups * 256u;

struct RmsWarpSmem {
    uint32_t stage_bytes, w_off, bar_off, total;

    __host__ __device__ RmsWarpSmem(int H, bool res, int warps)
    {
        stage_bytes = uint32_t(H) * 2u * (res ? 2u : 1u);
        w_off = stage_bytes * uint32_t(warps);
        bar_off = w_off + uint32_t(H) * 4u;
        total = bar_off + 8u * kWarpMaxSegs * uint32_t(warps);
    }
};

template <bool UE8M0, bool COL, bool RES>
__global__ void __launch_bounds__(kRmsMaxThreads, 2) rms_warp_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ residual, const uint16_t *__restrict__ w,
    uint8_t *__restrict__ q, float *__restrict__ scales, int T, int H, int G, float eps)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int nwarps = blockDim.x >> 5;
    const RmsWarpSmem L(H, RES, nwarps);
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, sub = lane & 3, quad = lane >> 2;
    const int rot = (lane >> 1) & 3;
    const uint32_t row_bytes = uint32_t(H) * 2u;
    const uint32_t stage = sbase + uint32_t(warp) * L.stage_bytes;   // this warp's
    const uint32_t bars = sbase + L.bar_off + 8u * kWarpMaxSegs * uint32_t(warp);
    const uint32_t wsm = sbase + L.w_off;
    const int nseg = (G + kSegGroups - 1) / kSegGroups;   // <= kWarpMaxSegs (host)

    if (lane == 0) {
        for (int j = 0; j < nseg; ++j)
            mbar_init(bars + 8u * j, 1);
        fence_barrier_init();
    }
    __syncwarp();
    wait_for_producer();
    allow_consumer_launch();

    // rows of this warp: first, first + rstep, ...  (the host keeps T < 2^30)
    const int first = blockIdx.x * nwarps + warp;
    const int rstep = gridDim.x * nwarps;
    auto issue_seg = [&](int64_t row, int j) {   // lane 0
        const uint32_t off = kSegBytes * uint32_t(j);
        const uint32_t n = row_bytes - off < kSegBytes ? row_bytes - off : kSegBytes;
        const uint32_t bar = bars + 8u * uint32_t(j);
        const uint64_t pol = policy_evict_first();
        mbar_arrive_expect_tx(bar, RES ? 2u * n : n);
        bulk_g2s(stage + off, reinterpret_cast<const char *>(x + row * H) + off, n, bar, pol);
        if (RES)
            bulk_g2s(stage + row_bytes + off, reinterpret_cast<const char *>(residual + row * H) + off, n, bar,
                     pol);
    };
    if (lane == 0 && first < T)
        for (int j = 0; j < nseg; ++j)
            issue_seg(first, j);
    fill_weight_table(w, H, wsm);
    __syncthreads();

    int k = 0;
    bool aborted = false;
    for (int row = first; row < T; row += rstep, ++k) {
        const uint32_t par = uint32_t(k) & 1u;
        const int64_t next = int64_t(row) + rstep;
        uint16_t *res_row = RES ? residual + int64_t(row) * H : nullptr;

        // ---- pass 1: residual add, exact sum of squares, segment by segment
        bool ok = true;
        float hi = 0.0f, lo = 0.0f;
        for (int j = 0; j < nseg; ++j) {
            ok = mbar_wait(bars + 8u * j, par) && ok;
#pragma unroll
            for (int h8 = 0; h8 < kSegGroups / 8; ++h8) {
                const int g = kSegGroups * j + 8 * h8 + quad;
                const bool act = g < G;
                const int gc = act ? g : G - 1;
                float h, l;
                pass1_group<RES>(stage + uint32_t(gc) * 256u + uint32_t(sub) * 64u, row_bytes, rot, act,
                                 res_row + gc * kGroup + sub * kValsPerLane, h, l);
                pair_add(hi, lo, act ? h : 0.0f, act ? l : 0.0f);
            }
        }
        if (__any_sync(0xFFFFFFFFu, !ok)) {
            aborted = true;
            break;
        }
#pragma unroll
        for (int o = 1; o <= 16; o <<= 1)
            pair_add(hi, lo, __shfl_xor_sync(0xFFFFFFFFu, hi, o), __shfl_xor_sync(0xFFFFFFFFu, lo, o));
        const float inv = rms_inv(hi, lo, H, eps);
        const uint64_t inv2 = f2_pack(inv, inv);

        // ---- pass 2: v = (z * inv) * w, codes; each segment refilled once read
        uint8_t *q_row = q + int64_t(row) * H;
        for (int j = 0; j < nseg; ++j) {
#pragma unroll
            for (int h8 = 0; h8 < kSegGroups / 8; ++h8) {
                const int g = kSegGroups * j + 8 * h8 + quad;
                const bool act = g < G;
                const int gc = act ? g : G - 1;
                const uint32_t line = uint32_t(gc) * 4u + uint32_t(sub);
                uint32_t codes[4][2];
                const float sc = pass2_group<UE8M0>(stage + uint32_t(gc) * 256u + uint32_t(sub) * 64u,
                                                    wsm + line * 128u, w_swizzle(line), rot, inv2, codes);
                if (act) {
                    uint8_t *ql = q_row + gc * kGroup + sub * kValsPerLane;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        stg64(ql + ((i + rot) & 3) * 8, codes[i][0], codes[i][1]);
                    if (sub == 0)
                        scales[COL ? int64_t(g) * T + row : int64_t(row) * G + g] = sc;
                }
            }
            if (RES)
                fence_proxy_async();   // z was written to this segment in pass 1
            __syncwarp();
            if (lane == 0 && next < T) {
                fence_proxy_async();
                issue_seg(next, j);
            }
        }
    }
    if (aborted && lane == 0) {
        raise_device_error(kErrBarrierTimeout);
        for (int j = 0; j < nseg; ++j)   // the current row's copies: let them land first
            mbar_wait(bars + 8u * j, uint32_t(k) & 1u);
    }
}

// -------------------------------------- CTA per row, row in registers ---
//
// One CTA per row (grid = T), one quad per group (NG groups per quad for
// rows of more than 64 groups): every lane loads its 32 * NG values and its
// 32 * NG weights straight into registers with 256-bit loads (128-bit when
// the buffers are only 16-byte aligned), so the row is read from HBM once and
// stays in registers between the sum of squares and the quantisation.  Each
// warp reduces its lanes' exact partial sums with a butterfly; one barrier
// joins the warps.  The weight is read through L1 (every CTA of a SM reads
// the same bytes).  Short-lived CTAs at ~64 registers leave room for six per
// SM, whose loads overlap the others' arithmetic.

template <int NG, bool UE8M0, bool COL, bool RES, bool V8>
__global__ void __launch_bounds__(kRmsMaxThreads, NG == 1 ? 4 : (NG == 2 ? 2 : 1)) rms_row_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ residual, const uint16_t *__restrict__ w,
    uint8_t *__restrict__ q, float *__restrict__ scales, int T, int H, int G, float eps)
{
    __shared__ float2 red[kRmsMaxThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, sub = tid & 3, quad = tid >> 2, warp = tid >> 5;
    const int nq = blockDim.x >> 2, nwarps = blockDim.x >> 5;
    const int row = blockIdx.x;
    const int64_t rbase = int64_t(row) * H;

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
            for (int e = 0; e < 16; ++e)
                z[j][e] = pack_bf16x2(__fadd_rn(bf_lo(z[j][e]), bf_lo(r[e])), __fadd_rn(bf_hi(z[j][e]), bf_hi(r[e])));
        }
        ld64_keep_l1<V8>(w + off, wr[j]);
    }
    if (RES) {
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int g = quad + nq * j;
            if (g < G)
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
        pair_add(hi, lo, __shfl_xor_sync(0xFFFFFFFFu, hi, o), __shfl_xor_sync(0xFFFFFFFFu, lo, o));
    if (lane == 0)
        red[warp] = make_float2(hi, lo);
    __syncthreads();
    float2 a = red[0];
    for (int i = 1; i < nwarps; ++i)   // every thread, in the same order
        pair_add(a.x, a.y, red[i].x, red[i].y);
    const float inv = rms_inv(a.x, a.y, H, eps);
    const uint64_t inv2 = f2_pack(inv, inv);

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
        const float rc = scale_recip<UE8M0>(sc);
        uint32_t codes[8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            quant8<UE8M0>(v[i], sc, rc, codes[2 * i], codes[2 * i + 1]);
        if (g < G) {
            st32<V8>(q + rbase + g * kGroup + sub * kValsPerLane, codes);
            if (sub == 0)
                scales[COL ? int64_t(g) * T + row : int64_t(row) * G + g] = sc;
        }
    }
}

// -------------------------------------------------- CTA-per-row kernel ---

struct RmsCtaSmem {
    uint32_t stage_bytes, w_off, bar_off, red_off, total;

    __host__ __device__ RmsCtaSmem(int H, bool res, int S)
    {
        stage_bytes = uint32_t(H) * 2u * (res ? 2u : 1u);
        w_off = stage_bytes * uint32_t(S);
        bar_off = w_off + uint32_t(H) * 4u;
        red_off = bar_off + 8u * kRmsMaxStages;
        total = red_off + 2u * 8u * (kRmsMaxThreads / 32);   // a (hi, lo) pair per warp, double-buffered
    }
};

template <bool UE8M0, bool COL, bool RES>
__global__ void __launch_bounds__(kRmsMaxThreads, 3) rms_cta_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ residual, const uint16_t *__restrict__ w,
    uint8_t *__restrict__ q, float *__restrict__ scales, int T, int H, int G, float eps, int S)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const RmsCtaSmem L(H, RES, S);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + L.bar_off;
    const uint32_t wsm = sbase + L.w_off;
    float2 *red = reinterpret_cast<float2 *>(smem + L.red_off);

    const int tid = threadIdx.x, lane = tid & 31, sub = tid & 3, quad = tid >> 2;
    const int nq = blockDim.x >> 2, nwarps = blockDim.x >> 5;
    const int rot = (lane >> 1) & 3;
    const int step = gridDim.x;
    const uint32_t row_bytes = uint32_t(H) * 2u;

    if (tid == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(bar0 + 8u * s, 1);
        fence_barrier_init();
    }
    wait_for_producer();
    allow_consumer_launch();

    const uint64_t pol_stream = policy_evict_first();
    auto issue = [&](int j) {   // thread 0: the copies of this CTA's j-th row
        const int64_t row = int64_t(blockIdx.x) + int64_t(j) * step;
        const uint32_t dst = sbase + uint32_t(j % S) * L.stage_bytes;
        const uint32_t bar = bar0 + 8u * uint32_t(j % S);
        mbar_arrive_expect_tx(bar, L.stage_bytes);
        bulk_g2s(dst, x + row * H, row_bytes, bar, pol_stream);
        if (RES)
            bulk_g2s(dst + row_bytes, residual + row * H, row_bytes, bar, pol_stream);
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < S && int64_t(blockIdx.x) + int64_t(issued) * step < T; ++issued)
            issue(issued);
    fill_weight_table(w, H, wsm);
    __syncthreads();

    int j = 0;
    bool aborted = false;
    for (int row = blockIdx.x; row < T; row += step, ++j) {   // the host keeps T below 2^30
        const int s = j % S;
        const bool ok = mbar_wait(bar0 + 8u * s, uint32_t(j / S) & 1u);
        const uint32_t stage = sbase + uint32_t(s) * L.stage_bytes;
        uint16_t *res_row = RES ? residual + int64_t(row) * H : nullptr;

        float hi = 0.0f, lo = 0.0f;
        for (int gb = 0; gb < G; gb += nq) {
            const int g = gb + quad;
            const bool act = g < G;
            const int gc = act ? g : G - 1;
            float h, l;
            pass1_group<RES>(stage + uint32_t(gc) * 256u + uint32_t(sub) * 64u, row_bytes, rot, act,
                             res_row + gc * kGroup + sub * kValsPerLane, h, l);
            if (act)
                pair_add(hi, lo, h, l);
        }
        // each warp adds its lanes' partial sums, exactly; one (hi, lo) per warp
        // goes to shared memory (two buffers, alternating by row, so that a
        // warp may write the next row's pair while a slower one still reads)
#pragma unroll
        for (int o = 1; o <= 16; o <<= 1)
            pair_add(hi, lo, __shfl_xor_sync(0xFFFFFFFFu, hi, o), __shfl_xor_sync(0xFFFFFFFFu, lo, o));
        float2 *red_row = red + (j & 1) * (kRmsMaxThreads / 32);
        if (lane == 0)
            red_row[tid >> 5] = make_float2(hi, lo);

        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        // Every thread is done with the previous row's stage: refill it.
        if (tid == 0 && S > 1 && j > 0 && int64_t(blockIdx.x) + int64_t(j - 1 + S) * step < T) {
            fence_proxy_async();
            issue(j - 1 + S);
            issued = j + S;
        }
        // every thread adds the warps' pairs in the same order
        float2 a = red_row[0];
        for (int i = 1; i < nwarps; ++i) {
            const float2 b = red_row[i];
            pair_add(a.x, a.y, b.x, b.y);
        }
        const float inv = rms_inv(a.x, a.y, H, eps);
        const uint64_t inv2 = f2_pack(inv, inv);

        uint8_t *q_row = q + int64_t(row) * H;
        for (int gb = 0; gb < G; gb += nq) {
            const int g = gb + quad;
            const bool act = g < G;
            const int gc = act ? g : G - 1;
            const uint32_t line = uint32_t(gc) * 4u + uint32_t(sub);
            uint32_t codes[4][2];
            const float sc = pass2_group<UE8M0>(stage + uint32_t(gc) * 256u + uint32_t(sub) * 64u,
                                                wsm + line * 128u, w_swizzle(line), rot, inv2, codes);
            if (act) {
                uint8_t *ql = q_row + gc * kGroup + sub * kValsPerLane;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    stg64(ql + ((i + rot) & 3) * 8, codes[i][0], codes[i][1]);
                if (sub == 0)
                    scales[COL ? int64_t(g) * T + row : int64_t(row) * G + g] = sc;
            }
        }
        if (RES)
            fence_proxy_async();   // z was written to the stage the copy engine refills next
        if (S == 1) {
            // a single stage is refilled only once this row is finished
            __syncthreads();
            if (tid == 0 && int64_t(row) + step < T) {
                fence_proxy_async();
                issue(j + 1);
                issued = j + 2;
            }
        }
    }

    if (aborted && tid == 0) {
        raise_device_error(kErrBarrierTimeout);
        for (int k = j; k < issued; ++k)   // let copies in flight land first
            mbar_wait(bar0 + 8u * (k % S), uint32_t(k / S) & 1u);
    }
}

}  // namespace fp8q
