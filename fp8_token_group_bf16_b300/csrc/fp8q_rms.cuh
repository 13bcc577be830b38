// rms_norm_per_block_quant for sm_103a: token rows staged in shared memory by
// bulk asynchronous copies, an error-free row sum of squares, then the group
// quantisation of the normalised row.
//
// One CTA works through rows t = blockIdx.x, blockIdx.x + gridDim.x, ...
// (persistent: the grid is the number of CTAs resident at once).  Shared
// memory holds S row stages, the weight, S + 1 mbarriers and the reduction
// scratch.  Thread 0 keeps S - 1 rows in flight ahead of the row being
// processed: each row (and its residual row) arrives with one bulk copy that
// completes a stage barrier; the weight arrives once per CTA.
//
// Per row:
//   pass 1  every quad of lanes takes a 128-value group (32 values a lane)
//           from shared memory; with a residual, z = bf16(x + r) is written
//           back to the stage and to the residual tensor; each lane sums its
//           squares without rounding error (below), the quads' partial sums
//           go to shared memory;
//   warp 0  adds the partial sums (still without error), rounds once, and
//           forms inv = 1 / sqrt(ss / H + eps);
//   pass 2  every quad reads its group again with the weight, v = (z inv) w,
//           group amax, scale, codes, stores.
// Reads of a lane's 64 bytes are rotated by (lane >> 1) & 3 sixteen-byte
// pieces, so the 32 lanes of a warp hit all 32 banks evenly (four wavefronts
// per 512 bytes); codes are stored in the same rotated order, eight bytes at
// a time, to their own places.
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

// Byte offsets of the pieces of dynamic shared memory.
struct RmsSmem {
    uint32_t stage_bytes, stages, w_off, bar_off, red_off, inv_off, total;

    __host__ __device__ RmsSmem(int H, bool res, int S)
    {
        stage_bytes = uint32_t(H) * 2u * (res ? 2u : 1u);
        stages = uint32_t(S);
        w_off = stage_bytes * stages;
        bar_off = w_off + uint32_t(H) * 2u;                       // 256-byte aligned
        red_off = bar_off + 8u * (kRmsMaxStages + 1);
        inv_off = red_off + 8u * (kRmsMaxThreads / 4);
        total = inv_off + 16u;
    }
};

// Squares of one lane's 32 values (16 bf16x2 words), summed exactly:
// returns (hi, lo) with hi + lo equal to the sum up to lo's own rounding.
__device__ __forceinline__ void lane_sumsq(const uint32_t (&w)[16], float &hi, float &lo)
{
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
        m = absmax3(m, bf_lo(w[k]), bf_hi(w[k]));
    const float pm = __fmul_rn(m, m);
    uint64_t s = f2_pack(pm, pm), c = f2_pack(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint64_t z = f2_from_bf16x2(w[k]);
        const uint64_t p = f2_mul(z, z);
        const uint64_t t = f2_add(s, p);
        c = f2_add(c, f2_sub(p, f2_sub(t, s)));   // Fast2Sum error, |s| >= |p|
        s = t;
    }
    float s0, s1, c0, c1;
    f2_unpack(s, s0, s1);
    f2_unpack(c, c0, c1);
    const float inf = __int_as_float(0x7F800000);
    if (!(s0 < inf && s1 < inf)) {   // the squares overflow fp32: so does the row sum
        hi = inf;
        lo = 0.0f;
        return;
    }
    float e;
    two_sum(__fsub_rn(s0, pm), __fsub_rn(s1, pm), hi, e);   // both differences exact
    lo = __fadd_rn(__fadd_rn(c0, c1), e);
}

template <bool UE8M0, bool COL, bool RES>
__global__ void __launch_bounds__(kRmsMaxThreads) rms_quant_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ residual, const uint16_t *__restrict__ w,
    uint8_t *__restrict__ q, float *__restrict__ scales, int T, int H, int G, float eps, int S)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const RmsSmem L(H, RES, S);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + L.bar_off;          // stage barriers, then the weight's
    const uint32_t wbar = bar0 + 8u * uint32_t(S);
    float2 *red = reinterpret_cast<float2 *>(smem + L.red_off);
    float *inv_sm = reinterpret_cast<float *>(smem + L.inv_off);

    const int tid = threadIdx.x, lane = tid & 31, sub = tid & 3, quad = tid >> 2;
    const int nq = blockDim.x >> 2;
    const int rot = (lane >> 1) & 3;
    const int step = gridDim.x;
    const uint32_t row_bytes = uint32_t(H) * 2u;

    if (tid == 0) {
        for (int s = 0; s <= S; ++s)
            mbar_init(bar0 + 8u * s, 1);
        fence_barrier_init();
    }
    __syncthreads();
    wait_for_producer();
    allow_consumer_launch();

    const uint64_t pol_stream = policy_evict_first();
    int issued = 0;   // row iterations whose copies thread 0 has issued
    auto issue = [&](int j) {
        const int64_t row = int64_t(blockIdx.x) + int64_t(j) * step;
        const int s = j % S;
        const uint32_t dst = sbase + uint32_t(s) * L.stage_bytes;
        const uint32_t bar = bar0 + 8u * s;
        mbar_arrive_expect_tx(bar, L.stage_bytes);
        bulk_g2s(dst, x + row * H, row_bytes, bar, pol_stream);
        if (RES)
            bulk_g2s(dst + row_bytes, residual + row * H, row_bytes, bar, pol_stream);
    };
    if (tid == 0) {
        mbar_arrive_expect_tx(wbar, row_bytes);
        bulk_g2s(sbase + L.w_off, w, row_bytes, wbar, policy_evict_last());
        for (; issued < S && int64_t(blockIdx.x) + int64_t(issued) * step < T; ++issued)
            issue(issued);
    }
    bool ok = mbar_wait(wbar, 0);

    int j = 0;
    bool aborted = false;
    for (int row = blockIdx.x; row < T; row += step, ++j) {   // the host keeps T below 2^30
        const int s = j % S;
        ok = mbar_wait(bar0 + 8u * s, uint32_t(j / S) & 1u) && ok;
        const uint32_t stage = sbase + uint32_t(s) * L.stage_bytes;

        // ---- pass 1: residual add, exact sum of squares
        float hi = 0.0f, lo = 0.0f;
        for (int gb = 0; gb < G; gb += nq) {
            const int g = gb + quad;
            const bool act = g < G;
            const int gc = act ? g : G - 1;
            const uint32_t base = stage + uint32_t(gc) * 256u + uint32_t(sub) * 64u;
            uint32_t z[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t off = uint32_t((i + rot) & 3) * 16u;
                uint32_t p[4];
                lds128(base + off, p);
                if (RES) {
                    uint32_t r[4];
                    lds128(base + row_bytes + off, r);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        p[k] = pack_bf16x2(__fadd_rn(bf_lo(p[k]), bf_lo(r[k])),
                                           __fadd_rn(bf_hi(p[k]), bf_hi(r[k])));
                    if (act) {
                        sts128(base + off, p);
                        stg128(residual + int64_t(row) * H + gc * kGroup + sub * kValsPerLane +
                                   ((i + rot) & 3) * 8, p);
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    z[4 * i + k] = p[k];
            }
            float h, l;
            lane_sumsq(z, h, l);
            if (act)
                pair_add(hi, lo, h, l);
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1)
            pair_add(hi, lo, __shfl_xor_sync(0xFFFFFFFFu, hi, o), __shfl_xor_sync(0xFFFFFFFFu, lo, o));
        if (sub == 0)
            red[quad] = make_float2(hi, lo);

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
        if (tid < 32) {
            float2 a = lane < nq ? red[lane] : make_float2(0.0f, 0.0f);
            if (lane + 32 < nq) {
                const float2 b = red[lane + 32];
                pair_add(a.x, a.y, b.x, b.y);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                pair_add(a.x, a.y, __shfl_xor_sync(0xFFFFFFFFu, a.x, o), __shfl_xor_sync(0xFFFFFFFFu, a.y, o));
            if (lane == 0) {
                const float ss = __fadd_rn(a.x, a.y);
                inv_sm[0] = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, float(H)), eps)));
            }
        }
        __syncthreads();
        const float inv = inv_sm[0];
        const uint64_t inv2 = f2_pack(inv, inv);

        // ---- pass 2: v = (z * inv) * w, group scale, codes
        for (int gb = 0; gb < G; gb += nq) {
            const int g = gb + quad;
            const bool act = g < G;
            const int gc = act ? g : G - 1;
            const uint32_t off_g = uint32_t(gc) * 256u + uint32_t(sub) * 64u;
            uint64_t v[4][4];
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t off = off_g + uint32_t((i + rot) & 3) * 16u;
                uint32_t zp[4], wp[4];
                lds128(stage + off, zp);
                lds128(sbase + L.w_off + off, wp);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[i][k] = f2_mul(f2_mul(f2_from_bf16x2(zp[k]), inv2), f2_from_bf16x2(wp[k]));
                    float a, b;
                    f2_unpack(v[i][k], a, b);
                    m = absmax3(m, a, b);
                }
            }
            const float amax = quad_max(m);
            const float sc = group_scale<UE8M0>(amax, kScaleFloor);
            const float rc = scale_recip<UE8M0>(sc);
            uint8_t *qrow = q + int64_t(row) * H + gc * kGroup + sub * kValsPerLane;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t c0, c1;
                quant8<UE8M0>(v[i], sc, rc, c0, c1);
                if (act)
                    stg64(qrow + ((i + rot) & 3) * 8, c0, c1);
            }
            if (act && sub == 0)
                scales[COL ? int64_t(g) * T + row : int64_t(row) * G + g] = sc;
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
        // let the copies still in flight land before shared memory goes away
        mbar_wait(wbar, 0);
        for (int k = j; k < issued; ++k)
            mbar_wait(bar0 + 8u * (k % S), uint32_t(k / S) & 1u);
    }
}

}  // namespace fp8q
