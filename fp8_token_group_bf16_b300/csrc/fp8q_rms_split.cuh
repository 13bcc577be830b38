// rms_norm_per_block_quant for a handful of rows (decode): one row split
// over a thread-block cluster of C CTAs.
//
// With one CTA per row, T rows keep only T SMs busy, and each of them runs
// the whole row's chain (the loads, the 32-value lane sums, the warp
// butterflies, the row barrier, 1/rms, the group scales) on its own four
// schedulers.  Here CTA rank r of a row owns groups [r gpc, (r + 1) gpc),
// one quad per group as in rms_row_kernel, so a row is spread over C SMs and
// each SM carries 1/C of it.  The CTAs' exact partial sums meet through
// distributed shared memory: warp 0 of every CTA writes its CTA's (hi, lo)
// pair straight into slot `rank` of each CTA of the cluster and arrives at
// the cluster barrier with release semantics (the other warps arrive
// relaxed); after the wait (acquire) every CTA adds the C pairs in rank
// order with TwoSum, so all CTAs of a row form the same 1/rms.  A relaxed
// arrive at kernel start, waited on just before the remote stores, makes
// sure every CTA of the cluster is running before its shared memory is
// written.  Every thread executes each cluster barrier once, in uniform
// control flow (no early return), and the hardware launches a cluster's CTAs
// together, so no barrier waits for a thread that never arrives.
#pragma once

#include "fp8q_rms.cuh"
#include "fp8q_token.cuh"

namespace fp8q {

// Store the pair v at the address of `local` in the shared memory of CTA
// `rank` of this cluster.
__device__ __forceinline__ void st_cluster_f32x2(float2 *local, uint32_t rank, float2 v)
{
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(v.x), "f"(v.y) : "memory");
}

// Grid: T * C CTAs in clusters of C (1 <= C <= 8) along x; CTA rank r of row
// t = blockIdx.x / C owns groups [r gpc, min((r + 1) gpc, G)), gpc <= 64.
// Per-group scale layouts only (the per-token variant keeps rms_row_kernel).
template <bool UE8M0, int LAYOUT, bool RES, bool V8>
__global__ void __launch_bounds__(kRmsMaxThreads) rms_split_kernel(
    const uint16_t *__restrict__ x, uint16_t *__restrict__ residual, const uint16_t *__restrict__ w,
    uint8_t *__restrict__ q, float *__restrict__ scales, int T, int H, int G, int gpc, int C, float eps)
{
    static_assert(LAYOUT != kPerToken, "per-group scale layouts only");
    __shared__ float2 part[kTokenMaxCluster + kRmsMaxThreads / 32];   // [0, C) CTA sums, then warp sums
    const int tid = threadIdx.x, lane = tid & 31, sub = tid & 3, quad = tid >> 2, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row = blockIdx.x / C, rank = blockIdx.x - row * C;
    const int g0 = rank * gpc, g = g0 + quad;
    const bool act = quad < gpc && g < G;
    const int off = (act ? g : g0) * kGroup + sub * kValsPerLane;   // inactive quads read their CTA's first group
    const int64_t rbase = int64_t(row) * H;

    cluster_arrive_relaxed();
    wait_for_producer();
    allow_consumer_launch();

    uint32_t z[16], wr[16];
    ld64_stream<V8>(x + rbase + off, z);
    if (RES) {
        uint32_t r[16];
        ld64_rw<V8>(residual + rbase + off, r);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            // x + r for both halves in one packed add (no product near it to fuse)
            float lo, hi;
            f2_unpack(f2_add(f2_from_bf16x2(z[e]), f2_from_bf16x2(r[e])), lo, hi);
            z[e] = pack_bf16x2(lo, hi);
        }
    }
    ld64_keep_l1<V8>(w + off, wr);
    if (RES && act)
        st64<V8>(residual + rbase + off, z);

    // this CTA's exact partial sum of squares
    float hi, lo;
    lane_sumsq(z, hi, lo);
    if (!act)
        hi = lo = 0.0f;
#pragma unroll
    for (int o = 1; o <= 16; o <<= 1)
        pair_add(hi, lo, __shfl_xor_sync(0xFFFFFFFFu, hi, o), __shfl_xor_sync(0xFFFFFFFFu, lo, o));
    if (nwarps > 1) {
        if (lane == 0)
            part[kTokenMaxCluster + warp] = make_float2(hi, lo);
        __syncthreads();
        if (warp == 0) {
            float2 a = part[kTokenMaxCluster];
            for (int i = 1; i < nwarps; ++i)   // in warp order
                pair_add(a.x, a.y, part[kTokenMaxCluster + i].x, part[kTokenMaxCluster + i].y);
            hi = a.x;
            lo = a.y;
        }
    }

    // the row's sum: every CTA's pair into every CTA of the cluster, then in rank order
    cluster_wait_acquire();
    if (warp == 0) {
        if (lane < C)
            st_cluster_f32x2(&part[rank], uint32_t(lane), make_float2(hi, lo));
        __syncwarp();
        cluster_arrive_release();
    } else {
        cluster_arrive_relaxed();
    }
    cluster_wait_acquire();
    float2 s = part[0];
    for (int r = 1; r < C; ++r)
        pair_add(s.x, s.y, part[r].x, part[r].y);
    const float inv = rms_inv(s.x, s.y, H, eps);
    const uint64_t inv2 = UE8M0 ? f2_pack(inv, inv) : f2_pack(-inv, -inv);   // v, or -v for quant8

    // v = (z * inv) * w, group scale, codes
    uint64_t v[4][4];
    float mm[2] = {0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = 4 * i + e;
            v[i][e] = f2_mul(f2_mul(f2_from_bf16x2(z[k]), inv2), f2_from_bf16x2(wr[k]));
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
    if (act) {
        st32<V8>(q + rbase + off, codes);
        if (sub == 0)
            store_scale<LAYOUT>(scales, sc, row, g, T, G);
    }
}

}  // namespace fp8q
