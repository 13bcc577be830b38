// Per-token ("dynamic per-token") quantisation for sm_103a: one scale per
// token row instead of one per 128-group.  dynamic_per_token_scaled_fp8_quant
// is token_quant_kernel, silu_and_mul_dynamic_per_token_quant is
// token_silu_kernel; the RMSNorm variant is rms_row_kernel with the
// kPerToken scale layout.
//
// The row-wide amax is the only step the per-group kernels do not have.  A
// row of up to 64 groups (8192 values) is one CTA of quads, as in the group
// kernels, each lane holding 32 values.  A longer row is
// split over a thread-block cluster of C <= 8 CTAs (one per 64 groups or
// fewer), and the CTAs exchange their partial maxima through distributed
// shared memory: each CTA's maximum is written straight into the matching
// slot of every CTA of the cluster, one cluster barrier later every CTA reads
// all C partials from its own shared memory.  Nothing is re-read
// from HBM and no second kernel is needed.
#pragma once

#include "fp8q_kernels.cuh"

namespace fp8q {

constexpr int kTokenMaxCluster = 8;                        // portable cluster size
constexpr int kTokenMaxWarps = kCtaThreads / 32;           // 8
constexpr int kTokenMaxGroups = kTokenMaxCluster * kGroupsPerCta;   // 512 groups = 65536 values

// Cluster barrier halves.  Every thread of every CTA of the cluster executes
// each of them exactly once, in uniform control flow (like __syncthreads), so
// no barrier can wait on a thread that never arrives.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store v at the address of `local` in the shared memory of CTA `rank` of
// this cluster.
__device__ __forceinline__ void st_cluster_f32(float *local, uint32_t rank, float v)
{
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// The row maximum from each warp's maximum m: every CTA of the row's cluster
// (C of them, rank `rank`; C = 1 is a single CTA) ends with the maximum over
// the whole row.  `part` is this CTA's slot array (64 floats): with C = 1 the
// warp maxima; with C > 1, slots [0, C) receive the CTA maxima of the
// cluster's CTAs and slots [8, 16) this CTA's warp maxima.  With C > 1 the
// caller has executed cluster_arrive_relaxed() once at the start of the
// kernel; the wait here pairs with it, so that every CTA of the cluster is
// known to be running before its shared memory is written.  One warp per CTA
// sends the CTA's maximum and arrives with release semantics (its remote
// stores ordered before the barrier); the other warps arrive relaxed and
// skip the memory fence a release costs: 110.6 us instead of 128.2 us for
// silu_and_mul_dynamic_per_token_quant at T = 4096, I = 25600, where every
// warp sent its own maximum with release.
__device__ __forceinline__ float row_max_exchange(float m, float *part, int rank, int C)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 1; o <= 16; o <<= 1)
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (C == 1) {
        if (lane == 0)
            part[warp] = m;
        __syncthreads();
    } else {
        if (lane == 0)
            part[kTokenMaxCluster + warp] = m;   // this CTA's warp maxima
        __syncthreads();
        float cm = 0.0f;
        if (warp == 0) {
            cm = lane < nwarps ? part[kTokenMaxCluster + lane] : 0.0f;
#pragma unroll
            for (int o = 1; o <= 4; o <<= 1)
                cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
        }
        cluster_wait_acquire();
        if (warp == 0) {
            if (lane < C)
                st_cluster_f32(&part[rank], uint32_t(lane), cm);
            __syncwarp();
            cluster_arrive_release();
        } else {
            cluster_arrive_relaxed();
        }
        cluster_wait_acquire();
        float amax = 0.0f;
        for (int r = 0; r < C; ++r)
            amax = fmaxf(amax, part[r]);
        return amax;
    }
    float amax = 0.0f;
    for (int r = 0; r < C; ++r)
        for (int w = 0; w < nwarps; ++w)
            amax = fmaxf(amax, part[r * kTokenMaxWarps + w]);
    return amax;
}

// Launch shape of both per-token kernels: grid = T * C CTAs, clusters of C
// along x (C = 1: an ordinary launch); CTA rank r of row t owns groups
// [r * gpc, min((r + 1) * gpc, G)) with one quad per group.  cols is the
// output row length.  Inactive quads read their CTA's first group,
// contribute 0 to the maximum and store nothing.

// dynamic_per_token_scaled_fp8_quant.  Only the 16 raw bf16x2 words of a
// lane stay live across the row exchange (the maximum of |x| is taken on the
// bf16 values, which is exact); the fp32 values are formed afterwards, as in
// the per-group kernel, which keeps the register count at the per-group
// kernel's.  The PF build prefetches like token_silu_kernel below (3 x the
// SM count ahead, issued after the CTA's own loads): 16.8 us against 18.1 us
// at T = 4096, H = 7168, 56.7 against 64.8 us at T = 16384.
constexpr int kTokenQuantMinCtas = 5;   // per SM, at 256 threads: 51 registers

template <bool UE8M0, bool V8, bool PF>
__global__ void __launch_bounds__(kCtaThreads, kTokenQuantMinCtas) token_quant_kernel(
    const uint16_t *__restrict__ x, uint8_t *__restrict__ q, float *__restrict__ scales, int cols, int G, int gpc,
    int C, float eps, int pf)
{
    __shared__ float part[kTokenMaxCluster * kTokenMaxWarps];
    const int tid = threadIdx.x, sub = tid & 3, quad = tid >> 2;
    const int row = blockIdx.x / C, rank = blockIdx.x - row * C;
    const int g0 = rank * gpc, g = g0 + quad;
    const bool act = quad < gpc && g < G;
    const int64_t off = int64_t(row) * cols + int64_t(act ? g : g0) * kGroup + sub * kValsPerLane;

    if (C > 1)
        cluster_arrive_relaxed();
    wait_for_producer();
    allow_consumer_launch();

    uint32_t raw[16];
    ld64_stream<V8>(x + off, raw);
    // With this CTA's loads issued, the input of CTA blockIdx.x + pf into L2.
    if (PF && tid == 0 && int64_t(blockIdx.x) + pf < int64_t(gridDim.x)) {
        const int bp = int(blockIdx.x) + pf, rp = bp / C, gp = (bp - rp * C) * gpc;
        const uint32_t bytes = uint32_t(G - gp < gpc ? G - gp : gpc) * kGroup * 2;
        prefetch_l2_bulk(x + int64_t(rp) * cols + int64_t(gp) * kGroup, bytes);
    }
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
        m = absmax3(m, bf_lo(raw[k]), bf_hi(raw[k]));
    const float amax = row_max_exchange(act ? m : 0.0f, part, rank, C);

    const float s = group_scale<UE8M0>(amax, eps);
    const ScaleRecip rc = scale_recip<UE8M0>(s);
    uint32_t codes[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        constexpr bool neg = !UE8M0;   // v, or -v for quant8
        const uint64_t v[4] = {f2_from_bf16x2_neg<neg>(raw[4 * i]), f2_from_bf16x2_neg<neg>(raw[4 * i + 1]),
                               f2_from_bf16x2_neg<neg>(raw[4 * i + 2]), f2_from_bf16x2_neg<neg>(raw[4 * i + 3])};
        quant8<UE8M0>(v, s, rc, codes[2 * i], codes[2 * i + 1]);
    }
    if (act)
        st32<V8>(q + off, codes);
    if (rank == 0 && tid == 0)
        scales[row] = s;
}

// silu_and_mul_dynamic_per_token_quant.  The SiLU products must be kept until
// the row maximum is known and cannot be cheaply recomputed (the SiLU is
// most of the kernel's instructions), so each lane holds its 32 products in
// registers across the exchange.  Staging the inputs in shared memory with
// cp.async instead, to free those registers for more CTAs per SM, measured
// slower (174 us against 142 us at T = 4096, I = 25600).
//
// While a cluster's warps wait on its barrier their loads are done, so in
// the PF build (launched when CTAs wait for a later wave) thread 0 hands the
// input of CTA blockIdx.x + pf to the L2 once its own loads are issued
// (pf = 3 x the SM count, set by the host; about half the CTAs resident at
// once), and that CTA then finds its bytes there: 105.9 us against 123.5 us
// at T = 4096, I = 25600 (fp32 scales), 30.6 against 34.5 us at T = 1024.  Issued before
// the CTA's own loads it gained less (109.5 us); distances of 1, 2 and 4 x
// the SM count measured within 3 % of 3 x.
constexpr int kTokenSiluMinCtas = 4;   // per SM, at 256 threads: 64 registers

template <bool UE8M0, bool V8, bool PF>
__global__ void __launch_bounds__(kCtaThreads, kTokenSiluMinCtas) token_silu_kernel(const uint16_t *__restrict__ x,
                                                                  uint8_t *__restrict__ q,
                                                                  float *__restrict__ scales, int cols,
                                                                  int G, int gpc, int C, float eps, int pf)
{
    __shared__ float part[kTokenMaxCluster * kTokenMaxWarps];
    const int tid = threadIdx.x, sub = tid & 3, quad = tid >> 2;
    const int row = blockIdx.x / C, rank = blockIdx.x - row * C;
    const int g0 = rank * gpc, g = g0 + quad;
    const bool act = quad < gpc && g < G;
    const int64_t lo = int64_t(act ? g : g0) * kGroup + sub * kValsPerLane;
    const uint16_t *pa = x + int64_t(row) * 2 * cols + lo;

    if (C > 1)
        cluster_arrive_relaxed();
    wait_for_producer();
    allow_consumer_launch();

    uint32_t ra[16], rb[16];
    ld64_stream<V8>(pa, ra);
    ld64_stream<V8>(pa + cols, rb);
    // With this CTA's loads issued, the gate and up segments of CTA
    // blockIdx.x + pf into L2.
    if (PF && tid == 0 && int64_t(blockIdx.x) + pf < int64_t(gridDim.x)) {
        const int bp = int(blockIdx.x) + pf, rp = bp / C, gp = (bp - rp * C) * gpc;
        const uint32_t bytes = uint32_t(G - gp < gpc ? G - gp : gpc) * kGroup * 2;
        const uint16_t *pp = x + int64_t(rp) * 2 * cols + int64_t(gp) * kGroup;
        prefetch_l2_bulk(pp, bytes);
        prefetch_l2_bulk(pp + cols, bytes);
    }
    uint64_t v[16];
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        v[k] = silu_mul2<!UE8M0>(ra[k], rb[k]);   // v, or -v for quant8
        float v0, v1;
        f2_unpack(v[k], v0, v1);
        m = absmax3(m, v0, v1);
    }
    const float amax = row_max_exchange(act ? m : 0.0f, part, rank, C);

    const float s = group_scale<UE8M0>(amax, eps);
    const ScaleRecip rc = scale_recip<UE8M0>(s);
    uint32_t codes[8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        quant8<UE8M0>(*reinterpret_cast<const uint64_t(*)[4]>(&v[4 * i]), s, rc, codes[2 * i], codes[2 * i + 1]);
    if (act)
        st32<V8>(q + int64_t(row) * cols + lo, codes);
    if (rank == 0 && tid == 0)
        scales[row] = s;
}

}  // namespace fp8q
