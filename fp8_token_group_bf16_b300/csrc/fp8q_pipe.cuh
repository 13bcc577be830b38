// Shared-memory staging for the streaming kernels: bulk asynchronous copies
// (TMA, cp.async.bulk) from global memory into shared-memory stages, each
// stage guarded by an mbarrier that completes when its bytes have landed;
// bounded waits on those barriers; a device-wide error word; and the
// error-free sums used by the row sum of squares.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fp8q_device.cuh"

namespace fp8q {

// ----------------------------------------------------------- error word ---
//
// Set (atomicOr) by a kernel that gave up waiting on a barrier.  The host reads
// and clears it with fp8q_take_device_error().  A kernel that sets it has
// stopped early: its outputs are incomplete.
constexpr uint32_t kErrBarrierTimeout = 1u;

__device__ uint32_t g_device_error;

__device__ __forceinline__ void raise_device_error(uint32_t bits) { atomicOr(&g_device_error, bits); }

// --------------------------------------------------------- shared memory ---

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void lds128(uint32_t a, uint32_t (&w)[4])
{
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(a)
                 : "memory");
}

__device__ __forceinline__ void sts128(uint32_t a, const uint32_t (&w)[4])
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3])
                 : "memory");
}

__device__ __forceinline__ void stg64(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void stg128(void *p, const uint32_t (&w)[4])
{
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3])
                 : "memory");
}

// -------------------------------------------------------------- mbarrier ---

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation (generic proxy) visible to the copy engine
// (async proxy) before the first copy names the barrier.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(20000u)   // suspend at most ~20 us per try
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` to complete, giving up after about one
// second of wall time.  Returns false on timeout (nothing is raised here: the
// caller decides, after agreeing with the rest of the CTA).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (global_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

// ----------------------------------------------------------- bulk copies ---

// L2 policies for the copies: streamed inputs are read once (evict first);
// the RMSNorm weight is read by every CTA (evict last).
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// `bytes` (a multiple of 16) from global `src` (16-byte aligned) into shared
// `dst` (16-byte aligned); completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// ------------------------------------------------------- error-free sums ---
//
// The row sum of squares is formed without rounding error until the very end
// (Knuth's TwoSum and Dekker's Fast2Sum: for floating-point a, b the rounding
// error of RN(a + b) is itself a floating-point number, obtained exactly from
// a few further additions), so that the fp32 value it rounds to is the sum
// of the squares rounded once, whatever order the GPU adds them in.

// s + e == a + b exactly, s = RN(a + b)  (TwoSum: six additions, any a, b).
// A non-finite s yields e = 0.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    if (!(fabsf(s) < __int_as_float(0x7F800000)))
        e = 0.0f;
}

// (hi, lo) += (h2, l2): the high parts summed without error, the low parts
// (already tiny next to the high parts) summed plainly.
__device__ __forceinline__ void pair_add(float &hi, float &lo, float h2, float l2)
{
    float s, e;
    two_sum(hi, h2, s, e);
    lo = __fadd_rn(__fadd_rn(lo, l2), e);
    hi = s;
}

}  // namespace fp8q
