// C ABI of libfp8q: argument checks, variant dispatch and launches.
// The contract of every entry point is stated in include/fp8q.h.
#include "fp8q.h"
#include "fp8q_kernels.cuh"
#include "fp8q_rms.cuh"
#include "fp8q_rms_split.cuh"
#include "fp8q_rope.cuh"
#include "fp8q_token.cuh"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <cuda_runtime.h>

namespace {

using namespace fp8q;

static_assert(FP8Q_TOKEN_MAX_COLS == kTokenMaxGroups * kGroup, "per-token row limit");

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(const void *x, const void *q, const float *scales, int64_t T, int64_t H,
                 int32_t group_size, int32_t ue8m0, int32_t scale_layout)
{
    if (T < 0 || H <= 0 || group_size <= 0 || H % group_size != 0)
        return FP8Q_ERR_INVALID_ARG;
    if (scale_layout != FP8Q_SCALES_ROW_MAJOR && scale_layout != FP8Q_SCALES_COL_MAJOR &&
        scale_layout != FP8Q_SCALES_UE8M0_PACKED && scale_layout != FP8Q_SCALES_UE8M0_MX)
        return FP8Q_ERR_INVALID_ARG;
    if ((scale_layout == FP8Q_SCALES_UE8M0_PACKED || scale_layout == FP8Q_SCALES_UE8M0_MX) && !ue8m0)
        return FP8Q_ERR_INVALID_ARG;   // exponent bytes hold powers of two only
    if (group_size != kGroup)
        return FP8Q_ERR_UNSUPPORTED;
    if (T == 0)
        return FP8Q_OK;
    if (!x || !q || !scales)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scales, 4))
        return FP8Q_ERR_MISALIGNED;
    return FP8Q_OK;
}

// T*G groups must fit the kernels' 32-bit group split (2^31 groups of 128
// bf16 values would be 512 GiB of input, more than the device holds).
int check_groups(int64_t T, int64_t G)
{
    const int64_t n = T * G;
    if (n / T != G || n >= (int64_t(1) << 31))
        return FP8Q_ERR_UNSUPPORTED;
    return FP8Q_OK;
}

bool valid_scale_eps(float eps) { return std::isfinite(eps) && eps >= 1e-30f; }

int launch_status(cudaError_t launched)
{
    const cudaError_t last = cudaGetLastError();
    return (launched == cudaSuccess && last == cudaSuccess) ? FP8Q_OK : FP8Q_ERR_CUDA;
}

// SM count of the current device, cached per device.  It only sets prefetch
// distances (never a grid or an index); a failed query reads as 0 (no
// prefetch) and leaves its error for the launch status to report.
int sm_count()
{
    static std::atomic<int> cache[32];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    const bool keep = dev >= 0 && dev < 32;
    int n = keep ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 0)
            return 0;
        if (keep)
            cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// CTAs of `threads` threads at up to `regs` registers a thread that one SM
// holds at once (its 2048 threads, 65536 registers and 32 CTAs).
int resident_per_sm(int threads, int regs)
{
    return std::min({32, 2048 / threads, 65536 / (regs * threads)});
}

// CTAs of `threads` threads of `kernel` that one SM of the current device
// holds at once (the occupancy query, cached per kernel, device and block
// size); 0 if the query fails.
template <typename... KArgs>
int resident_ctas(void (*kernel)(KArgs...), int threads)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, int>, int> known;
    const auto key = std::make_tuple(reinterpret_cast<const void *>(kernel), dev, threads);
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(key);
    if (it != known.end())
        return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess) {
        cudaGetLastError();   // no answer: the caller launches unpadded
        return 0;
    }
    known[key] = n;
    return n;
}

// Launch with programmatic stream serialization allowed: the kernel may be
// scheduled while its predecessor on the stream drains, and waits for it
// (griddepcontrol.wait) before touching global memory.  cluster > 1 groups
// the CTAs into thread-block clusters of that many along x; smem is the
// dynamic shared memory per CTA.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, unsigned cluster, size_t smem,
                      cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
#ifndef FP8Q_NO_PDL
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
#endif
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st, Args... args)
{
    return launch_ex(kernel, grid, block, 1u, 0, st, args...);
}

// Grid of a group kernel with Q groups per CTA (see group_of).
template <bool TOKEN_MAJOR, int Q>
dim3 group_grid(int64_t T, int64_t G)
{
    return TOKEN_MAJOR ? dim3{unsigned((T + Q - 1) / Q * G)} : dim3{unsigned((T * G + Q - 1) / Q)};
}

template <bool U, int C, bool V>
cudaError_t launch_group(const uint16_t *x, uint8_t *q, float *s, int64_t G, int64_t T, float eps, cudaStream_t st)
{
    return launch(group_quant_kernel<U, C, V>, group_grid<kGroupTokenMajor<U, C>, kGroupQuantGroupsPerCta>(T, G),
                  dim3{unsigned(kGroupCtaThreads)}, st, x, q, s, G, T, eps);
}

template <bool U, int C, bool V>
cudaError_t launch_silu(const uint16_t *x, uint8_t *q, float *s, int64_t G, int64_t T, int64_t I, float eps,
                        cudaStream_t st)
{
    return launch(silu_quant_kernel<U, C, V>, group_grid<false, kSiluGroupsPerCta>(T, G),
                  dim3{unsigned(kSiluCtaThreads)}, st, x, q, s, G, T, I, eps);
}

// rms_norm_per_block_quant, one CTA per row with the row in registers: one
// quad per group up to 64 groups, 2 or 4 groups per quad beyond.
template <int NG, bool U, int C, bool R, bool V>
cudaError_t launch_rms_row(const uint16_t *x, uint16_t *res, const uint16_t *w, uint8_t *q, float *s, int T,
                           int H, int G, float eps, cudaStream_t st)
{
    // Rows of 1, 2 or 4 groups: 8, 4 or 2 to a warp, kRmsWarpRowsPerCta warps
    // per CTA (at T = 65536, against a warp per row: H = 128 6.97 / 34.4 us,
    // H = 256 11.8 / 34.5, H = 512 20.9 / 34.6); rows of at most kRmsWarpRowGroups
    // groups: a warp each, kRmsWarpRowsPerCta rows per CTA; rows of more
    // than 64 groups, one group per quad: a wide CTA each (up to 1024
    // threads); the rest: a CTA each.
    constexpr int kWarp = NG == 1 ? kRmsWarpRow : kRmsCtaRow;
    constexpr int kWide = NG == 1 ? kRmsWideRow : kRmsCtaRow;
    constexpr int kSub = NG == 1 ? kRmsSubWarpRow : kRmsCtaRow;
    if (NG == 1 && (G == 1 || G == 2 || G == 4)) {
        const int rows_per_cta = kRmsWarpRowsPerCta * (8 / G);
        return launch(rms_row_kernel<NG, U, C, R, V, false, kSub>, dim3{unsigned((T + rows_per_cta - 1) / rows_per_cta)},
                      dim3{unsigned(32 * kRmsWarpRowsPerCta)}, st, x, res, w, q, s, T, H, G, eps, 0);
    }
    const bool wpr = NG == 1 && G <= kRmsWarpRowGroups;
    const bool wide = NG == 1 && G > 64;
    const int rpc = wpr ? kRmsWarpRowsPerCta : 1;
    const int quads = (G + NG - 1) / NG;
    const int threads = wpr ? 32 * rpc : ((quads * 4 + 31) / 32) * 32;
    const dim3 grid{unsigned((T + rpc - 1) / rpc)}, block{unsigned(threads)};
    // The prefetching build, at a distance of 1.5 x the SM count in CTAs,
    // when rows wait for a later wave (more rows than resident at once),
    // without the residual.
    if constexpr (!R) {
        const int sms = sm_count();
        if (int64_t(T) >
            int64_t(sms) * rpc * resident_per_sm(threads, 65536 / (kRmsMaxThreads * kRmsMinCtas<NG>))) {
            if (wpr)
                return launch(rms_row_kernel<NG, U, C, R, V, true, kWarp>, grid, block, st, x, res, w, q, s, T, H,
                              G, eps, sms * 3 / 2 * rpc);
            if (wide)
                return launch(rms_row_kernel<NG, U, C, R, V, true, kWide>, grid, block, st, x, res, w, q, s, T, H,
                              G, eps, sms * 3 / 2);
            return launch(rms_row_kernel<NG, U, C, R, V, true>, grid, block, st, x, res, w, q, s, T, H, G, eps,
                          sms * 3 / 2);
        }
    }
    if (wpr)
        return launch(rms_row_kernel<NG, U, C, R, V, false, kWarp>, grid, block, st, x, res, w, q, s, T, H, G,
                      eps, 0);
    if (wide)
        return launch(rms_row_kernel<NG, U, C, R, V, false, kWide>, grid, block, st, x, res, w, q, s, T, H, G,
                      eps, 0);
    // A single wave: spread evenly over the SMs.  The CTA scheduler does not
    // deal a one-wave grid out evenly: some SMs take as many CTAs as fit while
    // others idle.  With one group per quad the CTA is padded with warps that
    // own no group (they leave at once, but their registers stay allocated)
    // to the smallest block of which a SM holds ceil(T / SMs) = cap, for
    // per-group scales, cap >= 3 and at most twice the threads that own
    // groups.  Measured alone (us, padded against not): H = 5120, T = 512
    // (6 CTAs of 160 threads fit a SM; padded to 256, 4 do) 3.94 / 4.19;
    // H = 4096, T = 768 4.02 / 4.30; H = 8192, T = 300 3.71 / 4.24, with the
    // residual 5.10 / 5.76; as op B of a chain of dependent launches (ops A,
    // B, C at T = 512) 3.76 / 4.28.  Not padded: cap 2 (H = 8192, T = 256
    // 3.62 / 3.52; to 512 threads at H = 5120 2.84 / 2.75) and the per-token
    // scale, whose second row barrier made it slower (H = 4096, T = 512:
    // 4.63 / 3.73).
    // Reserving unused shared memory per CTA to the same end measured faster
    // alone (3.61 us) but slower in the chain (5.61 us): a SM must drain
    // before its shared-memory configuration changes, so the launch no
    // longer overlapped its predecessor's drain.
    auto k = rms_row_kernel<NG, U, C, R, V, false>;
    unsigned block_x = unsigned(threads);
    const int sms = sm_count(), fit = sms > 0 ? resident_ctas(k, threads) : 0;
    if (fit > 0 && int64_t(T) <= int64_t(sms) * fit) {
        const int cap = (T + sms - 1) / sms;
        if (C != kPerToken && cap >= 3 && cap < fit) {
            for (int t = threads + 32; t <= std::min(kRmsBlockMax<NG>, 2 * threads); t += 32) {
                const int r = resident_ctas(k, t);
                if (r <= cap) {
                    if (r == cap)
                        block_x = unsigned(t);
                    break;
                }
            }
        }
    }
    return launch(k, grid, dim3{block_x}, st, x, res, w, q, s, T, H, G, eps, 0);
}

// rms_norm_per_block_quant for at most kRmsSplitMaxRows rows of more than 64
// groups: each row over a cluster of up to 8 CTAs (rms_split_kernel) of
// gpc = max(16, ceil(G / 8)) groups.  Measured at T = 1 / 8 / 32 against the
// CTA per row: H = 32768 2.08 / 2.25 / 3.01 us against 3.67 / 3.73 / 4.00;
// H = 16384 2.01 / 2.16 / 2.63 against 2.26 / 2.27 / 2.72; H = 12288 1.98 /
// 2.11 / 2.18 against 2.12 / 2.15 / 2.23; equal at T = 64.  For rows of up to
// 64 groups the split lost at every T from 1 to 512 (H = 5120, T = 1: 1.78
// against 1.58 us): its two cluster barriers cost more than the shorter
// per-SM chains save.
constexpr int kRmsSplitMaxRows = 64;

template <bool U, int C, bool R, bool V>
cudaError_t launch_rms_split(const uint16_t *x, uint16_t *res, const uint16_t *w, uint8_t *q, float *s, int T,
                             int H, int G, float eps, cudaStream_t st)
{
    int gpc = std::max(16, (G + 7) / 8);
    const int cl = (G + gpc - 1) / gpc;   // 2..8 for 64 < G <= 256
    gpc = (G + cl - 1) / cl;              // balanced: no CTA is left without groups
    const int threads = ((gpc * 4 + 31) / 32) * 32;
    return launch_ex(rms_split_kernel<U, C, R, V>, dim3{unsigned(T * cl)}, dim3{unsigned(threads)}, unsigned(cl), 0,
                     st, x, res, w, q, s, T, H, G, gpc, cl, eps);
}

template <bool U, int C, bool R>
cudaError_t launch_rms(const uint16_t *x, uint16_t *res, const uint16_t *w, uint8_t *q, float *s,
                       int T, int H, int G, float eps, cudaStream_t st)
{
    const bool v8 = aligned(x, 32) && aligned(q, 32) && aligned(w, 32) && (!res || aligned(res, 32));
    if constexpr (C != kPerToken) {
        if (G > 64 && T <= kRmsSplitMaxRows)
            return v8 ? launch_rms_split<U, C, R, true>(x, res, w, q, s, T, H, G, eps, st)
                      : launch_rms_split<U, C, R, false>(x, res, w, q, s, T, H, G, eps, st);
    }
#define FP8Q_ROW(NG)                                                                             \
    (v8 ? launch_rms_row<NG, U, C, R, true>(x, res, w, q, s, T, H, G, eps, st)                  \
        : launch_rms_row<NG, U, C, R, false>(x, res, w, q, s, T, H, G, eps, st))
    // One group per quad (a wide CTA of up to 1024 threads above 64 groups)
    // for every row with per-group scales; measured against 2 and 4 groups per quad (256-thread
    // CTAs holding 64 and 128 values a thread), UE8M0 row-major, us: H = 24576,
    // T = 8192 169.0 / 196.7; H = 8320, T = 8192 49.7 / 51.9; H = 32768,
    // T = 8192 215.1 / 226.0; H = 16384, T = 8192 91.6 / 90.0.  The
    // per-token scale keeps 2 and 4 groups per quad (31.2 / 30.3 us at
    // H = 16384, T = 2048 with one).
    if (G <= 64)
        return FP8Q_ROW(1);
    if constexpr (C != kPerToken) {
        return FP8Q_ROW(1);
    } else {
        if (G <= 128)
            return FP8Q_ROW(2);
        return FP8Q_ROW(4);
    }
#undef FP8Q_ROW
}

// fused_qk_norm_rope: LPH lanes per (token, head) unit, kRopeCtaThreads / LPH
// units per CTA.  Four lanes a head (32 values each), or eight (16 values,
// 60 registers, 17 CTAs per SM) when that grid fits in one wave: measured
// with 64 + 8 heads (neox), eight against four lanes: T = 16 1.28 / 1.54 us,
// T = 128 2.72 / 2.95, T = 256 3.34 / 4.03; past one wave four lanes win
// (T = 384 4.75 / 4.35, T = 4096 38.8 / 26.8).  Both are bit-identical.
template <int LPH, bool N, bool V>
cudaError_t launch_rope_lanes(uint16_t *x, const uint16_t *qw, const uint16_t *kw, const uint16_t *cs,
                              const int64_t *positions, int64_t n, int nh, int hq, int64_t row, int64_t P, float eps,
                              cudaStream_t st)
{
    constexpr int upc = kRopeCtaThreads / LPH;
    return launch(qk_norm_rope_kernel<LPH, N, V>, dim3{unsigned((n + upc - 1) / upc)},
                  dim3{unsigned(kRopeCtaThreads)}, st, x, qw, kw, cs, positions, n, nh, hq, row, P, eps);
}

template <bool N, bool V>
cudaError_t launch_rope(uint16_t *x, const uint16_t *qw, const uint16_t *kw, const uint16_t *cs,
                        const int64_t *positions, int64_t n, int nh, int hq, int64_t row, int64_t P, float eps,
                        cudaStream_t st)
{
    constexpr int upc8 = kRopeCtaThreads / 8;
    const int sms = sm_count();
    const int fit = sms > 0 ? resident_ctas(qk_norm_rope_kernel<8, N, V>, kRopeCtaThreads) : 0;
    if (fit > 0 && (n + upc8 - 1) / upc8 <= int64_t(sms) * fit)
        return launch_rope_lanes<8, N, V>(x, qw, kw, cs, positions, n, nh, hq, row, P, eps, st);
    return launch_rope_lanes<4, N, V>(x, qw, kw, cs, positions, n, nh, hq, row, P, eps, st);
}

// Per-token ops A and C: C CTAs per row (a cluster when C > 1), gpc =
// ceil(G / C) groups per CTA, one quad per group.  C is the smallest count
// from ceil(G / 64) to 8 whose CTAs leave the fewest idle lanes (200 groups:
// 5 CTAs of 40 quads rather than 4 of 50 quads in 56-quad blocks).
int token_ctas_per_row(int G)
{
    int best = (G + kGroupsPerCta - 1) / kGroupsPerCta, best_idle = 1 << 30;
    for (int C = best; C <= kTokenMaxCluster; ++C) {
        const int gpc = (G + C - 1) / C;
        if ((C - 1) * gpc >= G)
            continue;   // the last CTA would own no group
        const int idle = C * ((gpc * kLanesPerGroup + 31) / 32) * 32 - G * kLanesPerGroup;
        if (idle < best_idle) {
            best = C;
            best_idle = idle;
        }
    }
    return best;
}

template <bool SILU>
int launch_token(const uint16_t *x, uint8_t *q, float *s, int64_t T, int64_t cols, float eps, bool ue8m0,
                 cudaStream_t st)
{
    const int G = int(cols / kGroup);
    const int C = token_ctas_per_row(G);
    const int gpc = (G + C - 1) / C;
    if (C > kTokenMaxCluster || (C - 1) * gpc >= G || T * C >= (int64_t(1) << 31))
        return FP8Q_ERR_UNSUPPORTED;
    const int threads = ((gpc * kLanesPerGroup + 31) / 32) * 32;
    const bool v8 = aligned(x, 32) && aligned(q, 32);
    const dim3 grid{unsigned(T * C)}, block{unsigned(threads)};
    const int c = int(cols);
    cudaError_t e;
    // The prefetching builds, at a distance of 3 x the SM count, when CTAs
    // wait for a later wave (more CTAs than resident at once).
    const int sms = sm_count();
    const int regs = 65536 / (kCtaThreads * (SILU ? kTokenSiluMinCtas : kTokenQuantMinCtas));
    const int pf = T * C > int64_t(sms) * resident_per_sm(threads, regs) ? 3 * sms : 0;
#define FP8Q_TOKEN_PF(K, U, V, PF) launch_ex(K<U, V, PF>, grid, block, unsigned(C), 0, st, x, q, s, c, G, gpc, C, eps, pf)
#define FP8Q_TOKEN_K(K, U, V) (pf > 0 ? FP8Q_TOKEN_PF(K, U, V, true) : FP8Q_TOKEN_PF(K, U, V, false))
#define FP8Q_TOKEN(U, V) (SILU ? FP8Q_TOKEN_K(token_silu_kernel, U, V) : FP8Q_TOKEN_K(token_quant_kernel, U, V))
    if (ue8m0)
        e = v8 ? FP8Q_TOKEN(true, true) : FP8Q_TOKEN(true, false);
    else
        e = v8 ? FP8Q_TOKEN(false, true) : FP8Q_TOKEN(false, false);
#undef FP8Q_TOKEN
#undef FP8Q_TOKEN_K
#undef FP8Q_TOKEN_PF
    return launch_status(e);
}

// Checks shared by the per-token entry points (ops A and C): the row is a
// whole number of 128-value chunks, at most 512 of them.
int check_token(const void *x, const void *q, const float *scales, int64_t T, int64_t cols, float eps)
{
    if (T < 0 || cols <= 0 || !valid_scale_eps(eps))
        return FP8Q_ERR_INVALID_ARG;
    if (cols % kGroup != 0 || cols > int64_t(kTokenMaxGroups) * kGroup)
        return FP8Q_ERR_UNSUPPORTED;
    if (T == 0)
        return FP8Q_OK;
    if (!x || !q || !scales)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scales, 4))
        return FP8Q_ERR_MISALIGNED;
    return FP8Q_OK;
}

// Checks shared by the two RMSNorm entry points (after the scale checks).
int check_rms(const void *residual, const void *weight, int64_t T, int64_t H, float eps)
{
    if (!std::isfinite(eps) || eps < 0.0f)
        return FP8Q_ERR_INVALID_ARG;
    if (H > FP8Q_RMS_MAX_H)
        return FP8Q_ERR_UNSUPPORTED;
    if (T == 0)
        return FP8Q_OK;
    if (!weight)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(weight, 16) || (residual && !aligned(residual, 16)))
        return FP8Q_ERR_MISALIGNED;
    if (T >= (int64_t(1) << 30))
        return FP8Q_ERR_UNSUPPORTED;
    return FP8Q_OK;
}

}  // namespace

extern "C" {

int fp8q_per_token_group_quant(const void *x, void *q, float *scales, int64_t T, int64_t H,
                               int32_t group_size, float eps, int32_t ue8m0, int32_t scale_layout,
                               void *stream)
{
    int rc = check_common(x, q, scales, T, H, group_size, ue8m0, scale_layout);
    if (rc != FP8Q_OK)
        return rc;
    if (!valid_scale_eps(eps))
        return FP8Q_ERR_INVALID_ARG;
    if (T == 0)
        return FP8Q_OK;
    const int64_t G = H / kGroup;
    if ((rc = check_groups(T, G)) != FP8Q_OK)
        return rc;
    auto st = static_cast<cudaStream_t>(stream);
    auto xp = static_cast<const uint16_t *>(x);
    auto qp = static_cast<uint8_t *>(q);
    const bool col = scale_layout == FP8Q_SCALES_COL_MAJOR;
    const bool packed = scale_layout == FP8Q_SCALES_UE8M0_PACKED;
    const bool v8 = aligned(x, 32) && aligned(q, 32);
    cudaError_t e;
#define FP8Q_GROUP(U, C)                                                                         \
    (v8 ? launch_group<U, C, true>(xp, qp, scales, G, T, eps, st)                               \
        : launch_group<U, C, false>(xp, qp, scales, G, T, eps, st))
    if (packed)
        e = FP8Q_GROUP(true, kPackedUe8m0);
    else if (scale_layout == FP8Q_SCALES_UE8M0_MX)
        e = FP8Q_GROUP(true, kMxUe8m0);
    else if (ue8m0)
        e = col ? FP8Q_GROUP(true, kColMajor) : FP8Q_GROUP(true, kRowMajor);
    else
        e = col ? FP8Q_GROUP(false, kColMajor) : FP8Q_GROUP(false, kRowMajor);
#undef FP8Q_GROUP
    return launch_status(e);
}

int fp8q_silu_and_mul_per_block_quant(const void *x, void *q, float *scales, int64_t T, int64_t I,
                                      int32_t group_size, float eps, int32_t ue8m0,
                                      int32_t scale_layout, void *stream)
{
    int rc = check_common(x, q, scales, T, I, group_size, ue8m0, scale_layout);
    if (rc != FP8Q_OK)
        return rc;
    if (!valid_scale_eps(eps))
        return FP8Q_ERR_INVALID_ARG;
    if (T == 0)
        return FP8Q_OK;
    const int64_t G = I / kGroup;
    if ((rc = check_groups(T, G)) != FP8Q_OK)
        return rc;
    auto st = static_cast<cudaStream_t>(stream);
    auto xp = static_cast<const uint16_t *>(x);
    auto qp = static_cast<uint8_t *>(q);
    const bool col = scale_layout == FP8Q_SCALES_COL_MAJOR;
    const bool packed = scale_layout == FP8Q_SCALES_UE8M0_PACKED;
    const bool v8 = aligned(x, 32) && aligned(q, 32);
    cudaError_t e;
#define FP8Q_SILU(U, C)                                                                          \
    (v8 ? launch_silu<U, C, true>(xp, qp, scales, G, T, I, eps, st)                             \
        : launch_silu<U, C, false>(xp, qp, scales, G, T, I, eps, st))
    if (packed)
        e = FP8Q_SILU(true, kPackedUe8m0);
    else if (scale_layout == FP8Q_SCALES_UE8M0_MX)
        e = FP8Q_SILU(true, kMxUe8m0);
    else if (ue8m0)
        e = col ? FP8Q_SILU(true, kColMajor) : FP8Q_SILU(true, kRowMajor);
    else
        e = col ? FP8Q_SILU(false, kColMajor) : FP8Q_SILU(false, kRowMajor);
#undef FP8Q_SILU
    return launch_status(e);
}

int fp8q_rms_norm_per_block_quant(const void *x, void *residual, const void *weight, void *q,
                                  float *scales, int64_t T, int64_t H, int32_t group_size,
                                  float eps, int32_t ue8m0, int32_t scale_layout, void *stream)
{
    int rc = check_common(x, q, scales, T, H, group_size, ue8m0, scale_layout);
    if (rc != FP8Q_OK)
        return rc;
    if ((rc = check_rms(residual, weight, T, H, eps)) != FP8Q_OK || T == 0)
        return rc;
    const int G = int(H / kGroup);
    auto st = static_cast<cudaStream_t>(stream);
    auto xp = static_cast<const uint16_t *>(x);
    auto rp = static_cast<uint16_t *>(residual);
    auto wp = static_cast<const uint16_t *>(weight);
    auto qp = static_cast<uint8_t *>(q);
    const bool col = scale_layout == FP8Q_SCALES_COL_MAJOR;
    const bool packed = scale_layout == FP8Q_SCALES_UE8M0_PACKED;
    const int t = int(T), h = int(H);
    cudaError_t e;
#define FP8Q_RMS(U, C)                                                                           \
    (rp ? launch_rms<U, C, true>(xp, rp, wp, qp, scales, t, h, G, eps, st)                      \
        : launch_rms<U, C, false>(xp, rp, wp, qp, scales, t, h, G, eps, st))
    if (packed)
        e = FP8Q_RMS(true, kPackedUe8m0);
    else if (scale_layout == FP8Q_SCALES_UE8M0_MX)
        e = FP8Q_RMS(true, kMxUe8m0);
    else if (ue8m0)
        e = col ? FP8Q_RMS(true, kColMajor) : FP8Q_RMS(true, kRowMajor);
    else
        e = col ? FP8Q_RMS(false, kColMajor) : FP8Q_RMS(false, kRowMajor);
#undef FP8Q_RMS
    return launch_status(e);
}

int fp8q_dynamic_per_token_scaled_fp8_quant(const void *x, void *q, float *scales, int64_t T, int64_t H,
                                            float eps, int32_t ue8m0, void *stream)
{
    const int rc = check_token(x, q, scales, T, H, eps);
    if (rc != FP8Q_OK || T == 0)
        return rc;
    return launch_token<false>(static_cast<const uint16_t *>(x), static_cast<uint8_t *>(q), scales, T, H,
                               eps, ue8m0 != 0, static_cast<cudaStream_t>(stream));
}

int fp8q_silu_and_mul_dynamic_per_token_quant(const void *x, void *q, float *scales, int64_t T, int64_t I,
                                              float eps, int32_t ue8m0, void *stream)
{
    const int rc = check_token(x, q, scales, T, I, eps);
    if (rc != FP8Q_OK || T == 0)
        return rc;
    return launch_token<true>(static_cast<const uint16_t *>(x), static_cast<uint8_t *>(q), scales, T, I,
                              eps, ue8m0 != 0, static_cast<cudaStream_t>(stream));
}

int fp8q_rms_norm_dynamic_per_token_quant(const void *x, void *residual, const void *weight, void *q,
                                          float *scales, int64_t T, int64_t H, float eps, int32_t ue8m0,
                                          void *stream)
{
    if (T < 0 || H <= 0)
        return FP8Q_ERR_INVALID_ARG;
    if (H % kGroup != 0)
        return FP8Q_ERR_UNSUPPORTED;
    int rc = check_rms(residual, weight, T, H, eps);
    if (rc != FP8Q_OK || T == 0)
        return rc;
    if (!x || !q || !scales)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scales, 4))
        return FP8Q_ERR_MISALIGNED;
    auto st = static_cast<cudaStream_t>(stream);
    auto xp = static_cast<const uint16_t *>(x);
    auto rp = static_cast<uint16_t *>(residual);
    auto wp = static_cast<const uint16_t *>(weight);
    auto qp = static_cast<uint8_t *>(q);
    const int t = int(T), h = int(H), G = int(H / kGroup);
    cudaError_t e;
#define FP8Q_RMS(U)                                                                              \
    (rp ? launch_rms<U, kPerToken, true>(xp, rp, wp, qp, scales, t, h, G, eps, st)              \
        : launch_rms<U, kPerToken, false>(xp, rp, wp, qp, scales, t, h, G, eps, st))
    e = ue8m0 ? FP8Q_RMS(true) : FP8Q_RMS(false);
#undef FP8Q_RMS
    return launch_status(e);
}

int fp8q_fused_qk_norm_rope(void *qkv, const void *q_weight, const void *k_weight, const void *cos_sin,
                            const int64_t *positions, int64_t T, int64_t num_q_heads, int64_t num_kv_heads,
                            int64_t head_dim, int64_t max_position, float eps, int32_t is_neox, void *stream)
{
    if (T < 0 || num_q_heads < 0 || num_kv_heads < 0 || head_dim <= 0 || max_position <= 0 ||
        !std::isfinite(eps) || eps < 0.0f)
        return FP8Q_ERR_INVALID_ARG;
    if (head_dim != kHeadDim)
        return FP8Q_ERR_UNSUPPORTED;
    const int64_t nh = num_q_heads + num_kv_heads;
    if (T == 0 || nh == 0)
        return FP8Q_OK;
    if (!qkv || !q_weight || !k_weight || !cos_sin || !positions)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(qkv, 16) || !aligned(q_weight, 16) || !aligned(k_weight, 16) || !aligned(cos_sin, 16) ||
        !aligned(positions, 8))
        return FP8Q_ERR_MISALIGNED;
    const int64_t n = T * nh;
    if (nh >= (int64_t(1) << 20) || n / nh != T || n >= (int64_t(1) << 31))
        return FP8Q_ERR_UNSUPPORTED;
    const int64_t row = (num_q_heads + 2 * num_kv_heads) * head_dim;
    const bool v8 = aligned(qkv, 32) && aligned(q_weight, 32) && aligned(k_weight, 32) && aligned(cos_sin, 32);
    auto x = static_cast<uint16_t *>(qkv);
    auto qw = static_cast<const uint16_t *>(q_weight);
    auto kw = static_cast<const uint16_t *>(k_weight);
    auto cs = static_cast<const uint16_t *>(cos_sin);
    auto st = static_cast<cudaStream_t>(stream);
    const int nhi = int(nh), hq = int(num_q_heads);
    cudaError_t e;
#define FP8Q_ROPE(N, V) launch_rope<N, V>(x, qw, kw, cs, positions, n, nhi, hq, row, max_position, eps, st)
    if (is_neox)
        e = v8 ? FP8Q_ROPE(true, true) : FP8Q_ROPE(true, false);
    else
        e = v8 ? FP8Q_ROPE(false, true) : FP8Q_ROPE(false, false);
#undef FP8Q_ROPE
    return launch_status(e);
}

int fp8q_f32_to_e4m3(const float *v, void *out, int64_t n, void *stream)
{
    if (n < 0)
        return FP8Q_ERR_INVALID_ARG;
    if (n == 0)
        return FP8Q_OK;
    if (!v || !out)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(v, 16) || !aligned(out, 16))
        return FP8Q_ERR_MISALIGNED;
    const int64_t blocks = ((n + 3) / 4 + 255) / 256;
    if (blocks > 0x7FFFFFFF)
        return FP8Q_ERR_UNSUPPORTED;
    f32_to_e4m3_kernel<<<dim3{unsigned(blocks)}, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        v, static_cast<uint8_t *>(out), n);
    return launch_status(cudaSuccess);
}

int fp8q_silu_mul(const float *a, const float *b, float *out, int64_t n, void *stream)
{
    if (n < 0)
        return FP8Q_ERR_INVALID_ARG;
    if (n == 0)
        return FP8Q_OK;
    if (!a || !b || !out)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(a, 8) || !aligned(b, 8) || !aligned(out, 8))
        return FP8Q_ERR_MISALIGNED;
    const int64_t blocks = ((n + 1) / 2 + 255) / 256;
    if (blocks > 0x7FFFFFFF)
        return FP8Q_ERR_UNSUPPORTED;
    silu_mul_kernel<<<dim3{unsigned(blocks)}, 256, 0, static_cast<cudaStream_t>(stream)>>>(a, b, out, n);
    return launch_status(cudaSuccess);
}

int fp8q_group_scale(const float *amax, float *scales, int64_t n, float eps, int32_t ue8m0, void *stream)
{
    if (n < 0 || !valid_scale_eps(eps))
        return FP8Q_ERR_INVALID_ARG;
    if (n == 0)
        return FP8Q_OK;
    if (!amax || !scales)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(amax, 4) || !aligned(scales, 4))
        return FP8Q_ERR_MISALIGNED;
    const int64_t blocks = (n + 255) / 256;
    if (blocks > 0x7FFFFFFF)
        return FP8Q_ERR_UNSUPPORTED;
    auto st = static_cast<cudaStream_t>(stream);
    if (ue8m0)
        group_scale_kernel<true><<<dim3{unsigned(blocks)}, 256, 0, st>>>(amax, scales, n, eps);
    else
        group_scale_kernel<false><<<dim3{unsigned(blocks)}, 256, 0, st>>>(amax, scales, n, eps);
    return launch_status(cudaSuccess);
}

int fp8q_quant_pairs(const float *v, const float *s, void *out, int64_t n, void *stream)
{
    if (n < 0)
        return FP8Q_ERR_INVALID_ARG;
    if (n == 0)
        return FP8Q_OK;
    if (!v || !s || !out)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned(v, 4) || !aligned(s, 4))
        return FP8Q_ERR_MISALIGNED;
    const int64_t blocks = (n + 255) / 256;
    if (blocks > 0x7FFFFFFF)
        return FP8Q_ERR_UNSUPPORTED;
    quant_pairs_kernel<<<dim3{unsigned(blocks)}, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        v, s, static_cast<uint8_t *>(out), n);
    return launch_status(cudaSuccess);
}

const char *fp8q_status_string(int status)
{
    switch (status) {
    case FP8Q_OK: return "FP8Q_OK";
    case FP8Q_ERR_INVALID_ARG: return "FP8Q_ERR_INVALID_ARG: invalid argument";
    case FP8Q_ERR_UNSUPPORTED: return "FP8Q_ERR_UNSUPPORTED: unsupported group size or size";
    case FP8Q_ERR_MISALIGNED: return "FP8Q_ERR_MISALIGNED: pointer not aligned as required";
    case FP8Q_ERR_CUDA: return "FP8Q_ERR_CUDA: CUDA launch failed";
    default: return "unknown fp8q status";
    }
}

int fp8q_version(void) { return 500; }


}  // extern "C"
