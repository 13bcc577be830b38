/*
 * libfp8q — fused FP8 quantisation epilogues (and the fused QK-norm + rotary
 * embedding) for NVIDIA B300 (sm_103a).
 *
 * The three operations are the FP8 activation-quantisation custom ops of FP8
 * LLM inference named in "[RFC]: Using Helion for Selected vLLM CustomOps"
 * (Motivation, the list of kernels in the initial rollout):
 * per_token_group_fp8_quant, silu_and_mul_per_block_quant and
 * rms_norm_per_block_quant.  Their scale granularity is the Block_FP8
 * "1x128 activation scaling" of "Helion：用自动调优改进 vLLM 推理" (section
 * Scope): one fp32 scale per contiguous group of 128 values of a token row.
 * The power-of-two scale option is the "float32 ceiling E8M0" scale format of
 * the RFC's H100 end-to-end settings (also "UE8M0" in "Helion-Kernel in vLLM:
 * PyTorch FP8 ohne CUDA", section "Praktische Einschränkungen").
 *
 * Arithmetic of every op, per group of 128 values v_i (fp32):
 *   amax = max |v_i|;  s = RN32(max(amax, eps) / 448)
 *   ue8m0 != 0:  s <- smallest power of two >= s (exact)
 *   q_i  = e4m3fn(RN32(v_i / s)): round to nearest even, |.| > 448 -> +-448,
 *          subnormals kept, sign of zero kept.
 * The pages print no formula; this is the plain reading, and the library
 * reproduces it bit for bit for per_token_group_quant.
 *
 * Beside the three per-group ops the library holds their per-token variants
 * (one scale per token row) and fused_qk_norm_rope, from the list of kernels
 * in "Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA" (section "Welche Kernel
 * wurden in vLLM integriert"); each is specified at its declaration below.
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers (global memory of the current device).  The
 *    caller owns and allocates every buffer; the library allocates nothing.
 *    Its only state between calls is a per-device cache of the SM count,
 *    which chooses launch variants and never changes a result.
 *  - bf16 tensors are row-major and contiguous (row stride = row length);
 *    `q` is float8_e4m3fn bytes, row-major [T, H] (or [T, I]).
 *  - `x`, `q`, `residual` and `weight` must be 16-byte aligned, `scales`
 *    4-byte aligned.  `q` must not alias `x`; `residual` must not alias `x`.
 *  - Scale layout: FP8Q_SCALES_ROW_MAJOR stores s[t*G + g];
 *    FP8Q_SCALES_COL_MAJOR stores s[g*T + t], G = H / group_size;
 *    FP8Q_SCALES_UE8M0_PACKED and FP8Q_SCALES_UE8M0_MX store exponent
 *    bytes (below).  Either without ue8m0 is FP8Q_ERR_INVALID_ARG.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Calls only enqueue work and never synchronise, so they can be
 *    captured into CUDA graphs.
 *  - Return value: an fp8q_status.  Invalid arguments are rejected before
 *    anything is enqueued.  FP8Q_ERR_CUDA reports a failed launch
 *    (cudaGetLastError after the launch); a fault while the kernel runs is
 *    reported by CUDA at the caller's next synchronisation.  T == 0 returns
 *    FP8Q_OK without a launch.  Calls never abort or throw.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stdint.h>

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_INVALID_ARG = 1, /* negative T, H <= 0, H % group_size, NULL pointer, bad enum, bad eps */
    FP8Q_ERR_UNSUPPORTED = 2, /* group_size != 128, a row longer than the kernels handle, T*G >= 2^31 */
    FP8Q_ERR_MISALIGNED = 3,  /* a pointer below its required alignment */
    FP8Q_ERR_CUDA = 4         /* the CUDA launch failed */
} fp8q_status;

typedef enum {
    FP8Q_SCALES_ROW_MAJOR = 0,   /* fp32 s[t*G + g] */
    FP8Q_SCALES_COL_MAJOR = 1,   /* fp32 s[g*T + t] */
    FP8Q_SCALES_UE8M0_PACKED = 2, /* E8M0 exponent bytes, four groups per 32-bit word (below) */
    FP8Q_SCALES_UE8M0_MX = 3      /* E8M0 bytes in the MXFP8 GEMM scale-factor tiles (below) */
} fp8q_scale_layout;

/*
 * FP8Q_SCALES_UE8M0_PACKED (requires ue8m0 != 0): the power-of-two scales as
 * the 8-bit exponents block-scaled FP8 GEMMs on Blackwell read, byte e
 * standing for 2^(e - 127).  `scales` then addresses
 * FP8Q_PACKED_SCALE_BYTES(T, G) bytes: 32-bit words, word (k, t) at word
 * index k*T_pad + t (T_pad = T rounded up to a multiple of 4, k < ceil(G/4)),
 * whose byte j (little-endian) is the exponent of group 4k + j of token t.
 * Bytes of groups past G and of tokens past T are written as 0.  The pages
 * name the "float32 ceiling E8M0" / UE8M0 scales but print no packed layout;
 * this is the layout taken.
 */
#define FP8Q_PACKED_SCALE_BYTES(T, G) ((((G) + 3) / 4) * (((T) + 3) / 4 * 4) * 4)

/*
 * FP8Q_SCALES_UE8M0_MX (requires ue8m0 != 0): the same exponent bytes laid
 * out as the scale-factor operand of Blackwell's block-scaled FP8 GEMM
 * (MXFP8: one E8M0 byte per 32 values along K, tiles of 128 rows x 4 bytes,
 * the "32_4_4" swizzle), so the codes and these scales can be handed to such
 * a GEMM as they are.  A group's byte is repeated for its four 32-value
 * blocks.  The byte matrix [T_pad, 4G] (T_pad = T rounded up to 128) is
 * stored tile by tile, tile (t/128, g) at byte ((t/128)*G + g) * 512, and
 * inside a tile the 4 bytes of row r = t % 128 at byte (r % 32) * 16 +
 * (r / 32) * 4.  Rows past T are written as 0.  `scales` addresses
 * FP8Q_MX_SCALE_BYTES(T, G) bytes.
 */
#define FP8Q_MX_SCALE_BYTES(T, G) ((((T) + 127) / 128 * 128) * 4 * (G))

/* Longest rms_norm_per_block_quant row (H) the kernels accept (a row is held
 * in the registers of one CTA). */
#define FP8Q_RMS_MAX_H 32768

/*
 * per_token_group_fp8_quant.
 *   x       bf16 [T, H], read.
 *   q       e4m3 [T, H], written.
 *   scales  fp32 [T*G] in `scale_layout`, written.
 *   eps     floor of amax before the division by 448 (1e-10 in the reading
 *           above); must be finite and >= 1e-30 so that every scale is a
 *           normal fp32 number.
 * Result: bit-identical to the arithmetic in the header comment.
 */
FP8Q_API int fp8q_per_token_group_quant(const void *x, void *q, float *scales, int64_t T, int64_t H,
                               int32_t group_size, float eps, int32_t ue8m0, int32_t scale_layout,
                               void *stream);

/*
 * rms_norm_per_block_quant: RMSNorm of each token row, then the group
 * quantisation of the normalised row ("[RFC]: Using Helion for Selected vLLM
 * CustomOps", Motivation; the routed op keeps the "schema and mutation
 * contract" of the native op, section Routed Custom Op).
 *   x         bf16 [T, H], read.
 *   residual  bf16 [T, H] or NULL.  When given: z = bf16_RNE(x + residual) is
 *             written back into `residual` (the mutation), and z is normalised.
 *             Otherwise z = x.
 *   weight    bf16 [H], read.
 *   q, scales as for per_token_group_quant (scale floor 1e-10).
 *   eps       the RMSNorm variance epsilon (e.g. 1e-6), finite and >= 0.
 * Per row: ss = sum z_h^2 rounded once to fp32 (the GPU adds the squares
 * with error-free transformations, so ss is the exact sum rounded once unless
 * squares underflow fp32, |z| < ~1e-19); inv = RN32(1/RN32(sqrt(
 * RN32(RN32(ss/H) + eps)))); v_h = RN32(RN32(z_h * inv) * w_h); then the
 * group quantisation of v.  Outside the underflow case the result is
 * therefore the same, bit for bit, as a sequential evaluation of these steps
 * with the sum carried in double precision.  H <= FP8Q_RMS_MAX_H and
 * T < 2^30, else FP8Q_ERR_UNSUPPORTED.
 */
FP8Q_API int fp8q_rms_norm_per_block_quant(const void *x, void *residual, const void *weight, void *q,
                                  float *scales, int64_t T, int64_t H, int32_t group_size,
                                  float eps, int32_t ue8m0, int32_t scale_layout, void *stream);

/*
 * silu_and_mul_per_block_quant: SiLU(gate) * up, then the group quantisation
 * ("[RFC]: Using Helion for Selected vLLM CustomOps", Motivation).
 *   x       bf16 [T, 2I], read: gate a = x[t, 0:I], up b = x[t, I:2I].
 *   q       e4m3 [T, I], written.
 *   scales  fp32 [T*I/group_size] in `scale_layout`, written.
 *   eps     amax floor, as for per_token_group_quant.
 * v = RN32(RN32(a / RN32(1 + e^-a)) * b) (e^-a and the quotient as
 * fp8q_silu_mul states), then the group quantisation of v.
 */
FP8Q_API int fp8q_silu_and_mul_per_block_quant(const void *x, void *q, float *scales, int64_t T, int64_t I,
                                      int32_t group_size, float eps, int32_t ue8m0,
                                      int32_t scale_layout, void *stream);

/*
 * Per-token variants ("Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA",
 * section "Welche Kernel wurden in vLLM integriert": the three dynamic
 * per-token kernels listed next to the per-group ones).  The arithmetic is
 * that of the per-group op of the same name with the group spanning the
 * whole output row: one scale per token, s = RN32(max(amax_row, eps) / 448)
 * (ue8m0: rounded up to a power of two), q = e4m3(RN32(v / s)).
 *   scales  fp32 [T], written (s[t]); 4-byte aligned.
 *   The output row length (H, or I) must be a multiple of 128, else
 *   FP8Q_ERR_UNSUPPORTED (the kernels move 128-value chunks); pointers,
 *   eps and T == 0 as for the per-group calls.
 * Longest rows: FP8Q_TOKEN_MAX_COLS for the plain and the SiLU variant (a
 * row is spread over a cluster of up to 8 CTAs), FP8Q_RMS_MAX_H for the
 * RMSNorm variant; T * ceil(cols / 8192) < 2^31.
 */
#define FP8Q_TOKEN_MAX_COLS 65536

/* dynamic_per_token_scaled_fp8_quant: x bf16 [T, H] -> q e4m3 [T, H],
 * scales [T].  Bit-identical to the stated arithmetic. */
FP8Q_API int fp8q_dynamic_per_token_scaled_fp8_quant(const void *x, void *q, float *scales, int64_t T,
                                                     int64_t H, float eps, int32_t ue8m0, void *stream);

/* rms_norm_dynamic_per_token_quant: rms_norm_per_block_quant's residual,
 * RMSNorm and weight steps (same argument meaning, same exact sum of
 * squares, scale floor 1e-10), then one scale per row.  eps is the RMSNorm
 * variance epsilon. */
FP8Q_API int fp8q_rms_norm_dynamic_per_token_quant(const void *x, void *residual, const void *weight,
                                                   void *q, float *scales, int64_t T, int64_t H,
                                                   float eps, int32_t ue8m0, void *stream);

/* silu_and_mul_dynamic_per_token_quant: x bf16 [T, 2I] = [gate | up] ->
 * q e4m3 [T, I] of SiLU(gate) * up (as silu_and_mul_per_block_quant),
 * scales [T]. */
FP8Q_API int fp8q_silu_and_mul_dynamic_per_token_quant(const void *x, void *q, float *scales, int64_t T,
                                                       int64_t I, float eps, int32_t ue8m0, void *stream);

/*
 * fused_qk_norm_rope ("Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA",
 * section "Welche Kernel wurden in vLLM integriert"): per-head RMSNorm of
 * the query and key heads, then the rotary position embedding, in place.
 *   qkv        bf16 [T, (Hq + 2*Hkv) * D], read and written: per token the
 *              Hq query heads, then Hkv key heads, then Hkv value heads, D
 *              values each.  Query and key heads are replaced, value heads
 *              are not touched.
 *   q_weight, k_weight  bf16 [D], the norm weights of query and key heads.
 *   cos_sin    bf16 [max_position, D], row p = (cos_0..cos_{D/2-1},
 *              sin_0..sin_{D/2-1}) for position p (full rotary dimension).
 *   positions  int64 [T] (device), each in [0, max_position); a position
 *              outside is clamped into the table (the access stays in
 *              bounds; that token's result is unspecified).
 *   eps        RMSNorm variance epsilon, finite and >= 0.
 *   is_neox    nonzero: pairs (j, j + D/2); zero: pairs (2j, 2j + 1).
 * Per head: ss = sum z_i^2 (exact, rounded once), inv = RN32(1/RN32(sqrt(
 * RN32(RN32(ss/D) + eps)))), y_i = RN32(RN32(z_i inv) w_i); per pair (a, b)
 * with (c, s) = table[pos][j], table[pos][D/2 + j]: a' = RN32(RN32(a c) -
 * RN32(b s)), b' = RN32(RN32(b c) + RN32(a s)); the outputs are rounded to
 * bf16 (nearest even).  Bit-identical to this sequence.  D must be 128
 * (FP8Q_ERR_UNSUPPORTED otherwise); T * (Hq + Hkv) < 2^31.  Alignment: qkv,
 * the weights and the table 16 bytes, positions 8 bytes.
 */
FP8Q_API int fp8q_fused_qk_norm_rope(void *qkv, const void *q_weight, const void *k_weight, const void *cos_sin,
                                     const int64_t *positions, int64_t T, int64_t num_q_heads,
                                     int64_t num_kv_heads, int64_t head_dim, int64_t max_position, float eps,
                                     int32_t is_neox, void *stream);

/*
 * Elementwise fp32 -> float8_e4m3fn with round to nearest even and
 * saturation to +-448 (the rounding every op above applies to its
 * quotients).  v: fp32 [n] read, out: e4m3 [n] written; both 16-byte
 * aligned.  Exposed so the rounding can be checked on its own.
 */
FP8Q_API int fp8q_f32_to_e4m3(const float *v, void *out, int64_t n, void *stream);

/*
 * Elementwise out[i] = silu(a[i]) * b[i] in fp32, computed exactly as
 * silu_and_mul_per_block_quant computes the value it quantises:
 * RN32(RN32(a / RN32(1 + e^-a)) * b), the exponential from 2^(-a log2 e)
 * (PTX ex2.approx with the product's rounding error corrected), the quotient
 * from an approximate reciprocal with one exact-residual step.  Exposed so
 * the arithmetic can be checked on its own.  a, b, out: fp32 [n], 8-byte
 * aligned.
 */
FP8Q_API int fp8q_silu_mul(const float *a, const float *b, float *out, int64_t n, void *stream);

/*
 * Elementwise group scale: scales[i] = RN32(max(amax[i], eps) / 448), and
 * with ue8m0 != 0 the smallest power of two >= that value -- the scale every
 * op above forms from a group's (or row's) maximum |value|, computed by the
 * same device code (the division in two multiply-adds, correctly rounded).
 * Exposed so the division can be checked on its own over any fp32 amax.
 *   amax    fp32 [n], finite and >= 0, read;  scales fp32 [n], written;
 *           both 4-byte aligned.
 *   eps     as for per_token_group_quant (finite, >= 1e-30).
 */
FP8Q_API int fp8q_group_scale(const float *amax, float *scales, int64_t n, float eps, int32_t ue8m0, void *stream);

/*
 * Elementwise quotient codes: out[i] = e4m3(RN32(v[i] / s[i])), the code of
 * step A4 (quantise; "[RFC]: Using Helion for Selected vLLM CustomOps",
 * Motivation, the Block_FP8 1x128 scheme) as every op above forms it for a
 * scale that is not a power of two: the correctly rounded quotient from a
 * faithful start and one exact-residual step, computed by the same device
 * code.  Exposed so the quotient can be checked on its own over arbitrary
 * fp32 values and scales.
 *   v    fp32 [n], finite, read;  s  fp32 [n], positive and normal, with
 *        |v[i] / s[i]| finite in fp32, read;  both 4-byte aligned.
 *   out  float8_e4m3fn [n], written.
 */
FP8Q_API int fp8q_quant_pairs(const float *v, const float *s, void *out, int64_t n, void *stream);

/* Human-readable name of a status code (static storage, never NULL). */
FP8Q_API const char *fp8q_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
FP8Q_API int fp8q_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP8Q_H */
