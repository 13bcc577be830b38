/*
 * CPU oracle for the three fused FP8 quantisation epilogues.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg.  Shares no code with the CUDA library.
 * The arithmetic each function follows is stated in fp8q_oracle.c.
 *
 * All arrays are host memory, row-major and contiguous.  bf16 values travel
 * as their uint16_t bit patterns, float8_e4m3fn values as uint8_t codes.
 * `col_major` selects the scale layout: 0 -> s[t*G + g], 1 -> s[g*T + t].
 * `scales_pre` (may be NULL) receives each group's scale before the
 * power-of-two rounding (equal to `scales` when ue8m0 == 0).
 * The group size gs may be anything that divides the row, up to
 * ORACLE_MAX_ROW: gs = H gives the per-token variants (one scale per row).
 * Not thread-safe (row buffers are static).
 */
#ifndef FP8Q_ORACLE_H
#define FP8Q_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_MAX_ROW (1 << 20)
#define ORACLE_SCALE_EPS 1e-10f

float oracle_bf16_to_f32(uint16_t b);
uint16_t oracle_f32_to_bf16(float f);
uint8_t oracle_f32_to_e4m3(float v);
float oracle_e4m3_to_f32(uint8_t c);
float oracle_ue8m0_ceil(float s);
float oracle_group_scale(float amax, float eps, int ue8m0, float *pre);
void oracle_group_scale_n(const float *amax, float *out, int64_t n, float eps, int ue8m0);
float oracle_rms_inv(float ss, int64_t H, float eps);
float oracle_silu_mul(float a, float b);

/* op A: x bf16 [T,H] -> q e4m3 [T,H], scales fp32 [T*H/gs] */
int oracle_per_token_group_quant(const uint16_t *x, uint8_t *q, float *scales, float *scales_pre,
                                 int64_t T, int64_t H, int64_t gs, float eps, int ue8m0,
                                 int col_major);

/* op B: x bf16 [T,H], residual bf16 [T,H] in/out or NULL, w bf16 [H];
 * eps is the RMSNorm variance epsilon; the scale floor is ORACLE_SCALE_EPS.
 * inv_out (may be NULL) receives each row's 1/rms; v_out (may be NULL) the
 * fp32 values [T,H] that are quantised. */
int oracle_rms_norm_per_block_quant(const uint16_t *x, uint16_t *residual, const uint16_t *w,
                                    uint8_t *q, float *scales, float *scales_pre, float *inv_out,
                                    float *v_out, int64_t T, int64_t H, int64_t gs, float eps,
                                    int ue8m0, int col_major);

/* op C: x bf16 [T,2I] (gate | up) -> q e4m3 [T,I], scales fp32 [T*I/gs];
 * v_out (may be NULL) receives the fp32 values [T,I] that are quantised. */
int oracle_silu_and_mul_per_block_quant(const uint16_t *x, uint8_t *q, float *scales,
                                        float *scales_pre, float *v_out, int64_t T, int64_t I,
                                        int64_t gs, float eps, int ue8m0, int col_major);

/* fused_qk_norm_rope: qkv bf16 [T, (Hq + 2*Hkv) * D] in/out (query and key
 * heads normalised and rotated in place, value heads untouched), q_w / k_w
 * bf16 [D], cos_sin bf16 [P, D] (cos | sin halves), positions [T] in [0, P). */
int oracle_fused_qk_norm_rope(uint16_t *qkv, const uint16_t *q_w, const uint16_t *k_w,
                              const uint16_t *cos_sin, const int64_t *positions, int64_t T,
                              int64_t Hq, int64_t Hkv, int64_t D, int64_t P, float eps, int is_neox);

/* Packed UE8M0 scales (layout in fp8q_oracle.c): scales_tg fp32 [T,G]
 * row-major powers of two -> ceil(G/4) * round_up(T,4) * 4 bytes. */
int oracle_pack_ue8m0(const float *scales_tg, int64_t T, int64_t G, uint8_t *out);

/* The MXFP8 scale-factor tile layout of the same bytes (layout in
 * fp8q_oracle.c): round_up(T,128) * 4 * G bytes. */
int oracle_pack_ue8m0_mx(const float *scales_tg, int64_t T, int64_t G, uint8_t *out);

void oracle_f32_to_e4m3_n(const float *v, uint8_t *out, int64_t n);
void oracle_ue8m0_ceil_n(const float *s, float *out, int64_t n);
void oracle_silu_mul_n(const float *a, const float *b, float *out, int64_t n);
void oracle_quant_pairs(const float *v, const float *s, uint8_t *out, int64_t n);
void oracle_row_sumsq(const uint16_t *z, int64_t T, int64_t H, float *out);

#ifdef __cplusplus
}
#endif
#endif
