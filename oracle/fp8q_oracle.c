/*
 * CPU oracle for the three fused FP8 quantisation epilogues.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so, which
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load.  The CUDA library never links it, includes it or calls it, and this
 * file includes nothing from the CUDA library: the two share no code.
 *
 * Plain, slow, single-threaded C11.  Every floating-point step is one IEEE
 * binary32 operation in the order written (the build passes
 * -ffp-contract=off, so no multiply-add is fused, and x86-64 evaluates float
 * expressions in float).  Bit patterns travel as uint16_t (bf16), uint8_t
 * (float8_e4m3fn) and float (fp32 scales).
 *
 * What is computed, and where it comes from:
 *
 *  - Block_FP8 activation scaling: one scale per contiguous 1x128 group of a
 *    token row ("Helion：用自动调优改进 vLLM 推理", section "Scope"/范围,
 *    the Block_FP8 bullet).
 *  - The three ops per_token_group_fp8_quant, silu_and_mul_per_block_quant
 *    and rms_norm_per_block_quant ("[RFC]: Using Helion for Selected vLLM
 *    CustomOps", Motivation, the initial-rollout list).
 *  - Power-of-two "ceiling E8M0" scales ("[RFC]: Using Helion for Selected
 *    vLLM CustomOps", End-to-End Model Performance, H100 settings: "float32
 *    ceiling E8M0 scales"; "Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA",
 *    section "Praktische Einschränkungen": UE8M0 scales).
 *
 * The pages print no formula.  The arithmetic below is the plain reading
 * that the rest supports, one step per line:
 *
 *   amax   = max_i |x_i| over the group                      (exact)
 *   s      = RN32( max(amax, eps) / 448 ),  eps = 1e-10f
 *   ue8m0: s <- smallest power of two >= s                   (exact, bit ops)
 *   q_i    = e4m3( RN32( x_i / s ) )
 *   e4m3(v): round to nearest, ties to the even code, |v| > 448 -> +-448,
 *            subnormals kept (smallest 2^-9), sign of zero kept.
 *
 *   rms:   z_h = bf16_RNE( RN32(x_h + r_h) )  (residual given; z written back)
 *          ss  = (float) sum_h z_h^2  (accumulated in double, rounded once)
 *          inv = RN32( 1 / RN32( sqrt( RN32( RN32(ss / H) + eps_rms ))))
 *          v_h = RN32( RN32(z_h * inv) * w_h ),  then the group quant of v.
 *   silu:  a = x[t, g*gs + i] (gate, first half), b = x[t, I + g*gs + i] (up)
 *          v = RN32( RN32( a / RN32(1 + expf(-a)) ) * b ),  then the group quant.
 *
 * Scale layouts: row-major s[t*G + g], column-major s[g*T + t], G = H/gs.
 *
 * Per-token variants.  "Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA",
 * section "Welche Kernel wurden in vLLM integriert", lists three per-token
 * kernels next to the per-group ones: dynamic_per_token_scaled_fp8_quant,
 * rms_norm_dynamic_per_token_quant and silu_and_mul_dynamic_per_token_quant.
 * The pages give them no formula either; the plain reading is the same
 * arithmetic with the group spanning the whole row (gs = H, or gs = I), i.e.
 * one scale per token, s[t].  The functions below take any gs that divides
 * the row, so the per-token ops are these functions called with gs = H.
 */
#include "fp8q_oracle.h"

#include <math.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even on the 16 dropped bits. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t low = u & 0xFFFFu;
    uint32_t high = u >> 16;
    if (low > 0x8000u || (low == 0x8000u && (high & 1u)))
        high += 1u; /* carry may ripple into the exponent: that is correct */
    return (uint16_t)high;
}

/* ------------------------------------------------------- float8 e4m3fn -- */

/*
 * Round an fp32 value to float8_e4m3fn.
 *
 * Format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  A normal
 * code with exponent field E in 1..15 and mantissa M is (1 + M/8) * 2^(E-7);
 * E = 0 codes are subnormal, M * 2^-9.  S.1111.111 is NaN; there is no
 * infinity, so the largest finite magnitude is 448 = S.1111.110.
 *
 * For |v| in binade [2^k, 2^(k+1)), k >= -6, the representable values are
 * n * 2^(k-3) for integers n in [8, 16]; below 2^-6 the spacing stays 2^-9
 * (k is clamped to -6).  So: n = |v| / 2^(k-3) (exact: a power-of-two
 * scaling), round n to the nearest integer with ties to even, and the code
 * is (k + 6) * 8 + n.  n = 16 carries into the next exponent, which the same
 * formula already encodes.  Magnitudes >= 448 saturate to 448.
 */
uint8_t oracle_f32_to_e4m3(float v)
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    uint8_t sign = (u >> 31) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    float a = fabsf(v);
    if (a >= 448.0f)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0f)
        return sign;

    int e;
    (void)frexpf(a, &e); /* a = f * 2^e, f in [0.5, 1): floor(log2 a) = e - 1 */
    int k = e - 1;
    if (k < -6)
        k = -6;
    float n = ldexpf(a, 3 - k); /* exact; in [8, 16) for k > -6, [0, 16) for k = -6 */

    float fl = floorf(n);
    float frac = n - fl; /* exact */
    float r;
    if (frac > 0.5f)
        r = fl + 1.0f;
    else if (frac < 0.5f)
        r = fl;
    else
        r = (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;

    int code = (k + 6) * 8 + (int)r;
    return (uint8_t)(sign | code);
}

float oracle_e4m3_to_f32(uint8_t c)
{
    int sgn = c & 0x80;
    int E = (c >> 3) & 0xF;
    int M = c & 0x7;
    float mag;
    if (E == 0xF && M == 0x7)
        mag = NAN;
    else if (E == 0)
        mag = ldexpf((float)M, -9);
    else
        mag = ldexpf(1.0f + (float)M / 8.0f, E - 7);
    return sgn ? -mag : mag;
}

/* ------------------------------------------------------------ scales -- */

/*
 * Smallest power of two >= s, for s > 0 (the "ceiling E8M0" rounding).
 * s = f * 2^e with f in [0.5, 1): s is a power of two exactly when f = 0.5;
 * otherwise the answer is 2^e.  Exact, no rounding involved.
 */
float oracle_ue8m0_ceil(float s)
{
    if (!(s > 0.0f) || isinf(s))
        return s;
    int e;
    float f = frexpf(s, &e);
    if (f == 0.5f)
        return s;
    return ldexpf(1.0f, e);
}

float oracle_group_scale(float amax, float eps, int ue8m0, float *pre)
{
    float s = fmaxf(amax, eps) / 448.0f;
    if (pre)
        *pre = s;
    return ue8m0 ? oracle_ue8m0_ceil(s) : s;
}

static int64_t scale_index(int64_t t, int64_t g, int64_t T, int64_t G, int col_major)
{
    return col_major ? g * T + t : t * G + g;
}

/* Quantise one group v[0..gs) (fp32) given its precomputed fp32 scale. */
static void quant_group(const float *v, int64_t gs, float s, uint8_t *q)
{
    for (int64_t i = 0; i < gs; ++i) {
        float p = v[i] / s; /* RN32 quotient */
        q[i] = oracle_f32_to_e4m3(p);
    }
}

static float group_amax(const float *v, int64_t gs)
{
    float m = 0.0f;
    for (int64_t i = 0; i < gs; ++i) {
        float a = fabsf(v[i]);
        if (a > m)
            m = a;
    }
    return m;
}

static int check_shape(int64_t T, int64_t H, int64_t gs)
{
    if (T < 0 || H <= 0 || gs <= 0 || H % gs != 0)
        return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/* ------------------------------------------- op A: per-token-group quant -- */

int oracle_per_token_group_quant(const uint16_t *x, uint8_t *q, float *scales, float *scales_pre,
                                 int64_t T, int64_t H, int64_t gs, float eps, int ue8m0,
                                 int col_major)
{
    int rc = check_shape(T, H, gs);
    if (rc)
        return rc;
    if (gs > ORACLE_MAX_ROW)
        return ORACLE_ERR_ARG;
    const int64_t G = H / gs;
    static float v[ORACLE_MAX_ROW];
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t g = 0; g < G; ++g) {
            const uint16_t *xg = x + t * H + g * gs;
            for (int64_t i = 0; i < gs; ++i)
                v[i] = oracle_bf16_to_f32(xg[i]);
            float pre;
            float s = oracle_group_scale(group_amax(v, gs), eps, ue8m0, &pre);
            int64_t si = scale_index(t, g, T, G, col_major);
            scales[si] = s;
            if (scales_pre)
                scales_pre[si] = pre;
            quant_group(v, gs, s, q + t * H + g * gs);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------- op B: RMSNorm + per-block quant -- */

float oracle_rms_inv(float ss, int64_t H, float eps)
{
    float mean = ss / (float)H;
    float var = mean + eps;
    float rstd = sqrtf(var);
    return 1.0f / rstd;
}

int oracle_rms_norm_per_block_quant(const uint16_t *x, uint16_t *residual, const uint16_t *w,
                                    uint8_t *q, float *scales, float *scales_pre, float *inv_out,
                                    float *v_out, int64_t T, int64_t H, int64_t gs, float eps,
                                    int ue8m0, int col_major)
{
    int rc = check_shape(T, H, gs);
    if (rc)
        return rc;
    if (H > ORACLE_MAX_ROW)
        return ORACLE_ERR_ARG;
    const int64_t G = H / gs;
    static float z[ORACLE_MAX_ROW];
    static float v[ORACLE_MAX_ROW];
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *xr = x + t * H;
        /* optional residual add: z = bf16(x + r), written back to residual */
        if (residual) {
            uint16_t *rr = residual + t * H;
            for (int64_t h = 0; h < H; ++h) {
                float sum = oracle_bf16_to_f32(xr[h]) + oracle_bf16_to_f32(rr[h]);
                uint16_t zb = oracle_f32_to_bf16(sum);
                rr[h] = zb;
                z[h] = oracle_bf16_to_f32(zb);
            }
        } else {
            for (int64_t h = 0; h < H; ++h)
                z[h] = oracle_bf16_to_f32(xr[h]);
        }
        /* sum of squares over the whole row, in double, rounded once */
        double acc = 0.0;
        for (int64_t h = 0; h < H; ++h)
            acc += (double)z[h] * (double)z[h];
        float ss = (float)acc;
        float inv = oracle_rms_inv(ss, H, eps);
        if (inv_out)
            inv_out[t] = inv;
        for (int64_t h = 0; h < H; ++h) {
            float n = z[h] * inv;
            v[h] = n * oracle_bf16_to_f32(w[h]);
            if (v_out)
                v_out[t * H + h] = v[h];
        }
        for (int64_t g = 0; g < G; ++g) {
            float pre;
            float s = oracle_group_scale(group_amax(v + g * gs, gs), ORACLE_SCALE_EPS, ue8m0, &pre);
            int64_t si = scale_index(t, g, T, G, col_major);
            scales[si] = s;
            if (scales_pre)
                scales_pre[si] = pre;
            quant_group(v + g * gs, gs, s, q + t * H + g * gs);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------ op C: SiLU-and-mul + block quant -- */

float oracle_silu_mul(float a, float b)
{
    float d = 1.0f + expf(-a);
    float sg = a / d;
    return sg * b;
}

int oracle_silu_and_mul_per_block_quant(const uint16_t *x, uint8_t *q, float *scales,
                                        float *scales_pre, float *v_out, int64_t T, int64_t I,
                                        int64_t gs, float eps, int ue8m0, int col_major)
{
    int rc = check_shape(T, I, gs);
    if (rc)
        return rc;
    if (gs > ORACLE_MAX_ROW)
        return ORACLE_ERR_ARG;
    const int64_t G = I / gs;
    static float v[ORACLE_MAX_ROW];
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *xr = x + t * 2 * I;
        for (int64_t g = 0; g < G; ++g) {
            for (int64_t i = 0; i < gs; ++i) {
                float a = oracle_bf16_to_f32(xr[g * gs + i]);
                float b = oracle_bf16_to_f32(xr[I + g * gs + i]);
                v[i] = oracle_silu_mul(a, b);
                if (v_out)
                    v_out[t * I + g * gs + i] = v[i];
            }
            float pre;
            float s = oracle_group_scale(group_amax(v, gs), eps, ue8m0, &pre);
            int64_t si = scale_index(t, g, T, G, col_major);
            scales[si] = s;
            if (scales_pre)
                scales_pre[si] = pre;
            quant_group(v, gs, s, q + t * I + g * gs);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------ fused_qk_norm_rope (f4) -- */

/*
 * fused_qk_norm_rope ("Helion-Kernel in vLLM: PyTorch FP8 ohne CUDA",
 * section "Welche Kernel wurden in vLLM integriert", and its speed-up in
 * "Leistung auf Kernel-Ebene"; the pages give the name only).  The plain
 * reading of the name, as Qwen3 attention uses it: per-head RMSNorm of the
 * query and key heads ("QK norm", one weight vector of length D for all query
 * heads, another for all key heads), then the rotary position embedding of
 * each normalised head, written back in place; the value heads are not
 * touched.  Per token t and head h (Hq query heads, then Hkv key heads, then
 * Hkv value heads, each D contiguous bf16 values):
 *
 *   z_i   = x_i                                   (bf16 -> fp32, exact)
 *   ss    = (float) sum_i z_i^2                   (double, rounded once)
 *   inv   = RN32(1 / RN32(sqrt(RN32(RN32(ss / D) + eps))))   (as op B)
 *   y_i   = RN32( RN32(z_i * inv) * w_i )         (w = q_weight or k_weight)
 *   c_j, s_j = cos_sin[pos_t][j], cos_sin[pos_t][D/2 + j], j < D/2 (bf16)
 *   pairs (a, b) = (y_j, y_{j+D/2}) (neox style) or (y_{2j}, y_{2j+1})
 *   a' = RN32( RN32(a * c_j) - RN32(b * s_j) )
 *   b' = RN32( RN32(b * c_j) + RN32(a * s_j) )
 *   x  <- bf16_RNE(a'), bf16_RNE(b')
 *
 * cos_sin is bf16 [P, D] (full rotary dimension); every position must lie in
 * [0, P).
 */
int oracle_fused_qk_norm_rope(uint16_t *qkv, const uint16_t *q_w, const uint16_t *k_w,
                              const uint16_t *cos_sin, const int64_t *positions, int64_t T,
                              int64_t Hq, int64_t Hkv, int64_t D, int64_t P, float eps, int is_neox)
{
    if (T < 0 || Hq < 0 || Hkv < 0 || D <= 0 || D % 2 != 0 || D > ORACLE_MAX_ROW || P <= 0)
        return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < T; ++t)
        if (positions[t] < 0 || positions[t] >= P)
            return ORACLE_ERR_ARG;
    const int64_t row = (Hq + 2 * Hkv) * D, half = D / 2;
    static float y[ORACLE_MAX_ROW];
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *cs = cos_sin + positions[t] * D;
        for (int64_t h = 0; h < Hq + Hkv; ++h) {
            uint16_t *x = qkv + t * row + h * D;
            const uint16_t *w = h < Hq ? q_w : k_w;
            double acc = 0.0;
            for (int64_t i = 0; i < D; ++i) {
                double z = (double)oracle_bf16_to_f32(x[i]);
                acc += z * z;
            }
            float inv = oracle_rms_inv((float)acc, D, eps);
            for (int64_t i = 0; i < D; ++i) {
                float n = oracle_bf16_to_f32(x[i]) * inv;
                y[i] = n * oracle_bf16_to_f32(w[i]);
            }
            for (int64_t j = 0; j < half; ++j) {
                const int64_t ia = is_neox ? j : 2 * j;
                const int64_t ib = is_neox ? j + half : 2 * j + 1;
                float c = oracle_bf16_to_f32(cs[j]);
                float sn = oracle_bf16_to_f32(cs[half + j]);
                float a = y[ia], b = y[ib];
                float ac = a * c, bs = b * sn, bc = b * c, as = a * sn;
                x[ia] = oracle_f32_to_bf16(ac - bs);
                x[ib] = oracle_f32_to_bf16(bc + as);
            }
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------- packed UE8M0 scales -- */

/*
 * Power-of-two ("ceiling E8M0") scales as the 8-bit exponents that block-
 * scaled FP8 GEMMs on Blackwell read: an E8M0 byte b stands for 2^(b - 127).
 * Layout: 32-bit words, token-major in the fast dimension and four groups per
 * word: word (k, t), k < ceil(G/4), t < T_pad = T rounded up to a multiple
 * of 4, lives at word index k * T_pad + t, and its byte j (little-endian,
 * j = 0..3) is the exponent of group 4k + j of token t.  Bytes of groups
 * past G and of tokens past T are 0.  Input: the fp32 scales, row-major
 * [T, G], each a power of two.  Output: ceil(G/4) * T_pad * 4 bytes.
 */
int oracle_pack_ue8m0(const float *scales_tg, int64_t T, int64_t G, uint8_t *out)
{
    if (T < 0 || G <= 0)
        return ORACLE_ERR_ARG;
    const int64_t T_pad = (T + 3) / 4 * 4;
    const int64_t K = (G + 3) / 4;
    memset(out, 0, (size_t)(K * T_pad * 4));
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t g = 0; g < G; ++g) {
            float s = scales_tg[t * G + g];
            int e;
            float f = frexpf(s, &e); /* s = f * 2^e, f in [0.5, 1) */
            if (f != 0.5f || e - 1 + 127 < 1 || e - 1 + 127 > 254)
                return ORACLE_ERR_ARG; /* not a normal power of two */
            int64_t word = (g / 4) * T_pad + t;
            out[word * 4 + (g % 4)] = (uint8_t)(e - 1 + 127); /* s = 2^(e-1) */
        }
    }
    return ORACLE_OK;
}

/*
 * The same exponent bytes in the scale-factor layout of Blackwell's
 * block-scaled (MXFP8) GEMM operands: one E8M0 byte per 32 values along the
 * row, so a 1x128 group's byte is repeated for its four 32-value blocks; the
 * [T_pad, 4G] byte matrix (T_pad = T rounded up to 128) is stored as tiles of
 * 128 rows x 4 columns, tile (T_pad-row block rb, column block cb) at byte
 * (rb * G + cb) * 512 (column blocks = G), and inside a tile the byte of row
 * r, column c at (r % 32) * 16 + (r / 32) * 4 + c.  Column block cb is then
 * exactly group cb.  Rows past T are 0.  Output: T_pad * 4 * G bytes.
 */
int oracle_pack_ue8m0_mx(const float *scales_tg, int64_t T, int64_t G, uint8_t *out)
{
    if (T < 0 || G <= 0)
        return ORACLE_ERR_ARG;
    const int64_t T_pad = (T + 127) / 128 * 128;
    memset(out, 0, (size_t)(T_pad * 4 * G));
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t g = 0; g < G; ++g) {
            float s = scales_tg[t * G + g];
            int e;
            float f = frexpf(s, &e);
            if (f != 0.5f || e - 1 + 127 < 1 || e - 1 + 127 > 254)
                return ORACLE_ERR_ARG;
            for (int64_t c = 4 * g; c < 4 * g + 4; ++c) { /* the group's four 32-value blocks */
                int64_t rb = t / 128, r = t % 128, cb = c / 4, cc = c % 4;
                int64_t at = (rb * G + cb) * 512 + (r % 32) * 16 + (r / 32) * 4 + cc;
                out[at] = (uint8_t)(e - 1 + 127);
            }
        }
    }
    return ORACLE_OK;
}

/* ----------------------------------------------- batch helpers (tests) -- */

/* The group scale of each amax[i], as every op forms it (test helper). */
void oracle_group_scale_n(const float *amax, float *out, int64_t n, float eps, int ue8m0)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_group_scale(amax[i], eps, ue8m0, NULL);
}

void oracle_f32_to_e4m3_n(const float *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_e4m3(v[i]);
}

void oracle_ue8m0_ceil_n(const float *s, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_ue8m0_ceil(s[i]);
}

void oracle_silu_mul_n(const float *a, const float *b, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_silu_mul(a[i], b[i]);
}

/* Quotient codes for explicit (value, scale) pairs: e4m3(RN32(v / s)). */
void oracle_quant_pairs(const float *v, const float *s, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_e4m3(v[i] / s[i]);
}

/* Row sums of squares exactly as the rms op forms them (double, rounded once). */
void oracle_row_sumsq(const uint16_t *z, int64_t T, int64_t H, float *out)
{
    for (int64_t t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double f = (double)oracle_bf16_to_f32(z[t * H + h]);
            acc += f * f;
        }
        out[t] = (float)acc;
    }
}
