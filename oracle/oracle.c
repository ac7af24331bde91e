/*
 * oracle.c -- plain, slow CPU reference for the fused RMSNorm -> Linear
 * projection and its quantised, two-stage and skinny forms.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the package's smoke check and
 * the benchmark's CPU-baseline leg load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls
 * it.
 *
 * Sources (the four web pages this method is described on):
 *   [AT10]  "PyPTO-Gym operator design pattern AT-10: RMSNorm + Linear fusion
 *           (V->C layout) -- principles and MLAProlog in practice"
 *           (pwwt.cn/news/4832734):
 *           sec. 2 "CV layout and standard compute flow",
 *           sec. 3 "V stage: the two RMSNorm variants" (variant A rsqrt,
 *                  variant B sqrt + div, the AT-03 parameter table),
 *           sec. 4 "C stage: the three Linear modes" (BF16, INT8 W8A8, MXFP8),
 *           sec. 5 "MLAProlog" (q_a_proj -> rms_norm -> *gamma_cq -> cast ->
 *                  q_b_proj),
 *           sec. 8 "tuning" (the mhc_pre skinny form),
 *           sec. 9 "golden comparison".
 *   [SK03]  "SK-03 Linear Projection (Norm->MatMul) skeleton" (lpqz.cn/news/36925):
 *           "quantised variant (AT-11) in the source" (common.py quant),
 *           "shape variant: huge reduction x tiny output width (mhc_pre)".
 *   [SK14]  "SK-14 general multi-MatMul skeleton" (pgsm.cn/news/456816):
 *           "variant A in practice: QuantMatMulReduceSum" (dequant order).
 *
 * Precision.  Everything is IEEE binary64 (plain loops, no blocking, no
 * reordering beyond a sequential sum), except the W8A8 front end
 * (orc_quant_rows_f32): there floating point decides integer codes, so it is
 * done in binary32, the precision the pages fix for the norm (FP32 inside
 * the V stage, [AT10] sec. 2/3, rule C-API-05), in the pages' order of
 * operations.  Build with -ffp-contract=off so no multiply-add is fused.
 *
 * bf16 values are passed as their 16-bit patterns (uint16_t).
 */
#include <limits.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EARG (-1)
#define ORC_ENOMEM (-2)
#define ORC_OVERFLOW 1

/* ------------------------------------------------------------------------ */
/* bfloat16 codec, written from the format's definition: 1 sign bit, the 8   */
/* exponent bits of binary32 (bias 127), 7 stored fraction bits; rounding is */
/* to nearest, ties to even.                                                 */
/* ------------------------------------------------------------------------ */

uint16_t orc_bf16_rne(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v))
        return (uint16_t)(sign | 0x7FC0u);
    if (isinf(v))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1 */
    int biased = e - 1 + 127;
    if (biased <= 0) {
        /* below the smallest normal: fixed quantum 2^-133 (2^-126 * 2^-7) */
        double r = nearbyint(ldexp(a, 133)); /* r <= 128; 128 == smallest normal */
        return (uint16_t)(sign | (uint16_t)r);
    }
    double r = nearbyint(m * 256.0); /* 8 significant bits */
    if (r == 256.0) {
        r = 128.0;
        biased += 1;
    }
    if (biased >= 255)
        return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)(biased << 7) | (uint16_t)((int)r - 128));
}

double orc_bf16_value(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static float bf16_as_float(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

void orc_bf16_rne_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_rne(v[i]);
}

int orc_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* AT-03 RMSNorm of one row, binary64.  [AT10] sec. 3.                      */
/*   variant 0 (A, "rsqrt"):    ms = (sum x^2) * (1/D); rstd = 1/sqrt(ms+eps) */
/*   variant 1 (B, sqrt + div): ms = sum (x^2 * (1/D)); std = sqrt(ms+eps);  */
/*                              rstd = 1/std                                 */
/* In binary64 the two differ only by rounding.                              */
/* ------------------------------------------------------------------------ */

static double row_rstd_f64(const uint16_t *xr, int64_t K, double eps, int variant)
{
    double inv_d = 1.0 / (double)K;
    double s = 0.0;
    if (variant == 0) {
        for (int64_t k = 0; k < K; ++k) {
            double v = orc_bf16_value(xr[k]);
            s += v * v;
        }
        double ms = s * inv_d;
        return 1.0 / sqrt(ms + eps);
    }
    for (int64_t k = 0; k < K; ++k) {
        double v = orc_bf16_value(xr[k]);
        s += (v * v) * inv_d;
    }
    double sd = sqrt(s + eps);
    return 1.0 / sd;
}

/* y[t,k] = x[t,k] * rstd[t] (* gamma[k] when gamma != NULL), binary64. */
int orc_rmsnorm_f64(const uint16_t *x, const uint16_t *gamma, int64_t T, int64_t K,
                    double eps, int variant, double *y, double *rstd)
{
    if (!x || T < 0 || K <= 0 || (variant != 0 && variant != 1))
        return ORC_EARG;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *xr = x + t * K;
        double r = row_rstd_f64(xr, K, eps, variant);
        if (rstd)
            rstd[t] = r;
        if (y) {
            for (int64_t k = 0; k < K; ++k) {
                double v = orc_bf16_value(xr[k]) * r;
                if (gamma)
                    v = v * orc_bf16_value(gamma[k]);
                y[t * K + k] = v;
            }
        }
    }
    return ORC_OK;
}

static double *decode_matrix(const uint16_t *m, int64_t n)
{
    double *d = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!d)
        return NULL;
    for (int64_t i = 0; i < n; ++i)
        d[i] = orc_bf16_value(m[i]);
    return d;
}

/* ------------------------------------------------------------------------ */
/* AT-10 RMSNorm + Linear.  [AT10] sec. 2 (compute flow) and sec. 4 (AT-09   */
/* BF16 mode: matmul(x, w, BF16, b_trans=True), W stored [N, K]).            */
/*                                                                           */
/* form 0 (AT-10):  a = bf16(x * rstd * gamma); out = bf16(sum_k a*W[n,k]).  */
/* form 1 (mhc_pre, [AT10] sec. 8 / [SK03] shape variant): the normed values */
/*                  stay in full precision, the matmul is FP32 and so is the */
/*                  output: out = fp32(sum_k (x*rstd*gamma)*W[n,k]).         */
/* ref[t,n] receives the binary64 sum before the final rounding; out is      */
/* uint16_t (bf16 bits) for form 0 and float for form 1.                     */
/* ------------------------------------------------------------------------ */

int orc_rmsnorm_linear(const uint16_t *x, const uint16_t *gamma, const uint16_t *W,
                       int64_t T, int64_t K, int64_t N, double eps, int variant, int form,
                       double *ref, void *out)
{
    if (!x || !W || T < 0 || K <= 0 || N <= 0 || (variant != 0 && variant != 1) ||
        (form != 0 && form != 1))
        return ORC_EARG;
    double *wd = decode_matrix(W, N * K);
    if (!wd)
        return ORC_ENOMEM;
    int status = ORC_OK;
#pragma omp parallel
    {
        double *a = (double *)malloc((size_t)K * sizeof(double));
        if (!a) {
#pragma omp atomic write
            status = ORC_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            if (!a)
                continue;
            const uint16_t *xr = x + t * K;
            double r = row_rstd_f64(xr, K, eps, variant);
            for (int64_t k = 0; k < K; ++k) {
                double v = orc_bf16_value(xr[k]) * r;
                if (gamma)
                    v = v * orc_bf16_value(gamma[k]);
                a[k] = (form == 0) ? orc_bf16_value(orc_bf16_rne(v)) : v;
            }
            for (int64_t n = 0; n < N; ++n) {
                const double *wr = wd + n * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += a[k] * wr[k];
                if (ref)
                    ref[t * N + n] = acc;
                if (out) {
                    if (form == 0)
                        ((uint16_t *)out)[t * N + n] = orc_bf16_rne(acc);
                    else
                        ((float *)out)[t * N + n] = (float)acc;
                }
            }
        }
        free(a);
    }
    free(wd);
    return status;
}

/* ------------------------------------------------------------------------ */
/* AT-10 with the options of its two atoms.                                  */
/*   [AT10] sec. 6 (Qwen3PreAttn): the norm is applied to x_add, the input   */
/*          after the residual add: x_add = bf16(x + residual), the sum of   */
/*          two bf16 values rounded once (exact in binary64 before that).    */
/*   [AT10] sec. 3, AT-03 parameter table: has_bias (a bias added to the     */
/*          normed row, after gamma: y = x_add * rstd * gamma + beta) and    */
/*          output_rstd (rstd per row, as InplaceAddRmsNorm returns it).     */
/*   [AT10] sec. 4, AT-09 parameters: has_bias of the projection, added to   */
/*          the accumulator before the output cast:                          */
/*          out = bf16(sum_k a[k] * W[n,k] + bias[n]).                        */
/* residual, gamma, beta, bias may each be NULL (option off).  x_sum (bf16   */
/* bits of x_add, [T,K]), rstd ([T]) and ref ([T,N], binary64 before the     */
/* output cast) are optional outputs.                                        */
/* ------------------------------------------------------------------------ */

int orc_rmsnorm_linear_ex(const uint16_t *x, const uint16_t *residual, const uint16_t *gamma,
                          const uint16_t *beta, const uint16_t *W, const uint16_t *bias,
                          int64_t T, int64_t K, int64_t N, double eps, int variant,
                          double *ref, uint16_t *out, uint16_t *x_sum, double *rstd)
{
    if (!x || !W || T < 0 || K <= 0 || N <= 0 || (variant != 0 && variant != 1))
        return ORC_EARG;
    double *wd = decode_matrix(W, N * K);
    if (!wd)
        return ORC_ENOMEM;
    int status = ORC_OK;
#pragma omp parallel
    {
        uint16_t *xa = (uint16_t *)malloc((size_t)K * sizeof(uint16_t));
        double *a = (double *)malloc((size_t)K * sizeof(double));
        if (!xa || !a) {
#pragma omp atomic write
            status = ORC_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            if (!xa || !a)
                continue;
            const uint16_t *xr = x + t * K;
            for (int64_t k = 0; k < K; ++k) {
                if (residual)
                    xa[k] = orc_bf16_rne(orc_bf16_value(xr[k]) +
                                         orc_bf16_value(residual[t * K + k]));
                else
                    xa[k] = xr[k];
                if (x_sum)
                    x_sum[t * K + k] = xa[k];
            }
            double r = row_rstd_f64(xa, K, eps, variant);
            if (rstd)
                rstd[t] = r;
            for (int64_t k = 0; k < K; ++k) {
                double v = orc_bf16_value(xa[k]) * r;
                if (gamma)
                    v = v * orc_bf16_value(gamma[k]);
                if (beta)
                    v = v + orc_bf16_value(beta[k]);
                a[k] = orc_bf16_value(orc_bf16_rne(v));
            }
            for (int64_t n = 0; n < N; ++n) {
                const double *wr = wd + n * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += a[k] * wr[k];
                if (bias)
                    acc = acc + orc_bf16_value(bias[n]);
                if (ref)
                    ref[t * N + n] = acc;
                if (out)
                    out[t * N + n] = orc_bf16_rne(acc);
            }
        }
        free(xa);
        free(a);
    }
    free(wd);
    return status;
}

/* ------------------------------------------------------------------------ */
/* The V stage after the QKV projection.  [AT10] sec. 6 (Qwen3PreAttn): the  */
/* projection output is split into Q, K and V, and Q and K each get a        */
/* per-head RMSNorm (their own gamma over head_dim) and RoPE.                */
/*   y [T, (Hq + 2 Hkv) * D] bf16: columns [0, Hq D) are the q heads,        */
/*     [Hq D, (Hq + Hkv) D) the k heads, the rest the v heads.               */
/*   q / k head row h (D values): ms = mean(h^2) (binary64), r = 1/sqrt(ms   */
/*     + eps), z = bf16(h * r * gamma) (the norm's bf16 output); RoPE with   */
/*     the rotate-half pairing, angle table cs [P, D] (cos in [0, D/2), sin  */
/*     in [D/2, D)) at position pos[t]:                                      */
/*       o[i]       = bf16(z[i] * c_i - z[i + D/2] * s_i)                    */
/*       o[i + D/2] = bf16(z[i + D/2] * c_i + z[i] * s_i),  i < D/2          */
/*   v heads are copied unchanged.                                           */
/* Outputs q [T, Hq, D], k [T, Hkv, D], v [T, Hkv, D] (bf16 bits).           */
/* Returns ORC_EARG for a position outside [0, P).                           */
/* ------------------------------------------------------------------------ */

int orc_qkv_rope(const uint16_t *y, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                 const uint16_t *q_gamma, const uint16_t *k_gamma, double eps,
                 const int32_t *pos, const float *cs, int64_t P, uint16_t *q, uint16_t *k,
                 uint16_t *v)
{
    if (!y || !q_gamma || !k_gamma || !pos || !cs || !q || !k || !v || T < 0 || Hq < 0 ||
        Hkv < 0 || D <= 0 || (D % 2) != 0 || P <= 0)
        return ORC_EARG;
    const int64_t N = (Hq + 2 * Hkv) * D;
    const int64_t half = D / 2;
    for (int64_t t = 0; t < T; ++t) {
        if (pos[t] < 0 || pos[t] >= P)
            return ORC_EARG;
        const float *c = cs + (int64_t)pos[t] * D;
        const float *s = c + half;
        for (int64_t h = 0; h < Hq + 2 * Hkv; ++h) {
            const uint16_t *yh = y + t * N + h * D;
            uint16_t *dst;
            const uint16_t *g;
            if (h < Hq) {
                dst = q + (t * Hq + h) * D;
                g = q_gamma;
            } else if (h < Hq + Hkv) {
                dst = k + (t * Hkv + (h - Hq)) * D;
                g = k_gamma;
            } else {
                dst = v + (t * Hkv + (h - Hq - Hkv)) * D;
                for (int64_t i = 0; i < D; ++i)
                    dst[i] = yh[i];
                continue;
            }
            double ss = 0.0;
            for (int64_t i = 0; i < D; ++i) {
                double a = orc_bf16_value(yh[i]);
                ss += a * a;
            }
            double r = 1.0 / sqrt(ss / (double)D + eps);
            for (int64_t i = 0; i < half; ++i) {
                double z0 = orc_bf16_value(orc_bf16_rne(orc_bf16_value(yh[i]) * r *
                                                        orc_bf16_value(g[i])));
                double z1 = orc_bf16_value(orc_bf16_rne(orc_bf16_value(yh[i + half]) * r *
                                                        orc_bf16_value(g[i + half])));
                double ci = (double)c[i], si = (double)s[i];
                dst[i] = orc_bf16_rne(z0 * ci - z1 * si);
                dst[i + half] = orc_bf16_rne(z1 * ci + z0 * si);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* QuantMatMulReduceSum.  [SK14] "variant A in practice: QuantMatMulReduceSum" */
/* (and its parameter table): x1 int8 [B, M, K], x2 int8 [B, K, N] (ND),      */
/* x1_scale fp32 [B, M], x2_scale bf16 [N], out bf16 [M, N]:                  */
/*   acc_b = x1[b] @ x2[b]                  exact integers (int64 here)       */
/*   mm_b = fp32(acc_b)                     the page's cast to DT_FP32        */
/*   sc_b = fp32(x1_scale[b, m] * fp32(x2_scale[n]))   (scale product, FP32)  */
/*   scaled_b = fp32(mm_b * sc_b)                                             */
/*   out = bf16(sum_b scaled_b)             FP32 sum over the batch, b = 0..  */
/* The page fixes FP32 for every step after the integer matmul, so this one   */
/* is computed in binary32 (each step one correctly rounded operation, the    */
/* batch sum in increasing b), not binary64.  ref receives the fp32 sum.      */
/* Returns ORC_OVERFLOW if an acc leaves the int32 range (the page's INT32).  */
/* ------------------------------------------------------------------------ */

int orc_quant_matmul_reduce_sum(const int8_t *x1, const int8_t *x2, const float *x1_scale,
                                const uint16_t *x2_scale, int64_t B, int64_t M, int64_t K,
                                int64_t N, float *ref, uint16_t *out)
{
    if (!x1 || !x2 || !x1_scale || !x2_scale || !out || B <= 0 || M < 0 || K <= 0 || N <= 0)
        return ORC_EARG;
    int overflow = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : overflow)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float sum = 0.0f;
            const float ws = bf16_as_float(x2_scale[n]);
            for (int64_t b = 0; b < B; ++b) {
                int64_t acc = 0;
                const int8_t *ar = x1 + (b * M + m) * K;
                const int8_t *bc = x2 + b * K * N + n;
                for (int64_t k = 0; k < K; ++k)
                    acc += (int64_t)ar[k] * (int64_t)bc[k * N];
                if (acc > INT32_MAX || acc < INT32_MIN)
                    overflow = 1;
                const float mm = (float)(int32_t)acc;
                const float sc = x1_scale[b * M + m] * ws;
                const float scaled = mm * sc;
                sum = sum + scaled;
            }
            if (ref)
                ref[m * N + n] = sum;
            out[m * N + n] = orc_bf16_rne((double)sum);
        }
    }
    return overflow ? ORC_OVERFLOW : ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* MXFP8 mode of AT-09 / AT-11.  [AT10] sec. 4 (AT-09 quant_mode mxfp8:      */
/* y = scaled_mm(x_fp8, w_fp8, FP32, x_scale, w_scale)); [SK14] (GMM-MXFP8:  */
/* data E4M3FN, scale factors E8M0FNU, one scale per 64 elements).          */
/*                                                                          */
/* E4M3FN, written from the format: 1 sign bit, 4 exponent bits (bias 7),   */
/* 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); there is no */
/* infinity, S.1111.111 is NaN, the largest finite value is 448.            */
/* E8M0FNU: an unsigned biased exponent, value 2^(byte - 127), 255 = NaN.   */
/* ------------------------------------------------------------------------ */

double orc_e4m3_value(uint8_t c)
{
    const int sign = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0xF && m == 7)
        return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return sign ? -v : v;
}

/* Round to nearest, ties to even, saturating to the largest finite value
   (the "satfinite" conversion); NaN stays NaN. */
uint8_t orc_e4m3_rne_sat(double v)
{
    if (isnan(v))
        return 0x7F;
    const uint8_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x80 : 0;
    const double a = fabs(v);
    if (a < ldexp(1.0, -6)) { /* subnormal range: steps of 2^-9 */
        const double r = nearbyint(ldexp(a, 9));
        return sign | (uint8_t)r; /* r == 8 is the smallest normal, code 0x08 */
    }
    int E;
    frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    int k = E - 1; /* a in [2^k, 2^(k+1)) */
    double r = nearbyint(ldexp(a, 3 - k)); /* mantissa in eighths, [8, 16] */
    if (r == 16.0) {
        r = 8.0;
        k += 1;
    }
    if (k > 8 || (k == 8 && r > 14.0))
        return sign | 0x7E; /* 448 */
    return sign | (uint8_t)(((k + 7) << 3) | ((int)r - 8));
}

double orc_e8m0_value(uint8_t s)
{
    return s == 255 ? NAN : ldexp(1.0, (int)s - 127);
}

/* Per-token MXFP8 front end: the norm in binary32 exactly as
   orc_quant_rows_f32 (exact-sum rstd, y = (x * rstd) * gamma), then for each
   block of `block` elements: amax = max |y|, shared exponent
   X = floor(log2(amax)) - 8 (8 = the largest exponent of E4M3, so the block
   maximum lands in [256, 512) and saturates above 448), clamped to
   [-127, 127]; scale byte X + 127; codes = E4M3(y * 2^-X).  A block of zeros
   gets X = -127 and zero codes. */
int orc_mxfp8_quant_rows(const uint16_t *x, const uint16_t *gamma, int64_t T, int64_t K,
                         float eps, int variant, int64_t block, uint8_t *codes, uint8_t *scales)
{
    if (!x || !codes || !scales || T < 0 || K <= 0 || block <= 0 || K % block != 0 ||
        (variant != 0 && variant != 1))
        return ORC_EARG;
    const float inv_d = (float)(1.0 / (double)K);
    int status = ORC_OK;
#pragma omp parallel
    {
        float *y = (float *)malloc((size_t)K * sizeof(float));
        if (!y) {
#pragma omp atomic write
            status = ORC_ENOMEM;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < T; ++t) {
            if (!y)
                continue;
            const uint16_t *xr = x + t * K;
            double s64 = 0.0;
            float rstd;
            if (variant == 0) {
                for (int64_t k = 0; k < K; ++k) {
                    float v = bf16_as_float(xr[k]);
                    float sq = v * v;
                    s64 += (double)sq;
                }
                float s = (float)s64;
                float ms = s * inv_d;
                float var = ms + eps;
                rstd = 1.0f / sqrtf(var);
            } else {
                for (int64_t k = 0; k < K; ++k) {
                    float v = bf16_as_float(xr[k]);
                    float sq = v * v;
                    float sc = sq * inv_d;
                    s64 += (double)sc;
                }
                float s = (float)s64;
                float var = s + eps;
                float sd = sqrtf(var);
                rstd = 1.0f / sd;
            }
            for (int64_t k = 0; k < K; ++k) {
                float v = bf16_as_float(xr[k]) * rstd;
                if (gamma)
                    v = v * bf16_as_float(gamma[k]);
                y[k] = v;
            }
            for (int64_t b0 = 0; b0 < K; b0 += block) {
                float amax = 0.0f;
                for (int64_t k = b0; k < b0 + block; ++k)
                    if (fabsf(y[k]) > amax)
                        amax = fabsf(y[k]);
                int X = -127;
                if (amax > 0.0f) {
                    int E;
                    frexpf(amax, &E);
                    X = E - 1 - 8;
                    if (X < -127)
                        X = -127;
                    if (X > 127)
                        X = 127;
                }
                scales[t * (K / block) + b0 / block] = (uint8_t)(X + 127);
                for (int64_t k = b0; k < b0 + block; ++k)
                    codes[t * K + k] = orc_e4m3_rne_sat(ldexp((double)y[k], -X));
            }
        }
        free(y);
    }
    return status;
}

/* scaled_mm(x_fp8, w_fp8, FP32, x_scale, w_scale) with both operands stored
   [rows, K] (b_trans): ref = sum_k x[t,k] 2^(xs[t,k/block]-127) w[n,k]
   2^(ws[n,k/block]-127) in binary64, the FP32 result fp32(ref), and the
   output: out_dtype 0 = bf16(fp32(ref)) (the cast after scaled_mm), 1 = fp32. */
int orc_mxfp8_scaled_mm(const uint8_t *xq, const uint8_t *xs, const uint8_t *wq, const uint8_t *ws,
                        int64_t T, int64_t K, int64_t N, int64_t block, int out_dtype,
                        double *ref, void *out)
{
    if (!xq || !xs || !wq || !ws || T < 0 || K <= 0 || N <= 0 || block <= 0 || K % block != 0 ||
        (out_dtype != 0 && out_dtype != 1))
        return ORC_EARG;
    const int64_t nb = K / block;
    double *wd = (double *)malloc((size_t)N * K * sizeof(double));
    if (!wd)
        return ORC_ENOMEM;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            wd[n * K + k] = orc_e4m3_value(wq[n * K + k]) * orc_e8m0_value(ws[n * nb + k / block]);
    int status = ORC_OK;
#pragma omp parallel
    {
        double *a = (double *)malloc((size_t)K * sizeof(double));
        if (!a) {
#pragma omp atomic write
            status = ORC_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            if (!a)
                continue;
            for (int64_t k = 0; k < K; ++k)
                a[k] = orc_e4m3_value(xq[t * K + k]) * orc_e8m0_value(xs[t * nb + k / block]);
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += a[k] * wd[n * K + k];
                if (ref)
                    ref[t * N + n] = acc;
                const float f = (float)acc;
                if (out_dtype == 0)
                    ((uint16_t *)out)[t * N + n] = orc_bf16_rne((double)f);
                else
                    ((float *)out)[t * N + n] = f;
            }
        }
        free(a);
    }
    free(wd);
    return status;
}

/* ------------------------------------------------------------------------ */
/* MLA two-stage q chain.  [AT10] sec. 5 (MLAProlog) and sec. 9 (the golden  */
/* chain): q = bf16(matmul(x, wq_a)); qr = rms_norm(q) (variant B in the     */
/* page's code); qr = qr * gamma_cq (FP32); qr = bf16(qr);                   */
/* out = bf16(matmul(qr, wq_b)).  Both weights are stored [N, K] (b_trans).  */
/* qa (optional) receives the stage-1 bf16 output [T, N1].                   */
/* ------------------------------------------------------------------------ */

int orc_mla_q_chain(const uint16_t *x, const uint16_t *W_qa, const uint16_t *gamma_cq,
                    const uint16_t *W_qb, int64_t T, int64_t K, int64_t N1, int64_t N2,
                    double eps, int variant, uint16_t *qa, double *ref, uint16_t *out)
{
    if (!x || !W_qa || !gamma_cq || !W_qb || T < 0 || K <= 0 || N1 <= 0 || N2 <= 0 ||
        (variant != 0 && variant != 1))
        return ORC_EARG;
    double *wa = decode_matrix(W_qa, N1 * K);
    double *wb = decode_matrix(W_qb, N2 * N1);
    if (!wa || !wb) {
        free(wa);
        free(wb);
        return ORC_ENOMEM;
    }
    int status = ORC_OK;
#pragma omp parallel
    {
        double *xr = (double *)malloc((size_t)K * sizeof(double));
        uint16_t *q = (uint16_t *)malloc((size_t)N1 * sizeof(uint16_t));
        double *z = (double *)malloc((size_t)N1 * sizeof(double));
        if (!xr || !q || !z) {
#pragma omp atomic write
            status = ORC_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            if (!xr || !q || !z)
                continue;
            for (int64_t k = 0; k < K; ++k)
                xr[k] = orc_bf16_value(x[t * K + k]);
            /* stage 1: q_a projection, output rounded to bf16 */
            for (int64_t j = 0; j < N1; ++j) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += xr[k] * wa[j * K + k];
                q[j] = orc_bf16_rne(acc);
                if (qa)
                    qa[t * N1 + j] = q[j];
            }
            /* norm over the q_a row, times gamma_cq, cast to bf16 */
            double r = row_rstd_f64(q, N1, eps, variant);
            for (int64_t j = 0; j < N1; ++j) {
                double v = orc_bf16_value(q[j]) * r;
                v = v * orc_bf16_value(gamma_cq[j]);
                z[j] = orc_bf16_value(orc_bf16_rne(v));
            }
            /* stage 2: q_b projection */
            for (int64_t n = 0; n < N2; ++n) {
                double acc = 0.0;
                for (int64_t j = 0; j < N1; ++j)
                    acc += z[j] * wb[n * N1 + j];
                if (ref)
                    ref[t * N2 + n] = acc;
                if (out)
                    out[t * N2 + n] = orc_bf16_rne(acc);
            }
        }
        free(xr);
        free(q);
        free(z);
    }
    free(wa);
    free(wb);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Per-head RMSNorm after a projection.  [AT10] sec. 9 (the golden chain of */
/* the MLA prolog test): q_b_proj is reshaped to [num_heads, head_dim] and  */
/* normalised again, each head row on its own; the rms_norm_new helper of   */
/* that test has no gamma (an optional gamma [D] is accepted here).  Each   */
/* head row of D values of the bf16 input y [T, H*D] gets the row norm of   */
/* the chosen variant in binary64, (y * rstd) * gamma, cast to bf16.        */
/* ------------------------------------------------------------------------ */

int orc_head_rmsnorm(const uint16_t *y, int64_t T, int64_t H, int64_t D, const uint16_t *gamma,
                     double eps, int variant, uint16_t *out)
{
    if (!y || !out || T < 0 || H <= 0 || D <= 0 || (variant != 0 && variant != 1))
        return ORC_EARG;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            const uint16_t *yh = y + (t * H + h) * D;
            uint16_t *oh = out + (t * H + h) * D;
            const double r = row_rstd_f64(yh, D, eps, variant);
            for (int64_t i = 0; i < D; ++i) {
                double v = orc_bf16_value(yh[i]) * r;
                if (gamma)
                    v = v * orc_bf16_value(gamma[i]);
                oh[i] = orc_bf16_rne(v);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* W8A8 front end: AT-03 RMSNorm then AT-05 per-token symmetric INT8 quant,  */
/* in binary32, the pages' order.  [AT10] sec. 3 (norm steps), sec. 4       */
/* (AT-05: amax = max|y|, multiplier 127/amax, rounding + saturating casts), */
/* [SK03] AT-11 section (common.py quant: dequant scale = max|x| / 127).     */
/*                                                                           */
/*   x32 = float(x); terms x32*x32 (variant A) or (x32*x32)*(1/D) (B), each */
/*   a binary32 product; s = the binary32 value of their sum (see below);    */
/*   A: ms = s*(1/D); rstd = 1/sqrt(ms+eps)     B: rstd = 1/sqrt(s+eps)      */
/*   y = (x32*rstd)*float(gamma); amax = max|y|; qs = 127/amax;              */
/*   q = clamp(rint_half_even(y*qs), -127, 127); x_scale = amax/127.         */
/* An all-zero row (amax == 0) gives q = 0 and x_scale = 0 (the pages are    */
/* silent; no division by zero is performed).                                */
/* The pages fix FP32 but not the order of the K-term sum.  Reading: s is    */
/* the binary32 rounding of the exact sum of the binary32 terms.  The terms  */
/* are summed in binary64, exact for bf16 data (squares carry 16 bits) of    */
/* any realistic range, then rounded once; every later step is a single      */
/* correctly rounded binary32 operation, so the integer codes are a         */
/* function of the input alone, not of a summation order.                   */
/* ------------------------------------------------------------------------ */

int orc_quant_rows_f32(const uint16_t *x, const uint16_t *gamma, int64_t T, int64_t K,
                       float eps, int variant, int8_t *q, float *x_scale, float *rstd_out,
                       float *qv_out)
{
    if (!x || !q || !x_scale || T < 0 || K <= 0 || (variant != 0 && variant != 1))
        return ORC_EARG;
    const float inv_d = (float)(1.0 / (double)K);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *xr = x + t * K;
        double s64 = 0.0;
        float rstd;
        if (variant == 0) {
            for (int64_t k = 0; k < K; ++k) {
                float v = bf16_as_float(xr[k]);
                float sq = v * v;
                s64 += (double)sq;
            }
            float s = (float)s64;
            float ms = s * inv_d;
            float var = ms + eps;
            rstd = 1.0f / sqrtf(var);
        } else {
            for (int64_t k = 0; k < K; ++k) {
                float v = bf16_as_float(xr[k]);
                float sq = v * v;
                float sc = sq * inv_d;
                s64 += (double)sc;
            }
            float s = (float)s64;
            float var = s + eps;
            float sd = sqrtf(var);
            rstd = 1.0f / sd;
        }
        if (rstd_out)
            rstd_out[t] = rstd;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float y = bf16_as_float(xr[k]) * rstd;
            if (gamma)
                y = y * bf16_as_float(gamma[k]);
            float m = fabsf(y);
            if (m > amax)
                amax = m;
        }
        int8_t *qr = q + t * K;
        if (amax == 0.0f) {
            for (int64_t k = 0; k < K; ++k) {
                qr[k] = 0;
                if (qv_out)
                    qv_out[t * K + k] = 0.0f;
            }
            x_scale[t] = 0.0f;
            continue;
        }
        float qs = 127.0f / amax;
        for (int64_t k = 0; k < K; ++k) {
            float y = bf16_as_float(xr[k]) * rstd;
            if (gamma)
                y = y * bf16_as_float(gamma[k]);
            float v = y * qs;
            if (qv_out)
                qv_out[t * K + k] = v;
            float r = rintf(v); /* default rounding mode: nearest, ties to even */
            if (r > 127.0f)
                r = 127.0f;
            if (r < -127.0f)
                r = -127.0f;
            qr[k] = (int8_t)r;
        }
        x_scale[t] = amax / 127.0f;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* AT-09 INT8 W8A8 matmul: C[m,n] = sum_k A[m,k] * B[n,k] (B stored [N, K]), */
/* exact, accumulated in int64.  [AT10] sec. 4 (matmul(x_int8, w_int8,       */
/* dtype=INT32)).  Returns ORC_OVERFLOW if any sum leaves the int32 range    */
/* (C then holds the low 32 bits' two's-complement wrap, never relied on).  */
/* ------------------------------------------------------------------------ */

int orc_gemm_s8(const int8_t *A, const int8_t *B, int64_t M, int64_t N, int64_t K, int32_t *C)
{
    if (!A || !B || !C || M < 0 || N <= 0 || K <= 0)
        return ORC_EARG;
    int overflow = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : overflow)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t acc = 0;
            for (int64_t k = 0; k < K; ++k)
                acc += (int64_t)A[m * K + k] * (int64_t)B[n * K + k];
            if (acc > INT32_MAX || acc < INT32_MIN)
                overflow = 1;
            C[m * N + n] = (int32_t)(uint32_t)(uint64_t)acc;
        }
    }
    return overflow ? ORC_OVERFLOW : ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* AT-06 dequant, [SK14] QuantMatMulReduceSum: cast the int32 product to     */
/* float, form the scale product x_scale[m] * w_scale[n] first, multiply,    */
/* cast to bf16.  Binary64 here; ref receives the value before rounding.     */
/* ------------------------------------------------------------------------ */

int orc_dequant_bf16(const int32_t *acc, const float *x_scale, const float *w_scale,
                     int64_t M, int64_t N, double *ref, uint16_t *out)
{
    if (!acc || !x_scale || !w_scale || M < 0 || N <= 0)
        return ORC_EARG;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double scale = (double)x_scale[m] * (double)w_scale[n];
            double v = (double)acc[m * N + n] * scale;
            if (ref)
                ref[m * N + n] = v;
            if (out)
                out[m * N + n] = orc_bf16_rne(v);
        }
    }
    return ORC_OK;
}

/* AT-11 RMSNorm + Linear + Quant, composed from the three steps above. */
int orc_rmsnorm_linear_w8a8(const uint16_t *x, const uint16_t *gamma, const int8_t *Wq,
                            const float *w_scale, int64_t T, int64_t K, int64_t N, float eps,
                            int variant, int8_t *q, float *x_scale, int32_t *acc, double *ref,
                            uint16_t *out)
{
    if (!q || !x_scale || !acc)
        return ORC_EARG;
    int st = orc_quant_rows_f32(x, gamma, T, K, eps, variant, q, x_scale, NULL, NULL);
    if (st != ORC_OK)
        return st;
    int ovf = orc_gemm_s8(q, Wq, T, N, K, acc);
    if (ovf < 0)
        return ovf;
    st = orc_dequant_bf16(acc, x_scale, w_scale, T, N, ref, out);
    return st != ORC_OK ? st : ovf;
}
