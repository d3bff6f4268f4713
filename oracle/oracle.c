/*
 * CPU oracle for the small-M skinny GEMM and its two epilogues.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plain, single-threaded
 * statement of what the GPU path must compute. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product library
 * never does, and the two share no source, header, table or helper.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no threads, no
 * SIMD intrinsics, no FMA contraction, so x86-64 and aarch64 agree bit for bit).
 *
 * Sources (vLLM API pages of the "Muse Spark specialized decode" package),
 * restated:
 *   [unpooler]  cutedsl/gemm/unpooler, module docstring: the column block of a
 *               small-M product, out[m, n] = sum over k of x[m, k] * W[n, k], with
 *               BF16 operands and output, FP32 accumulation and 1 <= m <= 16; a
 *               negative zero is published as positive zero.
 *   [pooler]    cutedsl/moe/pooler_gather, module docstring: the pre-expert norm
 *               scales each row by the reciprocal RMS (eps under the root) and by
 *               (norm weight + gain_center), rounds to BF16, then quantizes to
 *               NVFP4 in blocks of 16 under one global scale: two e2m1 codes per
 *               byte, even column in the low nibble, and one float8_e4m3fn scale
 *               per block in plain row-major order. Helpers on the same page:
 *               cvt_e2m1x8_f32 and cvt_f32_to_e4m3 (round-to-nearest, saturate to
 *               the largest finite value) and nvfp4_compute_output_scale (the
 *               element multiplier is the reciprocal of sf / global_scale, and 0
 *               when sf is 0; sf is widened to FP32 exactly).
 *   [batt]      cutedsl/oproj/batt, AttentionBoundary: the BF16 o_proj partial is
 *               normalised (post_attn_norm), added with gates into the FP32
 *               residual stream in place, and the stream is normalised again
 *               (pre_ffn_norm) into a BF16 output.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - GEMM: the sum is taken in FP64 in k order; each BF16 x BF16 product is
 *     exact in FP64. One rounding, FP64 -> BF16, ties to even, no detour
 *     through FP32.
 *   - RMSNorm: mean over the full row, eps inside the square root, the weight
 *     widened from BF16 and added to gain_center in FP64 (not rounded to BF16),
 *     one rounding to BF16 at the end.
 *   - NVFP4 block scale: sf = e4m3_rn_satfinite((amax / 6) * gs), two FP32 ops in
 *     that order; the pages print only the inverse step.
 *   - NVFP4 output scale: the pages' approximate reciprocal is replaced by IEEE
 *     FP32 division, os = 1 / (float(sf) * (1 / gs)), three FP32 ops in that order.
 *   - Every NVFP4 decision is taken in FP32, the precision the pages' helpers
 *     use; everything else is FP64 with one final rounding per stored value.
 *   - e2m1 of a negative value that rounds to zero keeps its sign (code 0x8),
 *     as IEEE rounding does.
 *   - Dual norm: the post-norm output q stays in FP64 (it is never stored), the
 *     updated stream is rounded to FP32 once, and the pre-FFN norm reads that
 *     stored FP32 value.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Codecs.                                                                   */
/* ------------------------------------------------------------------------- */

/* Round a non-negative finite |v| to the grid of a binary format with
   `mant_bits` fraction bits whose smallest normal exponent is `emin`:
   the spacing in [2^e, 2^(e+1)) is 2^(e - mant_bits), and below 2^emin the
   spacing stays 2^(emin - mant_bits) (subnormals). Ties go to the even
   multiple of the spacing, which is the value with an even last fraction bit.
   Scaling by a power of two is exact in FP64, so the only rounding is rint(). */
static double round_to_grid(double a, int mant_bits, int emin)
{
    if (a == 0.0)
        return 0.0;
    int e2;
    frexp(a, &e2);         /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;        /* a in [2^e, 2^(e+1)) */
    if (e < emin)
        e = emin;
    double quantum = ldexp(1.0, e - mant_bits);
    double q = a / quantum;                     /* exact */
    return rint(q) * quantum;                   /* rint: ties to even */
}

/* BF16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
uint16_t oracle_bf16_from_double(double v)
{
    if (v != v)
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    double r = round_to_grid(a, 7, -126);
    /* The largest finite BF16 is (2 - 2^-7) * 2^127; rounding up past it is
       an overflow to infinity, which the FP32 conversion below produces. */
    float f = (float)r;    /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u >> 16) | sign);
}

double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Stored BF16 outputs never carry -0.0 ([unpooler] zero-copy epilogue and
   [pooler] edge layers: publishers store -0.0 as +0.0). */
static uint16_t bf16_store(double v)
{
    uint16_t b = oracle_bf16_from_double(v);
    return b == 0x8000 ? 0 : b;
}

/* float8_e4m3fn: 1 sign, 4 exponent (bias 7), 3 fraction bits, no infinity,
   S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
   Smallest normal 2^-6, subnormal spacing 2^-9.
   .rn.satfinite: round to nearest even, then clamp finite overflow to +-448. */
uint8_t oracle_e4m3_from_float(float v)
{
    if (v != v)
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    double r = round_to_grid(a, 3, -6);
    if (r > 448.0)
        r = 448.0;
    if (r == 0.0)
        return sign;
    uint8_t bits;
    if (r < ldexp(1.0, -6)) {
        bits = (uint8_t)(r / ldexp(1.0, -9));          /* subnormal: 0.mmm * 2^-6 */
    } else {
        int e2;
        double f = frexp(r, &e2);                       /* r = f * 2^e2 */
        int e = e2 - 1;                                 /* r = (2f) * 2^e, 2f in [1,2) */
        int mant = (int)((2.0 * f - 1.0) * 8.0);        /* exact */
        bits = (uint8_t)(((e + 7) << 3) | mant);
    }
    return (uint8_t)(sign | bits);
}

float oracle_e4m3_to_float(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
    if (e == 0xF && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (float)(s ? -mag : mag);
}

/* e2m1 (FP4): 1 sign, 2 exponent (bias 1), 1 fraction bit; magnitudes
   {0, 0.5, 1, 1.5, 2, 3, 4, 6} are codes 0..7, the sign is bit 3.
   .rn.satfinite: ties to the even code, finite overflow to +-6. */
uint8_t oracle_e2m1_from_float(float v)
{
    if (v != v)
        return 0x7;   /* no NaN in e2m1; out of contract */
    uint8_t sign = signbit(v) ? 0x8 : 0;
    double a = fabs((double)v);
    double r = round_to_grid(a, 1, 0);
    if (r > 6.0)
        r = 6.0;
    uint8_t code;
    if (r < 1.0) {
        code = (uint8_t)(r / 0.5);                      /* 0 or 1 (0.5) */
    } else {
        int e2;
        double f = frexp(r, &e2);
        int e = e2 - 1;
        int mant = (int)((2.0 * f - 1.0) * 2.0);
        code = (uint8_t)(((e + 1) << 1) | mant);
    }
    return (uint8_t)(sign | code);
}

float oracle_e2m1_to_float(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + m / 2.0, e - 1);
    return (float)(s ? -mag : mag);
}

/* ------------------------------------------------------------------------- */
/* GEMM ([unpooler] module docstring; [pooler] compile_pooler_gemm).         */
/* ------------------------------------------------------------------------- */

/* acc[m,n] = sum_k x[m,k] * w[n,k] in FP64, k ascending; absacc[m,n] =
   sum_k |x[m,k] * w[n,k]| (the scale of the summation error bound).
   Either output may be NULL. x is [m,k] BF16 bits, w is [n,k] BF16 bits. */
void oracle_gemm_f64(const uint16_t *x, const uint16_t *w, double *acc,
                     double *absacc, int m, int n, int k)
{
    for (int i = 0; i < m; ++i) {
        for (int j = 0; j < n; ++j) {
            const uint16_t *xr = x + (size_t)i * k;
            const uint16_t *wr = w + (size_t)j * k;
            double s = 0.0, sa = 0.0;
            for (int t = 0; t < k; ++t) {
                double p = oracle_bf16_to_double(xr[t]) * oracle_bf16_to_double(wr[t]);
                s += p;
                sa += fabs(p);
            }
            if (acc)
                acc[(size_t)i * n + j] = s;
            if (absacc)
                absacc[(size_t)i * n + j] = sa;
        }
    }
}

/* y[m,n] = bf16_rn(sum_k x[m,k] * w[n,k]), -0.0 stored as +0.0. */
void oracle_gemm_bf16(const uint16_t *x, const uint16_t *w, uint16_t *y, int m,
                      int n, int k)
{
    for (int i = 0; i < m; ++i) {
        for (int j = 0; j < n; ++j) {
            const uint16_t *xr = x + (size_t)i * k;
            const uint16_t *wr = w + (size_t)j * k;
            double s = 0.0;
            for (int t = 0; t < k; ++t)
                s += oracle_bf16_to_double(xr[t]) * oracle_bf16_to_double(wr[t]);
            y[(size_t)i * n + j] = bf16_store(s);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Pre-expert RMSNorm ([pooler] module docstring, PoolerLayer, pooler_layer: */
/* the weight is applied after the norm).                                    */
/* ------------------------------------------------------------------------- */

/* z[m,j] = bf16(y[m,j] * r[m] * (w[j] + gc)), r[m] = 1/sqrt(sum_j y^2 / n + eps).
   rinv (may be NULL) receives r[m]. */
void oracle_rmsnorm_bf16(const uint16_t *y, const uint16_t *w, double eps,
                         double gc, uint16_t *z, double *rinv, int m, int n)
{
    for (int i = 0; i < m; ++i) {
        const uint16_t *yr = y + (size_t)i * n;
        double ss = 0.0;
        for (int j = 0; j < n; ++j) {
            double v = oracle_bf16_to_double(yr[j]);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / n + eps);
        if (rinv)
            rinv[i] = r;
        for (int j = 0; j < n; ++j) {
            double g = oracle_bf16_to_double(w[j]) + gc;
            z[(size_t)i * n + j] = bf16_store(oracle_bf16_to_double(yr[j]) * r * g);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* NVFP4 quantization ([pooler] module docstring; cvt_e2m1x8_f32,            */
/* cvt_f32_to_e4m3, nvfp4_compute_output_scale). All steps in FP32.          */
/* ------------------------------------------------------------------------- */

/* One 16-element block: returns the e4m3 scale byte, writes 16 e2m1 codes. */
static uint8_t nvfp4_block(const uint16_t *z, float gs, uint8_t codes[16])
{
    float amax = 0.0f;
    for (int j = 0; j < 16; ++j) {
        float v = fabsf(bf16_to_float(z[j]));
        if (v > amax)
            amax = v;
    }
    float t = amax / 6.0f;
    t = t * gs;
    uint8_t sf = oracle_e4m3_from_float(t);
    float sff = oracle_e4m3_to_float(sf);          /* exact widening */
    float os;
    if (sff == 0.0f) {
        os = 0.0f;
    } else {
        float rgs = 1.0f / gs;
        float prod = sff * rgs;
        os = 1.0f / prod;
    }
    for (int j = 0; j < 16; ++j) {
        float v = bf16_to_float(z[j]) * os;
        codes[j] = oracle_e2m1_from_float(v);
    }
    return sf;
}

/* z [m,n] BF16 -> a [m,n/2] (code of column 2i in the low nibble, 2i+1 in the
   high nibble) and a_sf [m,n/16] (e4m3fn bytes, row-major, not swizzled).
   n must be a multiple of 16. */
void oracle_nvfp4_quantize(const uint16_t *z, float gs, uint8_t *a, uint8_t *a_sf,
                           int m, int n)
{
    for (int i = 0; i < m; ++i) {
        for (int b = 0; b < n / 16; ++b) {
            uint8_t codes[16];
            a_sf[(size_t)i * (n / 16) + b] = nvfp4_block(z + (size_t)i * n + 16 * b, gs, codes);
            for (int p = 0; p < 8; ++p)
                a[(size_t)i * (n / 2) + 8 * b + p] =
                    (uint8_t)((codes[2 * p] & 0xF) | ((codes[2 * p + 1] & 0xF) << 4));
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Attention-boundary dual norm ([batt] AttentionBoundary).                  */
/* ------------------------------------------------------------------------- */

/* For each row: r1 = 1/sqrt(mean(p^2) + eps_post);
   q = p * r1 * (w1 + gc_post)   (q = p * r1 when w1 is NULL);
   s <- float(alpha * s + beta * q)            (in place, FP32 storage);
   r2 = 1/sqrt(mean(s^2) + eps_pre) over the stored FP32 s;
   out = bf16(s * r2 * (w2 + gc_pre)), -0.0 stored as +0.0.
   r1_out / r2_out (may be NULL) receive r1 and r2 per row. */
void oracle_dual_norm(const uint16_t *p, float *s, const uint16_t *w1, double alpha,
                      const uint16_t *beta, const uint16_t *w2, uint16_t *out,
                      double eps_post, double eps_pre, double gc_post, double gc_pre,
                      double *r1_out, double *r2_out, int m, int h)
{
    for (int i = 0; i < m; ++i) {
        const uint16_t *pr = p + (size_t)i * h;
        float *sr = s + (size_t)i * h;
        double ss = 0.0;
        for (int j = 0; j < h; ++j) {
            double v = oracle_bf16_to_double(pr[j]);
            ss += v * v;
        }
        double r1 = 1.0 / sqrt(ss / h + eps_post);
        for (int j = 0; j < h; ++j) {
            double g = w1 ? oracle_bf16_to_double(w1[j]) + gc_post : 1.0;
            double q = oracle_bf16_to_double(pr[j]) * r1 * g;
            double sn = alpha * (double)sr[j] + oracle_bf16_to_double(beta[j]) * q;
            sr[j] = (float)sn;
        }
        double ss2 = 0.0;
        for (int j = 0; j < h; ++j)
            ss2 += (double)sr[j] * (double)sr[j];
        double r2 = 1.0 / sqrt(ss2 / h + eps_pre);
        for (int j = 0; j < h; ++j) {
            double g = oracle_bf16_to_double(w2[j]) + gc_pre;
            out[(size_t)i * h + j] = bf16_store((double)sr[j] * r2 * g);
        }
        if (r1_out)
            r1_out[i] = r1;
        if (r2_out)
            r2_out[i] = r2;
    }
}

/* ------------------------------------------------------------------------- */
/* Weight-only NVFP4 GEMM. Not on the pages: the weight W [n, k] is held in  */
/* the NVFP4 byte layout the pooler page's module docstring gives for the    */
/* experts' input, applied to the rows of W along K: two e2m1 codes per byte */
/* (column 2c in the low nibble), one float8_e4m3fn scale per 16 consecutive */
/* columns of a row, and one FP32 dequantization multiplier w_scale for the  */
/* whole tensor (the reciprocal of the global scale the codes were made      */
/* with). Readings (also in the design notes): a weight element is           */
/* e2m1(code) * e4m3(scale), exact in FP64; w_scale multiplies the finished  */
/* sum once per output, as a per-tensor factor commutes with the sum.        */
/* ------------------------------------------------------------------------- */

/* dq[n, k] = e2m1 value of the code of W[n, k] times the e4m3 value of its
   block scale (exact). wq is [n, k/2] bytes, wsf is [n, k/16] bytes. */
void oracle_nvfp4_dequant(const uint8_t *wq, const uint8_t *wsf, double *dq, int n, int k)
{
    for (int r = 0; r < n; ++r) {
        for (int j = 0; j < k; ++j) {
            uint8_t byte = wq[(size_t)r * (k / 2) + j / 2];
            uint8_t code = (j % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            double sf = (double)oracle_e4m3_to_float(wsf[(size_t)r * (k / 16) + j / 16]);
            dq[(size_t)r * k + j] = (double)oracle_e2m1_to_float(code) * sf;
        }
    }
}

/* y[m, n] = bf16_rn(w_scale * sum_k x[m, k] * dq[n, k]), -0.0 stored as +0.0.
   The sum is taken in FP64 in k order, multiplied by w_scale in FP64 and
   rounded once to BF16. acc (may be NULL) receives w_scale * sum, absacc (may
   be NULL) |w_scale| * sum_k |x * dq| (the scale of the summation error). */
void oracle_gemm_nvfp4w(const uint16_t *x, const uint8_t *wq, const uint8_t *wsf,
                        float w_scale, uint16_t *y, double *acc, double *absacc,
                        int m, int n, int k)
{
    double *dq = (double *)malloc(sizeof(double) * (size_t)n * k);
    if (!dq)
        return;
    oracle_nvfp4_dequant(wq, wsf, dq, n, k);
    for (int i = 0; i < m; ++i) {
        for (int r = 0; r < n; ++r) {
            const uint16_t *xr = x + (size_t)i * k;
            const double *wr = dq + (size_t)r * k;
            double s = 0.0, sa = 0.0;
            for (int t = 0; t < k; ++t) {
                double p = oracle_bf16_to_double(xr[t]) * wr[t];
                s += p;
                sa += fabs(p);
            }
            double v = (double)w_scale * s;
            if (y)
                y[(size_t)i * n + r] = bf16_store(v);
            if (acc)
                acc[(size_t)i * n + r] = v;
            if (absacc)
                absacc[(size_t)i * n + r] = fabs((double)w_scale) * sa;
        }
    }
    free(dq);
}
