/*
 * nvfp4_oracle.c -- CPU oracle for NVFP4 weight-only (W4A16) projection.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This file is a plain, slow,
 * deliberately unoptimised restatement of what the GPU library computes.
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline may load it.  It shares no code, header, table or constant
 * generator with the CUDA library; the two never include or link each other.
 *
 * Sources followed (pages of the serving engine's API docs):
 *   - "spark_model/layers/mtp_head/new.rs", MtpHead::new: projections are
 *     quantised once at load time by a global-absmax pass followed by a
 *     BF16->NVFP4 quantise pass; the LM head holds 0.5 byte per weight.
 *   - "spark_model/layers/qwen3_attention/prefill_weights.rs",
 *     predequant setup: the packed weight layout is [N, K/2].
 *   - same page, w4a16_gemm_m128_dispatch: the lossless prefill GEMM is an
 *     exact FP4->BF16 dequantisation followed by a BF16 matrix product.
 *   - "spark_model/layers/deepseek_v4_mtp.rs", argmax_grammar_masked: greedy
 *     argmax is a strict '>' scan in ascending index starting from -inf, so
 *     the lowest index wins ties, NaN never wins, and 0 is returned when no
 *     value beats -inf.
 *   - same page, constructor: the draft's RMSNorm applies its weight as
 *     stored ("vanilla"), not 1 + w.
 *   - "metrale_model_layers/layers/mtp_head.rs", module doc: the draft step
 *     is pre-fc norms, concat, fc, ..., final norm, NVFP4 LM head, argmax.
 * The number format itself (E2M1 codes with the codebook
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}, one E4M3 scale per 16-element K block, an
 * FP32 global scale equal to absmax / (6 * 448)) is not defined on those
 * pages; it is taken from the project's problem statement and the public
 * OCP microscaling / NVFP4 format description.
 *
 * Readings taken where the pages are silent:
 *   - quantiser arithmetic is this fixed sequence of binary32 operations:
 *       g   = fl32(amax / 2688)
 *       t_b = fl32(amax_b / fl32(6 * g));   s_b = E4M3_RNE_SATFINITE(t_b)
 *       d_b = fl32(dec(s_b) * g)
 *       c_i = E2M1_RNE_SATFINITE(fl32(x_i / d_b)), sign bit = sign of x_i
 *     with s_b = 0 when g == 0 or amax_b == 0, and c_i = +0 when d_b == 0;
 *   - packing: element 2j in the low nibble of byte j, 2j+1 in the high one;
 *   - scales: plain row-major [N, K/16];
 *   - the RMSNorm output is rounded to BF16 before the dot product;
 *   - the global scale multiplies the finished dot product.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (see oracle/build.py).
 * Floating point: every binary32 step above is one correctly rounded C float
 * operation (FLT_EVAL_METHOD 0 on x86-64 and aarch64, contraction off);
 * dot products accumulate in binary64.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE 2
#define ORACLE_ERR_NONFINITE 7

/* ---------------------------------------------------------------- format */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent 0 is subnormal: value = m * 0.5.  No infinities, no NaN. */
double oracle_e2m1_value(int code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (the "FN" variant): sign bit 7, exponent bits 6..3 (bias 7),
 * mantissa bits 2..0.  Exponent 0 is subnormal: value = m/8 * 2^-6.
 * No infinities; S.1111.111 is NaN.  Largest finite value 448. */
double oracle_e4m3_value(int byte)
{
    int s = (byte >> 7) & 1;
    int e = (byte >> 3) & 15;
    int m = byte & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest non-negative finite E4M3 value to t (t >= 0), found by trying
 * every finite code: ties go to the code whose mantissa LSB (bit 0) is 0,
 * values beyond the range land on the largest finite code 0x7E (448).
 * Returns -1 for a negative or NaN argument. */
int oracle_e4m3_encode(float t)
{
    if (!(t >= 0.0f))
        return -1;
    if (t >= 448.0f)
        return 0x7E; /* saturate (distances to huge t are not resolvable) */
    int best = 0;
    double bestd = fabs((double)t);
    for (int b = 1; b <= 0x7E; ++b) {
        double d = fabs((double)t - oracle_e4m3_value(b));
        if (d < bestd || (d == bestd && (b & 1) == 0 && (best & 1) == 1)) {
            best = b;
            bestd = d;
        }
    }
    return best;
}

/* Nearest E2M1 magnitude to |q| among the eight codebook entries, ties to
 * the even code, |q| beyond 6 saturating to 6; the sign bit is the sign
 * bit of q (so a negative q that rounds to zero gives code 0x8). */
int oracle_e2m1_encode(float q)
{
    double a = fabs((double)q);
    if (a >= 6.0)
        return 7 | (signbit(q) ? 8 : 0); /* saturate */
    int best = 0;
    double bestd = a;
    for (int c = 1; c <= 7; ++c) {
        double d = fabs(a - oracle_e2m1_value(c));
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return best | (signbit(q) ? 8 : 0);
}

/* ------------------------------------------------------------ BF16 helpers */

float oracle_bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a binary64 value to the nearest BF16 (8 significant bits, exponent
 * range of binary32, subnormals down to 2^-133), ties to even.  The rounding
 * is done once, directly from binary64, by scaling to an integer multiple of
 * the BF16 quantum and calling rint (round-half-even in the default mode). */
uint16_t oracle_bf16_from_double(double v)
{
    uint32_t u;
    float f;
    if (isnan(v)) {
        return 0x7FC0;
    }
    if (v == 0.0 || isinf(v)) {
        f = (float)v;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16);
    }
    int e;
    frexp(fabs(v), &e); /* |v| in [2^(e-1), 2^e) */
    int qexp = (e - 1) - 7; /* quantum of an 8-bit significand */
    if (qexp < -133)
        qexp = -133; /* BF16 subnormal quantum */
    double r = ldexp(rint(ldexp(v, -qexp)), qexp);
    if (fabs(r) >= ldexp(1.0, 128))
        r = v > 0 ? INFINITY : -INFINITY;
    f = (float)r; /* exact: r has at most 8 significant bits */
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------- quantiser */

/* Global absmax: the largest |w| over all count BF16 values.
 * Returns ORACLE_ERR_NONFINITE if any value is Inf or NaN. */
int oracle_global_absmax(const uint16_t *w, int64_t count, float *amax_out)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < count; ++i) {
        float x = oracle_bf16_to_float(w[i]);
        if (!isfinite(x))
            return ORACLE_ERR_NONFINITE;
        float ax = fabsf(x);
        if (ax > amax)
            amax = ax;
    }
    *amax_out = amax;
    return ORACLE_OK;
}

/* Global scale g = fl32(amax / (6 * 448)). */
float oracle_global_scale(float amax)
{
    return amax / 2688.0f;
}

/* Quantise rows [row0, row0 + nrows) of a BF16 matrix w[n, k] (row stride k)
 * with a given global scale g.  packed receives nrows * k/2 bytes, scales
 * nrows * k/16 bytes, both row-major starting at row0's row. */
int oracle_quantize_rows(const uint16_t *w, int64_t k, int64_t row0, int64_t nrows,
                         float g, uint8_t *packed, uint8_t *scales)
{
    if (k <= 0 || k % 16 != 0 || nrows < 0)
        return ORACLE_ERR_SHAPE;
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t *row = w + (row0 + r) * k;
        for (int64_t b = 0; b < k / 16; ++b) {
            float x[16];
            float amax_b = 0.0f;
            for (int i = 0; i < 16; ++i) {
                x[i] = oracle_bf16_to_float(row[b * 16 + i]);
                if (!isfinite(x[i]))
                    return ORACLE_ERR_NONFINITE;
                if (fabsf(x[i]) > amax_b)
                    amax_b = fabsf(x[i]);
            }
            int s = 0;
            if (g != 0.0f && amax_b != 0.0f) {
                float six_g = 6.0f * g;
                float t = amax_b / six_g;
                s = oracle_e4m3_encode(t);
            }
            scales[r * (k / 16) + b] = (uint8_t)s;
            float d = (float)oracle_e4m3_value(s) * g;
            int codes[16];
            for (int i = 0; i < 16; ++i) {
                if (d == 0.0f) {
                    codes[i] = 0;
                } else {
                    float q = x[i] / d;
                    codes[i] = oracle_e2m1_encode(q);
                }
            }
            for (int j = 0; j < 8; ++j)
                packed[r * (k / 2) + b * 8 + j] =
                    (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
        }
    }
    return ORACLE_OK;
}

/* Full load-time quantisation of w[n, k]: global absmax, global scale, then
 * every block.  Writes amax and g. */
int oracle_quantize(const uint16_t *w, int64_t n, int64_t k, uint8_t *packed,
                    uint8_t *scales, float *g_out, float *amax_out)
{
    if (n < 0 || k <= 0 || k % 16 != 0)
        return ORACLE_ERR_SHAPE;
    float amax;
    int rc = oracle_global_absmax(w, n * k, &amax);
    if (rc != ORACLE_OK)
        return rc;
    float g = oracle_global_scale(amax);
    *amax_out = amax;
    *g_out = g;
    return oracle_quantize_rows(w, k, 0, n, g, packed, scales);
}

/* One dequantised weight: g * dec(s_b) * e2m1(c_i), exact in binary64. */
static double dequant_one(const uint8_t *packed, const uint8_t *scales, float g,
                          int64_t k, int64_t row, int64_t i)
{
    uint8_t byte = packed[row * (k / 2) + i / 2];
    int code = (i & 1) ? (byte >> 4) : (byte & 15);
    int s = scales[row * (k / 16) + i / 16];
    return (double)g * oracle_e4m3_value(s) * oracle_e2m1_value(code);
}

/* Dense dequantisation of rows [row0, row0 + nrows) into out[nrows, k]. */
void oracle_dequant_rows(const uint8_t *packed, const uint8_t *scales, float g,
                         int64_t k, int64_t row0, int64_t nrows, double *out)
{
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t i = 0; i < k; ++i)
            out[r * k + i] = dequant_one(packed, scales, g, k, row0 + r, i);
}

/* ---------------------------------------------------------------- RMSNorm */

/* RMSNorm of one segment row x[ks] with weight gamma applied as stored:
 * r = 1 / sqrt(sum(x^2)/ks + eps) in binary64, a_i = bf16(x_i * r * gamma_i).
 * With gamma == NULL the segment is copied unchanged (no norm). */
void oracle_rmsnorm_row(const uint16_t *x, int64_t ks, const uint16_t *gamma,
                        float eps, uint16_t *out)
{
    if (gamma == NULL) {
        memcpy(out, x, (size_t)ks * 2);
        return;
    }
    double ss = 0.0;
    for (int64_t i = 0; i < ks; ++i) {
        double v = oracle_bf16_to_float(x[i]);
        ss += v * v;
    }
    double r = 1.0 / sqrt(ss / (double)ks + (double)eps);
    for (int64_t i = 0; i < ks; ++i) {
        double v = (double)oracle_bf16_to_float(x[i]) * r *
                   (double)oracle_bf16_to_float(gamma[i]);
        out[i] = oracle_bf16_from_double(v);
    }
}

/* ------------------------------------------------------------------- GEMV */

/* y[m, n] = sum_i a[m, i] * w[n, i] over the dequantised weight, binary64,
 * and sabs[m, n] = sum_i |a[m, i] * w[n, i]| (the error-bound scale).
 * a is BF16 [m, k] with row stride lda.  Rows [n0, n0 + nn) of the weight
 * are evaluated; y and sabs are [m, nn]. */
void oracle_gemv_rows(const uint16_t *a, int64_t m, int64_t lda,
                      const uint8_t *packed, const uint8_t *scales, float g,
                      int64_t k, int64_t n0, int64_t nn, double *y, double *sabs)
{
    for (int64_t r = 0; r < m; ++r) {
        for (int64_t j = 0; j < nn; ++j) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t i = 0; i < k; ++i) {
                double p = (double)oracle_bf16_to_float(a[r * lda + i]) *
                           dequant_one(packed, scales, g, k, n0 + j, i);
                acc += p;
                aacc += fabs(p);
            }
            y[r * nn + j] = acc;
            sabs[r * nn + j] = aacc;
        }
    }
}

/* Greedy argmax as the draft proposer scans it: start from -inf at index 0,
 * take index i only when y[i] > best (strictly), ascending.  Lowest index
 * wins ties, NaN never wins, and 0 comes back when nothing beats -inf. */
int64_t oracle_argmax(const double *y, int64_t n)
{
    int64_t best = 0;
    double bestv = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        if (y[i] > bestv) {
            bestv = y[i];
            best = i;
        }
    }
    return best;
}

/* ------------------------------------------------------------------- GEMM */

/* Selected outputs of C = A * Wdeq^T: for each of the count (row, col)
 * pairs, exact[p] = sum_k A[row, k] * w[col, k] in binary64 and
 * sabs[p] = sum_k |A[row, k] * w[col, k]|.  The caller rounds to BF16. */
void oracle_gemm_pairs(const uint16_t *A, int64_t lda, const uint8_t *packed,
                       const uint8_t *scales, float g, int64_t k,
                       const int64_t *rows, const int64_t *cols, int64_t count,
                       double *exact, double *sabs)
{
    for (int64_t p = 0; p < count; ++p) {
        double acc = 0.0, aacc = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            double v = (double)oracle_bf16_to_float(A[rows[p] * lda + i]) *
                       dequant_one(packed, scales, g, k, cols[p], i);
            acc += v;
            aacc += fabs(v);
        }
        exact[p] = acc;
        sabs[p] = aacc;
    }
}

/* ------------------------------------------------- masked argmax, log-prob */

/* Grammar-masked greedy argmax ("spark_model/layers/deepseek_v4_mtp.rs",
 * argmax_grammar_masked): token i takes part only when bit i%32 of word i/32
 * of the mask is set (words past nwords disallow); among those, the strict '>'
 * ascending scan from -inf.  Returns 0 when no token is allowed.  mask may be
 * NULL (every token allowed). */
int64_t oracle_argmax_masked(const double *y, int64_t n, const int32_t *mask, int64_t nwords)
{
    int64_t best = 0;
    double bestv = -INFINITY;
    int any = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (mask != NULL) {
            int64_t word = i / 32;
            if (word >= nwords || ((mask[word] >> (i % 32)) & 1) == 0)
                continue;
        }
        any = 1;
        if (y[i] > bestv) {
            bestv = y[i];
            best = i;
        }
    }
    return any ? best : 0;
}

/* Top-1 log-probability of token idx under softmax over the allowed tokens:
 * y[idx] - log(sum_j exp(y[j])), the sum taken in binary64 after subtracting
 * the largest allowed logit.  NaN when no token is allowed. */
double oracle_top1_logprob(const double *y, int64_t n, const int32_t *mask, int64_t nwords,
                           int64_t idx)
{
    double mx = -INFINITY;
    int any = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (mask != NULL) {
            int64_t word = i / 32;
            if (word >= nwords || ((mask[word] >> (i % 32)) & 1) == 0)
                continue;
        }
        any = 1;
        if (y[i] > mx)
            mx = y[i];
    }
    if (!any)
        return NAN;
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (mask != NULL) {
            int64_t word = i / 32;
            if (word >= nwords || ((mask[word] >> (i % 32)) & 1) == 0)
                continue;
        }
        s += exp(y[i] - mx);
    }
    return y[idx] - (mx + log(s));
}

/* ------------------------------------------------------------ FP8 weights
 * The pages' second projection precision: MtpHead::new
 * ("spark_model/layers/mtp_head/new.rs") resolves gemv_fp8w's
 * quantize_bf16_to_fp8 next to the NVFP4 pair, and the MtpQuantization::Fp8
 * arm resolves dense_gemv_fp8w; neither formula is printed.  Reading (one
 * kernel, so no separate global-absmax pass): E4M3 codes with one binary32
 * scale per output row,
 *     s_n = fl32(amax_n / 448),   c = E4M3_RNE_SATFINITE(fl32(x / s_n)),
 * the sign bit of c the sign of x, every code +0 when s_n == 0; the GEMV is
 *     y[m, n] = s_n * sum_i a[m, i] * e4m3(c[n, i]).
 * Layout: codes [N, K] row-major, scales [N].
 */
double oracle_fp8_value(int byte)
{
    const double v = oracle_e4m3_value(byte & 0x7F);
    return (byte & 0x80) ? -v : v;
}

int oracle_fp8_quantize_rows(const uint16_t *w, int64_t k, int64_t row0, int64_t nrows,
                             uint8_t *codes, float *row_scale)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t *x = w + (row0 + r) * k;
        float amax = 0.0f;
        for (int64_t i = 0; i < k; ++i) {
            const float v = oracle_bf16_to_float(x[i]);
            if (!isfinite(v))
                return 1;
            if (fabsf(v) > amax)
                amax = fabsf(v);
        }
        const float s = amax / 448.0f; /* binary32 division */
        row_scale[r] = s;
        for (int64_t i = 0; i < k; ++i) {
            const float v = oracle_bf16_to_float(x[i]);
            if (s == 0.0f) {
                codes[r * k + i] = 0;
                continue;
            }
            const float q = v / s; /* binary32 division */
            const int mag = oracle_e4m3_encode(fabsf(q));
            codes[r * k + i] = (uint8_t)(mag | (signbit(v) ? 0x80 : 0));
        }
    }
    return 0;
}

void oracle_fp8_gemv_rows(const uint16_t *a, int64_t m, int64_t lda, const uint8_t *codes,
                          const float *row_scale, int64_t k, int64_t n0, int64_t nn,
                          double *y, double *sabs)
{
    for (int64_t r = 0; r < m; ++r) {
        for (int64_t j = 0; j < nn; ++j) {
            double acc = 0.0, aacc = 0.0;
            const double s = (double)row_scale[n0 + j];
            for (int64_t i = 0; i < k; ++i) {
                double p = (double)oracle_bf16_to_float(a[r * lda + i]) *
                           (oracle_fp8_value(codes[(n0 + j) * k + i]) * s);
                acc += p;
                aacc += fabs(p);
            }
            y[r * nn + j] = acc;
            sabs[r * nn + j] = aacc;
        }
    }
}
