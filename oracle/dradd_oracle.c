/*
 * dradd_oracle.c -- plain, slow, single-threaded CPU oracle for the fused
 * residual-add + RMSNorm forward and its quantised variants (int8, fp8 e4m3,
 * fp4 e2m1), for its two halves (plain RMSNorm, no residual; the residual
 * update alone) and for the fused q/k RMSNorm with per-group e4m3 out.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only tests, the smoke check and the bench's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it follows (one web page is the authority on the op):
 *   ROCm/aiter issue #5151, "rmsnorm2d_fwd_with_add truncates fp32->bf16 on
 *   gfx942, biasing residual_out and compounding across layers".
 *   - section "Steps to Reproduce", function reference():
 *       acc = fp32(x) + fp32(residual)
 *       var = mean(acc^2) over the row
 *       out = cast((acc * rsqrt(var + eps)) * fp32(weight)),  residual_out = cast(acc)
 *   - section "Source": the truncating conversion (mode 2, keep the top 16 bits).
 *   - section "Problem Description" / "Notes": round-to-nearest-even is the
 *     unbiased conversion both stores must use.
 *   - section "Cost of fixing": the quantised configs emit int8 through a
 *     scaled cast instead of a bf16 store.
 *
 * Readings where the page leaves a step open (each one is listed in the
 * design notes of the repository):
 *   - mean(acc^2): every square is rounded to fp32 first, then summed by the
 *     textbook pairwise tree over the row padded with +0 to the next power of
 *     two (adjacent pairs, lowest index first), then divided by hidden.
 *   - rsqrt(v) is taken as 1 / sqrt(v) with both operations correctly rounded.
 *   - the two multiplications run left to right: (acc * inv) * weight.
 *   - no fused multiply-add anywhere, no flush-to-zero (IEEE subnormals).
 *   - int8 quant: per-row symmetric; amax = max |y|, scale = amax / 127,
 *     q = clamp(rint(y / scale), -127, 127) with ties to even; scale == 0
 *     gives q = 0.  y is the fp32 value before the bf16 store.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

/* Store modes for the two bf16 stores.  Only RNE is the method; the other
 * two are negative controls that reproduce the bias the page describes. */
enum {
    ORACLE_STORE_RNE = 0,       /* round to nearest, ties to even            */
    ORACLE_STORE_TRUNC = 1,     /* keep the top 16 bits (the page's mode 2)  */
    ORACLE_STORE_TIES_AWAY = 2  /* round to nearest, ties away from zero     */
};

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_ARG = 1,
    ORACLE_ERR_NOMEM = 2
};

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t bits_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* bf16 -> fp32 is exact: a bf16 value is the top half of an fp32 word. */
float oracle_bf16_to_f32(uint16_t b)
{
    return f32_from_bits((uint32_t)b << 16);
}

/* Round to nearest, ties to even, by comparing the two bf16 neighbours.
 * lo = the neighbour nearer zero (top 16 bits), hi = lo + 1 ulp in
 * magnitude.  Because bf16 is sign-magnitude, "lo + 1" on the bit pattern
 * is the next value away from zero; a carry into the exponent gives the
 * next binade, or infinity past the largest finite value.  NaN maps to a
 * quiet NaN with the sign kept. */
uint16_t oracle_bf16_rne(float f)
{
    uint32_t u = bits_from_f32(f);
    if (isnan(f))
        return (uint16_t)(0x7FC0u | ((u >> 16) & 0x8000u));
    uint16_t lo = (uint16_t)(u >> 16);
    uint32_t discarded = u & 0xFFFFu;
    if (discarded > 0x8000u)
        return (uint16_t)(lo + 1u);
    if (discarded < 0x8000u)
        return lo;
    /* exactly half way: take the neighbour whose last kept bit is 0 */
    return (lo & 1u) ? (uint16_t)(lo + 1u) : lo;
}

/* The page's mode 2: a plain shift, i.e. round toward zero. */
uint16_t oracle_bf16_trunc(float f)
{
    return (uint16_t)(bits_from_f32(f) >> 16);
}

/* Round to nearest, ties away from zero (second negative control). */
uint16_t oracle_bf16_ties_away(float f)
{
    uint32_t u = bits_from_f32(f);
    if (isnan(f))
        return (uint16_t)(0x7FC0u | ((u >> 16) & 0x8000u));
    uint16_t lo = (uint16_t)(u >> 16);
    return ((u & 0xFFFFu) >= 0x8000u) ? (uint16_t)(lo + 1u) : lo;
}

static uint16_t store_bf16(float f, int mode)
{
    switch (mode) {
    case ORACLE_STORE_TRUNC: return oracle_bf16_trunc(f);
    case ORACLE_STORE_TIES_AWAY: return oracle_bf16_ties_away(f);
    default: return oracle_bf16_rne(f);
    }
}

/* Convert `count` consecutive fp32 bit patterns starting at `first` (used by
 * the exhaustive checks of the conversion). */
int oracle_bf16_convert_range(uint16_t* dst, uint64_t first, int64_t count, int mode)
{
    if (!dst || count < 0)
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < count; ++i)
        dst[i] = store_bf16(f32_from_bits((uint32_t)(first + (uint64_t)i)), mode);
    return ORACLE_OK;
}

/* Convert n fp32 values to bf16 bit patterns. */
int oracle_bf16_convert_array(uint16_t* dst, const float* src, int64_t n, int mode)
{
    if ((!dst || !src) && n > 0)
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        dst[i] = store_bf16(src[i], mode);
    return ORACLE_OK;
}

static int64_t next_pow2(int64_t n)
{
    int64_t p = 1;
    while (p < n)
        p *= 2;
    return p;
}

/* Pairwise tree over v[0..len), len a power of two: the sum of a block is the
 * rounded sum of its lower half and its upper half. */
static float pairwise_pow2(const float* v, int64_t len)
{
    if (len == 1)
        return v[0];
    int64_t half = len / 2;
    float lower = pairwise_pow2(v, half);
    float upper = pairwise_pow2(v + half, half);
    return lower + upper;
}

/* Pairwise sum of v[0..n) after padding with +0 to the next power of two.
 * Returns +0 for n == 0. */
float oracle_pairwise_sum(const float* v, int64_t n)
{
    if (n <= 0)
        return 0.0f;
    int64_t p = next_pow2(n);
    float* padded = (float*)calloc((size_t)p, sizeof(float));
    if (!padded)
        return NAN;
    memcpy(padded, v, (size_t)n * sizeof(float));
    float s = pairwise_pow2(padded, p);
    free(padded);
    return s;
}

/* One row of the method.  acc and sq are caller scratch of length hidden and
 * next_pow2(hidden) (zero-filled past hidden).  y receives the fp32 value
 * before the store.  With residual == NULL (plain RMSNorm) acc is x alone and
 * residual_out is not written. */
static void add_rmsnorm_row(float* y, uint16_t* residual_out, float* acc, float* sq,
                            const uint16_t* x, const uint16_t* residual,
                            const uint16_t* weight, float eps, int64_t hidden,
                            int64_t padded, int store_mode,
                            float* sum_sq_out, float* inv_rms_out)
{
    for (int64_t i = 0; i < hidden; ++i) {
        if (residual) {
            acc[i] = oracle_bf16_to_f32(x[i]) + oracle_bf16_to_f32(residual[i]);
            residual_out[i] = store_bf16(acc[i], store_mode);
        } else {
            acc[i] = oracle_bf16_to_f32(x[i]);
        }
        sq[i] = acc[i] * acc[i];
    }
    float sum_sq = pairwise_pow2(sq, padded);
    float mean = sum_sq / (float)hidden;
    float var_eps = mean + eps;
    float root = sqrtf(var_eps);
    float inv_rms = 1.0f / root;
    for (int64_t i = 0; i < hidden; ++i) {
        float normed = acc[i] * inv_rms;
        y[i] = normed * oracle_bf16_to_f32(weight[i]);
    }
    if (sum_sq_out)
        *sum_sq_out = sum_sq;
    if (inv_rms_out)
        *inv_rms_out = inv_rms;
}

/* residual-add + RMSNorm forward with bf16 out.
 * Layout: x, residual, out, residual_out are row-major n_rows x hidden bf16
 * bit patterns; weight has hidden entries.  row_sum_sq and row_inv_rms are
 * optional (may be NULL) per-row outputs of the fp32 intermediates. */
int oracle_add_rmsnorm_fwd(uint16_t* out, uint16_t* residual_out,
                           const uint16_t* x, const uint16_t* residual,
                           const uint16_t* weight, float eps,
                           int64_t n_rows, int64_t hidden, int store_mode,
                           float* row_sum_sq, float* row_inv_rms)
{
    if (n_rows < 0 || hidden <= 0)
        return ORACLE_ERR_ARG;
    if (n_rows == 0)
        return ORACLE_OK;
    if (!out || !residual_out || !x || !residual || !weight)
        return ORACLE_ERR_ARG;
    int64_t padded = next_pow2(hidden);
    float* acc = (float*)malloc((size_t)hidden * sizeof(float));
    float* sq = (float*)calloc((size_t)padded, sizeof(float));
    float* y = (float*)malloc((size_t)hidden * sizeof(float));
    if (!acc || !sq || !y) {
        free(acc); free(sq); free(y);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t base = r * hidden;
        add_rmsnorm_row(y, residual_out + base, acc, sq, x + base, residual + base,
                        weight, eps, hidden, padded, store_mode,
                        row_sum_sq ? row_sum_sq + r : NULL,
                        row_inv_rms ? row_inv_rms + r : NULL);
        for (int64_t i = 0; i < hidden; ++i)
            out[base + i] = store_bf16(y[i], store_mode);
    }
    free(acc); free(sq); free(y);
    return ORACLE_OK;
}

/* Round to the nearest integer, ties to even, in the default rounding mode;
 * NaN gives 0. */
static int32_t round_half_even_to_int(float v)
{
    if (isnan(v))
        return 0;
    if (v > 2147483520.0f)
        return INT32_MAX;
    if (v < -2147483648.0f)
        return INT32_MIN;
    return (int32_t)rintf(v);
}

/* Per-row symmetric int8 codes of the fp32 row y: amax = max |y|,
 * scale = amax / 127, q = clamp(rint(y / scale), -127, 127); scale == 0
 * gives q = 0. */
static void quantize_row(int8_t* q_out, float* scale_out, const float* y, int64_t hidden)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < hidden; ++i)
        amax = fmaxf(amax, fabsf(y[i]));
    float s = amax / 127.0f;
    *scale_out = s;
    for (int64_t i = 0; i < hidden; ++i) {
        int32_t q = 0;
        if (s != 0.0f) {
            q = round_half_even_to_int(y[i] / s);
            if (q > 127) q = 127;
            if (q < -127) q = -127;
        }
        q_out[i] = (int8_t)q;
    }
}

/* ---- fp8 e4m3 (OCP "e4m3fn": 1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; no infinities; S.1111.111 is NaN; the largest finite
 * magnitude is 448 = 1.75 * 2^8; subnormals are m * 2^-9). */
#define E4M3_MAX 448.0f

/* Magnitude of the e4m3 code c (0 <= c <= 0x7E). */
static double e4m3_magnitude(unsigned c)
{
    unsigned e = (c >> 3) & 0xFu, m = c & 7u;
    if (e == 0)
        return ldexp((double)m, -9);
    return ldexp(1.0 + m / 8.0, (int)e - 7);
}

/* Magnitudes of the finite codes 0x00..0x7E, which increase with the code. */
static double e4m3_table[0x7F];
static int e4m3_table_ready;

static void e4m3_fill_table(void)
{
    if (e4m3_table_ready)
        return;
    for (unsigned c = 0; c < 0x7Fu; ++c)
        e4m3_table[c] = e4m3_magnitude(c);
    e4m3_table_ready = 1;  /* every caller writes the same values */
}

/* Round to the nearest e4m3 value, ties to the even code (last mantissa bit
 * 0); magnitudes above 448 saturate to 448 ("satfinite"); NaN gives 0x7F
 * with the sign kept.  |f| is placed between two consecutive finite
 * magnitudes by binary search and the nearer one is taken. */
uint8_t oracle_e4m3_rne(float f)
{
    uint8_t sign = (uint8_t)((bits_from_f32(f) >> 24) & 0x80u);
    if (isnan(f))
        return (uint8_t)(sign | 0x7Fu);
    double a = fabs((double)f);
    if (a >= (double)E4M3_MAX)
        return (uint8_t)(sign | 0x7Eu);
    e4m3_fill_table();
    unsigned lo = 0, hi = 0x7Eu;  /* largest code with magnitude <= a lies in [lo, hi) */
    while (hi - lo > 1) {
        unsigned mid = (lo + hi) / 2;
        if (e4m3_table[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    double d_lo = a - e4m3_table[lo], d_hi = e4m3_table[lo + 1] - a;
    unsigned c = lo;
    if (d_hi < d_lo || (d_hi == d_lo && (lo & 1u)))
        c = lo + 1;
    return (uint8_t)(sign | c);
}

/* Per-row symmetric e4m3 codes of the fp32 row y: amax = max |y|,
 * scale = amax / 448, q = e4m3_rne(y / scale); scale == 0 gives q = 0. */
static void quantize_row_e4m3(uint8_t* q_out, float* scale_out, const float* y, int64_t hidden)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < hidden; ++i)
        amax = fmaxf(amax, fabsf(y[i]));
    float s = amax / E4M3_MAX;
    *scale_out = s;
    for (int64_t i = 0; i < hidden; ++i)
        q_out[i] = s != 0.0f ? oracle_e4m3_rne(y[i] / s) : 0;
}

/* residual-add + RMSNorm forward with per-row e4m3 out (x, residual ==
 * NULL: plain RMSNorm, residual_out not written). */
int oracle_rmsnorm_e4m3_fwd(uint8_t* out_q, float* scale, uint16_t* residual_out,
                            const uint16_t* x, const uint16_t* residual,
                            const uint16_t* weight, float eps, int64_t n_rows, int64_t hidden)
{
    if (n_rows < 0 || hidden <= 0)
        return ORACLE_ERR_ARG;
    if (n_rows == 0)
        return ORACLE_OK;
    if (!out_q || !scale || !x || !weight || (residual && !residual_out))
        return ORACLE_ERR_ARG;
    int64_t padded = next_pow2(hidden);
    float* acc = (float*)malloc((size_t)hidden * sizeof(float));
    float* sq = (float*)calloc((size_t)padded, sizeof(float));
    float* y = (float*)malloc((size_t)hidden * sizeof(float));
    if (!acc || !sq || !y) {
        free(acc); free(sq); free(y);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t base = r * hidden;
        add_rmsnorm_row(y, residual ? residual_out + base : NULL, acc, sq, x + base,
                        residual ? residual + base : NULL, weight, eps, hidden, padded,
                        ORACLE_STORE_RNE, NULL, NULL);
        quantize_row_e4m3(out_q + base, scale + r, y, hidden);
    }
    free(acc); free(sq); free(y);
    return ORACLE_OK;
}

/* Convert n fp32 values to e4m3 codes (for the conversion checks). */
int oracle_e4m3_convert_array(uint8_t* dst, const float* src, int64_t n)
{
    if ((!dst || !src) && n > 0)
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_e4m3_rne(src[i]);
    return ORACLE_OK;
}

/* ---- fp4 e2m1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; the
 * magnitudes of codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinities or
 * NaN).  Two codes per byte: the even element in the low nibble. */
#define E2M1_MAX 6.0f

static const double e2m1_magnitudes[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Nearest e2m1 code, ties to the even code, magnitudes past 6 saturating to
 * 6; the sign bit (bit 3) follows the sign of f; NaN gives 0 (the format has
 * no NaN; outside this library's use). */
uint8_t oracle_e2m1_rne(float f)
{
    if (isnan(f))
        return 0;
    uint8_t sign = (uint8_t)((bits_from_f32(f) >> 28) & 0x8u);
    double a = fabs((double)f);
    if (a >= (double)E2M1_MAX)
        return (uint8_t)(sign | 7u);
    unsigned lo = 0;
    while (lo < 7u && e2m1_magnitudes[lo + 1] <= a)
        ++lo;
    double d_lo = a - e2m1_magnitudes[lo], d_hi = e2m1_magnitudes[lo + 1] - a;
    unsigned c = lo;
    if (d_hi < d_lo || (d_hi == d_lo && (lo & 1u)))
        c = lo + 1;
    return (uint8_t)(sign | c);
}

/* Per-row symmetric e2m1 codes of y, packed two per byte:
 * scale = amax / 6, code = e2m1_rne(y / scale); scale == 0 gives code 0. */
static void quantize_row_e2m1(uint8_t* q_out, float* scale_out, const float* y, int64_t hidden)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < hidden; ++i)
        amax = fmaxf(amax, fabsf(y[i]));
    float s = amax / E2M1_MAX;
    *scale_out = s;
    for (int64_t i = 0; i < hidden; i += 2) {
        uint8_t c0 = s != 0.0f ? oracle_e2m1_rne(y[i] / s) : 0;
        uint8_t c1 = s != 0.0f ? oracle_e2m1_rne(y[i + 1] / s) : 0;
        q_out[i / 2] = (uint8_t)(c0 | (c1 << 4));
    }
}

/* Residual-add + RMSNorm (or plain, residual == NULL) with per-row e2m1
 * out: out_q holds n_rows x hidden / 2 bytes.  hidden must be even. */
int oracle_rmsnorm_e2m1_fwd(uint8_t* out_q, float* scale, uint16_t* residual_out,
                            const uint16_t* x, const uint16_t* residual,
                            const uint16_t* weight, float eps, int64_t n_rows, int64_t hidden)
{
    if (n_rows < 0 || hidden <= 0 || hidden % 2)
        return ORACLE_ERR_ARG;
    if (n_rows == 0)
        return ORACLE_OK;
    if (!out_q || !scale || !x || !weight || (residual && !residual_out))
        return ORACLE_ERR_ARG;
    int64_t padded = next_pow2(hidden);
    float* acc = (float*)malloc((size_t)hidden * sizeof(float));
    float* sq = (float*)calloc((size_t)padded, sizeof(float));
    float* y = (float*)malloc((size_t)hidden * sizeof(float));
    if (!acc || !sq || !y) {
        free(acc); free(sq); free(y);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t base = r * hidden;
        add_rmsnorm_row(y, residual ? residual_out + base : NULL, acc, sq, x + base,
                        residual ? residual + base : NULL, weight, eps, hidden, padded,
                        ORACLE_STORE_RNE, NULL, NULL);
        quantize_row_e2m1(out_q + base / 2, scale + r, y, hidden);
    }
    free(acc); free(sq); free(y);
    return ORACLE_OK;
}

/* Convert n fp32 values to e2m1 codes, one per byte (for the conversion
 * checks). */
int oracle_e2m1_convert_array(uint8_t* dst, const float* src, int64_t n)
{
    if ((!dst || !src) && n > 0)
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_e2m1_rne(src[i]);
    return ORACLE_OK;
}

/* residual-add + RMSNorm forward with per-row symmetric int8 out.
 * out_q: n_rows x hidden int8; scale: n_rows fp32 (q * scale ~ y). */
int oracle_add_rmsnorm_quant_fwd(int8_t* out_q, float* scale, uint16_t* residual_out,
                                 const uint16_t* x, const uint16_t* residual,
                                 const uint16_t* weight, float eps,
                                 int64_t n_rows, int64_t hidden, int store_mode,
                                 float* row_sum_sq, float* row_inv_rms)
{
    if (n_rows < 0 || hidden <= 0)
        return ORACLE_ERR_ARG;
    if (n_rows == 0)
        return ORACLE_OK;
    if (!out_q || !scale || !residual_out || !x || !residual || !weight)
        return ORACLE_ERR_ARG;
    int64_t padded = next_pow2(hidden);
    float* acc = (float*)malloc((size_t)hidden * sizeof(float));
    float* sq = (float*)calloc((size_t)padded, sizeof(float));
    float* y = (float*)malloc((size_t)hidden * sizeof(float));
    if (!acc || !sq || !y) {
        free(acc); free(sq); free(y);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t base = r * hidden;
        add_rmsnorm_row(y, residual_out + base, acc, sq, x + base, residual + base,
                        weight, eps, hidden, padded, store_mode,
                        row_sum_sq ? row_sum_sq + r : NULL,
                        row_inv_rms ? row_inv_rms + r : NULL);
        quantize_row(out_q + base, scale + r, y, hidden);
    }
    free(acc); free(sq); free(y);
    return ORACLE_OK;
}

/* Plain RMSNorm: the row function without a residual.  Same layout as
 * oracle_add_rmsnorm_fwd, minus residual and residual_out. */
int oracle_rmsnorm_fwd(uint16_t* out, const uint16_t* x, const uint16_t* weight, float eps,
                       int64_t n_rows, int64_t hidden, int store_mode,
                       float* row_sum_sq, float* row_inv_rms)
{
    if (n_rows < 0 || hidden <= 0)
        return ORACLE_ERR_ARG;
    if (n_rows == 0)
        return ORACLE_OK;
    if (!out || !x || !weight)
        return ORACLE_ERR_ARG;
    int64_t padded = next_pow2(hidden);
    float* acc = (float*)malloc((size_t)hidden * sizeof(float));
    float* sq = (float*)calloc((size_t)padded, sizeof(float));
    float* y = (float*)malloc((size_t)hidden * sizeof(float));
    if (!acc || !sq || !y) {
        free(acc); free(sq); free(y);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t base = r * hidden;
        add_rmsnorm_row(y, NULL, acc, sq, x + base, NULL, weight, eps, hidden, padded, store_mode,
                        row_sum_sq ? row_sum_sq + r : NULL,
                        row_inv_rms ? row_inv_rms + r : NULL);
        for (int64_t i = 0; i < hidden; ++i)
            out[base + i] = store_bf16(y[i], store_mode);
    }
    free(acc); free(sq); free(y);
    return ORACLE_OK;
}

/* Plain RMSNorm with the per-row symmetric int8 output. */
int oracle_rmsnorm_quant_fwd(int8_t* out_q, float* scale, const uint16_t* x, const uint16_t* weight,
                             float eps, int64_t n_rows, int64_t hidden)
{
    if (n_rows < 0 || hidden <= 0)
        return ORACLE_ERR_ARG;
    if (n_rows == 0)
        return ORACLE_OK;
    if (!out_q || !scale || !x || !weight)
        return ORACLE_ERR_ARG;
    int64_t padded = next_pow2(hidden);
    float* acc = (float*)malloc((size_t)hidden * sizeof(float));
    float* sq = (float*)calloc((size_t)padded, sizeof(float));
    float* y = (float*)malloc((size_t)hidden * sizeof(float));
    if (!acc || !sq || !y) {
        free(acc); free(sq); free(y);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t base = r * hidden;
        add_rmsnorm_row(y, NULL, acc, sq, x + base, NULL, weight, eps, hidden, padded,
                        ORACLE_STORE_RNE, NULL, NULL);
        quantize_row(out_q + base, scale + r, y, hidden);
    }
    free(acc); free(sq); free(y);
    return ORACLE_OK;
}

/* The residual update alone: residual_out = store(fp32(x) + fp32(residual))
 * for n elements. */
int oracle_residual_add_fwd(uint16_t* residual_out, const uint16_t* x, const uint16_t* residual,
                            int64_t n, int store_mode)
{
    if (n < 0 || (n > 0 && (!residual_out || !x || !residual)))
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) {
        float acc = oracle_bf16_to_f32(x[i]) + oracle_bf16_to_f32(residual[i]);
        residual_out[i] = store_bf16(acc, store_mode);
    }
    return ORACLE_OK;
}

/* ---- fused q/k RMSNorm with per-group e4m3 out.
 * The page (section "Notes") names a second kernel whose bf16 residual
 * stores were not audited: the fused q/k RMSNorm + group quant kernel.  It
 * prints no formula for it; the reading taken here is the plainest one that
 * the name and the rest of the page support:
 *   - two independent sets of rows normalised in one call, "q" (n_q_rows x
 *     q_hidden, weight q_weight, eps q_eps) and "k" (n_k_rows x k_hidden,
 *     weight k_weight, eps k_eps); a per-head norm is the same call with
 *     rows = tokens x heads and hidden = head size;
 *   - each row is the row function above: q with an optional residual add
 *     (q_residual != NULL; q_residual_out gets the round-to-nearest-even
 *     bf16 of the fp32 sum), k plain;
 *   - "group quant": q's fp32 output is cut into consecutive groups of
 *     group_size elements, each quantised to e4m3 exactly as a row of the
 *     per-row e4m3 output (scale = amax / 448 over the group, code =
 *     e4m3_rne(y / scale)); q_scale holds n_q_rows x (q_hidden / group_size)
 *     scales, row-major.  group_size == 0 stores q as bf16 (round to nearest
 *     even) instead, with q_scale unused;
 *   - k's output is always bf16, rounded to nearest even.
 * q_out is uint16_t bf16 bit patterns when group_size == 0, else uint8_t
 * e4m3 codes.  Either row count may be 0. */
static int qk_rows(void* q_out, float* q_scale, uint16_t* residual_out, const uint16_t* x,
                   const uint16_t* residual, const uint16_t* weight, float eps, int64_t n_rows,
                   int64_t hidden, int64_t group_size)
{
    int64_t padded = next_pow2(hidden);
    float* acc = (float*)malloc((size_t)hidden * sizeof(float));
    float* sq = (float*)calloc((size_t)padded, sizeof(float));
    float* y = (float*)malloc((size_t)hidden * sizeof(float));
    if (!acc || !sq || !y) {
        free(acc); free(sq); free(y);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t base = r * hidden;
        add_rmsnorm_row(y, residual ? residual_out + base : NULL, acc, sq, x + base,
                        residual ? residual + base : NULL, weight, eps, hidden, padded,
                        ORACLE_STORE_RNE, NULL, NULL);
        if (group_size == 0) {
            uint16_t* o = (uint16_t*)q_out + base;
            for (int64_t i = 0; i < hidden; ++i)
                o[i] = store_bf16(y[i], ORACLE_STORE_RNE);
        } else {
            int64_t groups = hidden / group_size;
            for (int64_t g = 0; g < groups; ++g)
                quantize_row_e4m3((uint8_t*)q_out + base + g * group_size,
                                  q_scale + r * groups + g, y + g * group_size, group_size);
        }
    }
    free(acc); free(sq); free(y);
    return ORACLE_OK;
}

int oracle_qk_rmsnorm_fwd(void* q_out, float* q_scale, uint16_t* q_residual_out, uint16_t* k_out,
                          const uint16_t* q, const uint16_t* q_residual, const uint16_t* q_weight,
                          const uint16_t* k, const uint16_t* k_weight, float q_eps, float k_eps,
                          int64_t n_q_rows, int64_t q_hidden, int64_t n_k_rows, int64_t k_hidden,
                          int64_t group_size)
{
    if (n_q_rows < 0 || n_k_rows < 0 || group_size < 0)
        return ORACLE_ERR_ARG;
    if (n_q_rows > 0) {
        if (q_hidden <= 0 || !q_out || !q || !q_weight || (q_residual && !q_residual_out))
            return ORACLE_ERR_ARG;
        if (group_size > 0 && (q_hidden % group_size != 0 || !q_scale))
            return ORACLE_ERR_ARG;
        int rc = qk_rows(q_out, q_scale, q_residual_out, q, q_residual, q_weight, q_eps, n_q_rows,
                         q_hidden, group_size);
        if (rc != ORACLE_OK)
            return rc;
    }
    if (n_k_rows > 0) {
        if (k_hidden <= 0 || !k_out || !k || !k_weight)
            return ORACLE_ERR_ARG;
        return qk_rows(k_out, NULL, NULL, k, NULL, k_weight, k_eps, n_k_rows, k_hidden, 0);
    }
    return ORACLE_OK;
}

int oracle_abi_version(void)
{
    return 1;
}
