/*
 * lse_oracle.c -- plain CPU oracle for the log-sum-exp merge and for the
 * elementwise functions whose results must not depend on how a kernel is
 * launched.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only tests, the smoke check and the bench's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it follows: ROCm/TransformerEngine issue #693, "CP LSE merge switches
 * compiled variants on ROCm, breaking forward reproducibility":
 *   - "Summary": context parallelism merges the softmax log-sum-exp of the
 *     attention blocks computed on different ranks (two merge functions, one
 *     of them for the second half of the sequence);
 *   - "Root cause": log1p (and cosh) gave launch-configuration-dependent
 *     bits; exp, log and the others did not.
 * The merge of two partial log-sum-exps a = log(sum_i e^s_i) and
 * b = log(sum_j e^s_j) is log(e^a + e^b).  It is evaluated here in double
 * precision in the overflow-free form max + log1p(exp(min - max)), which is
 * the same quantity; the inputs are fp32, the results double (the kernels'
 * fp32 results are compared against these within a stated bound).
 * Special values: both inputs -inf (an empty block on both sides) gives
 * -inf; any NaN gives NaN; a +inf input gives +inf.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 */
#include <math.h>
#include <stdint.h>

enum { LSE_ORACLE_OK = 0, LSE_ORACLE_ERR_ARG = 1 };

/* Unary functions: 0 log1p, 1 cosh, 2 exp (the ones the page found
 * launch-dependent, and the exponential the merge uses). */
enum { LSE_UNARY_LOG1P = 0, LSE_UNARY_COSH = 1, LSE_UNARY_EXP = 2 };

double oracle_lse_merge1(float a, float b)
{
    if (isnan(a) || isnan(b))
        return NAN;
    double hi = a > b ? (double)a : (double)b;
    double lo = a > b ? (double)b : (double)a;
    if (isinf(hi))
        return hi; /* +inf, or -inf when both are -inf */
    if (isinf(lo))
        return hi; /* e^-inf = 0 */
    return hi + log1p(exp(lo - hi));
}

/* out[i] = merge(a[i], b[i]) for n elements. */
int oracle_lse_merge(double* out, const float* a, const float* b, int64_t n)
{
    if (n < 0 || (n > 0 && (!out || !a || !b)))
        return LSE_ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_lse_merge1(a[i], b[i]);
    return LSE_ORACLE_OK;
}

/* Row-strided form: out[r * n_cols + c] = merge(a[r * a_stride + c],
 * b[r * b_stride + c]) (strides in elements). */
int oracle_lse_merge_2d(double* out, const float* a, int64_t a_stride, const float* b, int64_t b_stride,
                        int64_t n_rows, int64_t n_cols)
{
    if (n_rows < 0 || n_cols < 0)
        return LSE_ORACLE_ERR_ARG;
    if (n_rows == 0 || n_cols == 0)
        return LSE_ORACLE_OK;
    if (!out || !a || !b || a_stride < n_cols || b_stride < n_cols)
        return LSE_ORACLE_ERR_ARG;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t c = 0; c < n_cols; ++c)
            out[r * n_cols + c] = oracle_lse_merge1(a[r * a_stride + c], b[r * b_stride + c]);
    return LSE_ORACLE_OK;
}

int oracle_unary(double* out, const float* x, int64_t n, int op)
{
    if (n < 0 || (n > 0 && (!out || !x)) || op < 0 || op > 2)
        return LSE_ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) {
        double v = (double)x[i];
        out[i] = op == LSE_UNARY_LOG1P ? log1p(v) : op == LSE_UNARY_COSH ? cosh(v) : exp(v);
    }
    return LSE_ORACLE_OK;
}
