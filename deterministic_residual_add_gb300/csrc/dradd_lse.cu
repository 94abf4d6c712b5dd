// dradd_lse.cu -- the log-sum-exp merge and the launch-invariant elementwise
// functions (ROCm/TransformerEngine issue #693, "CP LSE merge switches
// compiled variants on ROCm, breaking forward reproducibility").
//
// The page's failure: the same elementwise function (log1p, cosh) compiled
// into two kernel variants for two launch configurations gave different
// bits for the same input.  Here every element goes through one scalar
// device function whatever the launch: the configuration only decides which
// thread handles which element (VEC elements per thread per pass, any CTA
// size, any grid), never the arithmetic.  Every operation is an IEEE fp32
// operation or a CUDA math-library call compiled without fast-math options
// and without multiply-add contraction, so each element's bits are a fixed
// function of its inputs.  The merge's log1p is the series below (its
// argument lies in [0, 1]); the unary entry point keeps the library's
// log1pf, the function the page found launch-dependent.
#include <cmath>

#include "dradd_device.cuh"
#include "dradd_internal.h"

namespace dradd {

// log1p(u) for u in [0, 1]: 2 atanh(s) with s = u / (2 + u) <= 1/3, by the
// atanh series 2 s (1 + s^2/3 + s^4/5 + ... + s^16/17), whose truncation is
// below 2^-28 of the value.  Every step is an IEEE fp32 operation (the
// division correctly rounded, the series in fused multiply-adds), so
// tests/log1p_series_check.c runs the same operations on the CPU: against
// log1p in double, every fp32 u in [0, 1] is within 2.95 x 2^-24 relative
// (plus 2^-148 absolute for subnormal u).  About a third of the
// instructions of the general-purpose log1pf.
__device__ __forceinline__ float log1p_unit(float u)
{
    const float s = __fdiv_rn(u, __fadd_rn(2.0f, u));
    const float z = __fmul_rn(s, s);
    float p = 0x1.e1e1e2p-5f;              // 1/17
    p = __fmaf_rn(p, z, 0x1.111112p-4f);   // 1/15
    p = __fmaf_rn(p, z, 0x1.3b13b2p-4f);   // 1/13
    p = __fmaf_rn(p, z, 0x1.745d18p-4f);   // 1/11
    p = __fmaf_rn(p, z, 0x1.c71c72p-4f);   // 1/9
    p = __fmaf_rn(p, z, 0x1.24924ap-3f);   // 1/7
    p = __fmaf_rn(p, z, 0x1.99999ap-3f);   // 1/5
    p = __fmaf_rn(p, z, 0x1.555556p-2f);   // 1/3
    const float two_s = __fmul_rn(2.0f, s);
    return __fmaf_rn(__fmul_rn(two_s, z), p, two_s);
}

// log(e^a + e^b) as hi + log1p(exp(lo - hi)) (exp: the CUDA library's
// expf); both -inf gives -inf, +inf wins, NaN propagates.
__device__ __forceinline__ float lse_merge1(float a, float b)
{
    if (!(isfinite(a) && isfinite(b))) {
        if (isnan(a) || isnan(b))
            return __int_as_float(0x7fc00000);
        return a > b ? a : b;  // an infinite operand: +inf wins; -inf leaves the other
    }
    const float hi = a > b ? a : b;
    const float lo = a > b ? b : a;
    return __fadd_rn(hi, log1p_unit(expf(__fsub_rn(lo, hi))));
}

// Two merges at once: the same operations as lse_merge1 for each element,
// the subtraction, the series and the final addition on packed pairs (each
// lane the IEEE operation, so each element's bits are lse_merge1's).
__device__ __forceinline__ void lse_merge2(float a0, float a1, float b0, float b1, float& r0, float& r1)
{
    const float hi0 = a0 > b0 ? a0 : b0, lo0 = a0 > b0 ? b0 : a0;
    const float hi1 = a1 > b1 ? a1 : b1, lo1 = a1 > b1 ? b1 : a1;
    float d0, d1;
    sub2_rn(lo0, lo1, hi0, hi1, d0, d1);
    const float u0 = expf(d0), u1 = expf(d1);
    float t0, t1;
    add2_rn(2.0f, 2.0f, u0, u1, t0, t1);
    const float s0 = __fdiv_rn(u0, t0), s1 = __fdiv_rn(u1, t1);
    float z0, z1;
    mul2_rn(s0, s1, s0, s1, z0, z1);
    float p0 = 0x1.e1e1e2p-5f, p1 = 0x1.e1e1e2p-5f;
    fma2_rn(p0, p1, z0, z1, 0x1.111112p-4f, 0x1.111112p-4f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.3b13b2p-4f, 0x1.3b13b2p-4f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.745d18p-4f, 0x1.745d18p-4f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.c71c72p-4f, 0x1.c71c72p-4f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.24924ap-3f, 0x1.24924ap-3f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.99999ap-3f, 0x1.99999ap-3f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.555556p-2f, 0x1.555556p-2f, p0, p1);
    float w0, w1, q0, q1, l0, l1;
    mul2_rn(2.0f, 2.0f, s0, s1, w0, w1);
    mul2_rn(w0, w1, z0, z1, q0, q1);
    fma2_rn(q0, q1, p0, p1, w0, w1, l0, l1);
    add2_rn(hi0, hi1, l0, l1, r0, r1);
    if (!(isfinite(a0) && isfinite(b0)))
        r0 = lse_merge1(a0, b0);
    if (!(isfinite(a1) && isfinite(b1)))
        r1 = lse_merge1(a1, b1);
}

__device__ __forceinline__ float unary1(float x, int op)
{
    return op == 0 ? log1pf(x) : op == 1 ? coshf(x) : expf(x);
}

// Rows of n_cols elements; a unit is `blockDim.x * VEC` consecutive columns
// of one row, units_per_row of them per row; the grid strides over units
// (in row-major unit order).
// Thread t of a unit handles columns c0 + t + v * blockDim.x, v < VEC.
template <int VEC>
__global__ void __launch_bounds__(1024) lse_merge_kernel(float* out, int64_t out_stride, const float* a,
                                                         int64_t a_stride, const float* b, int64_t b_stride,
                                                         int64_t n_rows, int64_t n_cols)
{
    wait_prior_grids();
    allow_next_grid();
    const int64_t span = static_cast<int64_t>(blockDim.x) * VEC;
    const int64_t units_per_row = (n_cols + span - 1) / span;
    // unit u = row * units_per_row + cb, walked with a stride of gridDim.x:
    // (row, cb) advances by (gridDim.x / units_per_row, gridDim.x %
    // units_per_row) with a carry, so the loop divides only once here
    const int64_t step_rows = gridDim.x / units_per_row;
    const int64_t step_cb = gridDim.x - step_rows * units_per_row;
    int64_t row = blockIdx.x / units_per_row;
    int64_t cb = blockIdx.x - row * units_per_row;
    for (; row < n_rows; row += step_rows) {
        const int64_t c0 = cb * span + threadIdx.x;
        const float* ar = a + row * a_stride;
        const float* br = b + row * b_stride;
        float* orow = out + row * out_stride;
        float va[VEC], vb[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int64_t c = c0 + static_cast<int64_t>(v) * blockDim.x;
            if (c < n_cols) {
                va[v] = __ldcs(ar + c);
                vb[v] = __ldcs(br + c);
            }
        }
        if constexpr (VEC == 1) {
            if (c0 < n_cols)
                __stcs(orow + c0, lse_merge1(va[0], vb[0]));
        } else {
#pragma unroll
            for (int v = 0; v < VEC; v += 2) {
                const int64_t c = c0 + static_cast<int64_t>(v) * blockDim.x;
                const int64_t c1 = c + blockDim.x;
                float r0, r1;
                lse_merge2(va[v], va[v + 1], vb[v], vb[v + 1], r0, r1);
                if (c < n_cols)
                    __stcs(orow + c, r0);
                if (c1 < n_cols)
                    __stcs(orow + c1, r1);
            }
        }
        cb += step_cb;
        if (cb >= units_per_row) {
            cb -= units_per_row;
            ++row;
        }
    }
}

template <int VEC>
__global__ void __launch_bounds__(1024) unary_kernel(float* out, const float* x, int64_t n, int op)
{
    wait_prior_grids();
    allow_next_grid();
    const int64_t span = static_cast<int64_t>(blockDim.x) * VEC;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * span + threadIdx.x; base - threadIdx.x < n;
         base += static_cast<int64_t>(gridDim.x) * span) {
        float vx[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int64_t i = base + static_cast<int64_t>(v) * blockDim.x;
            if (i < n)
                vx[v] = __ldcs(x + i);
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int64_t i = base + static_cast<int64_t>(v) * blockDim.x;
            if (i < n)
                __stcs(out + i, unary1(vx[v], op));
        }
    }
}

cudaError_t launch_lse_merge(float* out, int64_t out_stride, const float* a, int64_t a_stride, const float* b,
                             int64_t b_stride, int64_t n_rows, int64_t n_cols, int vec, int grid, int threads,
                             bool serialize, cudaStream_t stream)
{
    void (*fn)(float*, int64_t, const float*, int64_t, const float*, int64_t, int64_t, int64_t) =
        vec == 1 ? lse_merge_kernel<1> : vec == 2 ? lse_merge_kernel<2> : vec == 4 ? lse_merge_kernel<4>
        : vec == 8 ? lse_merge_kernel<8> : nullptr;
    if (!fn)
        return cudaErrorInvalidValue;
    return launch(fn, grid, threads, 0, serialize, stream, out, out_stride, a, a_stride, b, b_stride, n_rows,
                  n_cols);
}

cudaError_t launch_unary(float* out, const float* x, int64_t n, int op, int vec, int grid, int threads,
                         bool serialize, cudaStream_t stream)
{
    void (*fn)(float*, const float*, int64_t, int) = vec == 1 ? unary_kernel<1> : vec == 2 ? unary_kernel<2>
                                                     : vec == 4 ? unary_kernel<4> : vec == 8 ? unary_kernel<8>
                                                                                             : nullptr;
    if (!fn)
        return cudaErrorInvalidValue;
    return launch(fn, grid, threads, 0, serialize, stream, out, x, n, op);
}

}  // namespace dradd
