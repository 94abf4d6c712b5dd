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
// function of its inputs.
#include <cmath>

#include "dradd_device.cuh"
#include "dradd_internal.h"

namespace dradd {

// log(e^a + e^b) as hi + log1p(exp(lo - hi)); both -inf gives -inf, +inf
// wins, NaN propagates.
__device__ __forceinline__ float lse_merge1(float a, float b)
{
    if (isnan(a) || isnan(b))
        return __int_as_float(0x7fc00000);
    const float hi = a > b ? a : b;
    const float lo = a > b ? b : a;
    if (isinf(hi) || isinf(lo))
        return hi;
    return __fadd_rn(hi, log1pf(expf(__fsub_rn(lo, hi))));
}

__device__ __forceinline__ float unary1(float x, int op)
{
    return op == 0 ? log1pf(x) : op == 1 ? coshf(x) : expf(x);
}

// Rows of n_cols elements; a unit is `blockDim.x * VEC` consecutive columns
// of one row, units_per_row of them per row; the grid strides over units.
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
    const int64_t units = units_per_row * n_rows;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t row = u / units_per_row;
        const int64_t c0 = (u - row * units_per_row) * span + threadIdx.x;
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
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int64_t c = c0 + static_cast<int64_t>(v) * blockDim.x;
            if (c < n_cols)
                __stcs(orow + c, lse_merge1(va[v], vb[v]));
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
