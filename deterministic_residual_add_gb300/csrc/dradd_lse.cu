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
// operation, a hardware approximation instruction or a CUDA math-library
// call, compiled without fast-math options and without multiply-add
// contraction, so each element's bits are a fixed function of its inputs.  The merge's log1p is the series below (its
// argument lies in [0, 1]); the unary entry point keeps the library's
// log1pf, the function the page found launch-dependent.
#include <cmath>

#include "dradd_device.cuh"
#include "dradd_internal.h"

namespace dradd {

// log1p(u) for u in [0, 1]: 2 atanh(s) with s = u / t, t = RN(2 + u), s <=
// 1/3, by the atanh series 2 s (1 + s^2/3 + s^4/5 + ... + s^12/13), whose
// truncation is below (1/9)^7 / 15 < 2^-26 of the value (the two further
// terms the series once carried change no worst case below); the series
// in fused multiply-adds.  The division is a reciprocal approximation with one
// correction step (Markstein): r = rcp.approx(t) (within 1 ulp),
// q0 = RN(u r), the remainder u - q0 t exact in one fused multiply-add,
// s = RN(q0 + rem r).  Before its last rounding that value is within
// 1.5 x 2^-46 (relative) of u / t, so s is the correctly rounded quotient
// unless u / t lies that close to a rounding midpoint, where it may be the
// other neighbour.  tests/log1p_series_check.c runs these operations on the
// CPU, with both neighbours wherever the quotient is that close to a
// midpoint: against log1p in double every fp32 u in [2^-125, 1] is within
// 2.95 x 2^-24 relative, and every smaller u within 2^-146 absolute.
__device__ __forceinline__ float series_tail(float z)
{
    float p = 0x1.3b13b2p-4f;              // 1/13
    p = __fmaf_rn(p, z, 0x1.745d18p-4f);   // 1/11
    p = __fmaf_rn(p, z, 0x1.c71c72p-4f);   // 1/9
    p = __fmaf_rn(p, z, 0x1.24924ap-3f);   // 1/7
    p = __fmaf_rn(p, z, 0x1.99999ap-3f);   // 1/5
    return __fmaf_rn(p, z, 0x1.555556p-2f); // 1/3
}

// The reciprocal approximation for an argument in [2, 3] (t = 2 + u): the
// flush-to-zero form of rcp.approx, without the subnormal handling of the
// plain form that a normal argument with a normal reciprocal never needs.
__device__ __forceinline__ float rcp_approx_normal(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float log1p_unit(float u)
{
    const float t = __fadd_rn(2.0f, u);
    const float r = rcp_approx_normal(t);
    const float q0 = __fmul_rn(u, r);
    const float s = __fmaf_rn(__fmaf_rn(-q0, t, u), r, q0);
    const float z = __fmul_rn(s, s);
    const float p = series_tail(z);
    const float two_s = __fmul_rn(2.0f, s);
    return __fmaf_rn(__fmul_rn(two_s, z), p, two_s);
}

// The merge where d = lo - hi is NaN, i.e. a NaN operand or two equal
// infinities: the infinity itself, else NaN.  Every other non-finite case
// falls out of the arithmetic: an infinite difference (an infinite operand,
// or lo - hi overflowing) gives e^d = 0 and the sum hi + 0.
__device__ __forceinline__ float lse_merge_nan_d(float a, float b)
{
    return a == b ? a : __int_as_float(0x7fc00000);
}

// log(e^a + e^b) as hi + log1p(exp(lo - hi)), exp by the CUDA intrinsic
// __expf (at most 2 + floor(1.173 |d|) ulp from e^d; scaled by
// e^d / (1 + e^d), an absolute error below 2^-23 in the sum, like the
// accurate expf's); both -inf gives -inf, +inf wins, NaN propagates.
// d = lo - hi is taken as -|RN(a - b)|: rounding is symmetric, so that is
// RN(lo - hi) (up to the sign of a zero difference, which only exp sees);
// hi = max(a, b).  A NaN operand or two equal infinities make d NaN.
__device__ __forceinline__ float lse_merge1(float a, float b)
{
    const float hi = fmaxf(a, b);
    const float d = -fabsf(__fsub_rn(a, b));
    if (isnan(d))
        return lse_merge_nan_d(a, b);
    return __fadd_rn(hi, log1p_unit(__expf(d)));
}

// Two merges at once: the same operations as lse_merge1 for each element,
// the element-wise steps on packed pairs (each lane the IEEE operation, so
// each element's bits are lse_merge1's).
__device__ __forceinline__ void lse_merge2(float a0, float a1, float b0, float b1, float& r0, float& r1)
{
    const float hi0 = fmaxf(a0, b0), hi1 = fmaxf(a1, b1);
    float e0d, e1d;
    sub2_rn(a0, a1, b0, b1, e0d, e1d);
    const float d0 = -fabsf(e0d), d1 = -fabsf(e1d);
    const float u0 = __expf(d0), u1 = __expf(d1);
    float t0, t1, q0, q1, s0, s1;
    add2_rn(2.0f, 2.0f, u0, u1, t0, t1);
    const float c0 = rcp_approx_normal(t0), c1 = rcp_approx_normal(t1);
    mul2_rn(u0, u1, c0, c1, q0, q1);
    const float e0 = __fmaf_rn(-q0, t0, u0), e1 = __fmaf_rn(-q1, t1, u1);
    fma2_rn(e0, e1, c0, c1, q0, q1, s0, s1);
    float z0, z1;
    mul2_rn(s0, s1, s0, s1, z0, z1);
    float p0 = 0x1.3b13b2p-4f, p1 = 0x1.3b13b2p-4f;
    fma2_rn(p0, p1, z0, z1, 0x1.745d18p-4f, 0x1.745d18p-4f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.c71c72p-4f, 0x1.c71c72p-4f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.24924ap-3f, 0x1.24924ap-3f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.99999ap-3f, 0x1.99999ap-3f, p0, p1);
    fma2_rn(p0, p1, z0, z1, 0x1.555556p-2f, 0x1.555556p-2f, p0, p1);
    float w0, w1, v0, v1, l0, l1;
    mul2_rn(2.0f, 2.0f, s0, s1, w0, w1);
    mul2_rn(w0, w1, z0, z1, v0, v1);
    fma2_rn(v0, v1, p0, p1, w0, w1, l0, l1);
    add2_rn(hi0, hi1, l0, l1, r0, r1);
    // d0, d1 <= 0 (or NaN), so their sum is NaN exactly when one of them is
    if (isnan(__fadd_rn(d0, d1))) {
        if (isnan(d0))
            r0 = lse_merge_nan_d(a0, b0);
        if (isnan(d1))
            r1 = lse_merge_nan_d(a1, b1);
    }
}

__device__ __forceinline__ float unary1(float x, int op)
{
    return op == 0 ? log1pf(x) : op == 1 ? coshf(x) : expf(x);
}

// Grid strides ahead of its loads at which a merge CTA prefetches a unit
// into L2.
constexpr int64_t kLseL2Ahead = 1;

// Rows of n_cols elements; a unit is `blockDim.x * VEC` consecutive columns
// of one row, units_per_row of them per row; the grid strides over units
// (in row-major unit order).  In a whole unit of 16-byte aligned rows
// (vec4: every base address 16-byte aligned and every row stride a
// multiple of 4, checked by the host) with VEC >= 4, thread t handles the
// four-column groups t + k * blockDim.x, k < VEC / 4 (16-byte loads and
// stores); otherwise columns t + v * blockDim.x, v < VEC.  Which thread
// handles a column never changes its arithmetic.
template <int VEC>
__global__ void __launch_bounds__(1024) lse_merge_kernel(float* out, int64_t out_stride, const float* a,
                                                         int64_t a_stride, const float* b, int64_t b_stride,
                                                         int64_t n_rows, int64_t n_cols, int vec4,
                                                         int l2_prefetch)
{
    const int64_t span = static_cast<int64_t>(blockDim.x) * VEC;
    const int64_t units_per_row = (n_cols + span - 1) / span;
    if (l2_prefetch && vec4 && threadIdx.x == 0) {
        // The CTA's first unit of a and b, into L2 while the previous grid
        // finishes (a hint; the loads come after the wait).  Whole 16-byte
        // pieces inside the row only.
        const int64_t row = blockIdx.x / units_per_row;
        const int64_t base = (blockIdx.x - row * units_per_row) * span;
        const int64_t end = base + span < n_cols ? base + span : n_cols;
        const uint32_t bytes = static_cast<uint32_t>(((end - base) * 4) & ~int64_t{15});
        if (row < n_rows && bytes > 0) {
            prefetch_l2(a + row * a_stride + base, bytes);
            prefetch_l2(b + row * b_stride + base, bytes);
        }
    }
    wait_prior_grids();
    allow_next_grid();
    // unit u = row * units_per_row + cb, walked with a stride of gridDim.x:
    // (row, cb) advances by (gridDim.x / units_per_row, gridDim.x %
    // units_per_row) with a carry, so the loop divides only once here
    const int64_t step_rows = gridDim.x / units_per_row;
    const int64_t step_cb = gridDim.x - step_rows * units_per_row;
    int64_t row = blockIdx.x / units_per_row;
    int64_t cb = blockIdx.x - row * units_per_row;
    // The unit kLseL2Ahead grid strides ahead, walked the same way: thread 0
    // prefetches it into L2 (a hint; whole 16-byte units of device memory
    // only), so more bytes are on their way than the registers hold.  Only
    // thread 0 pays for locating it.
    const int64_t first_ahead = static_cast<int64_t>(blockIdx.x) + kLseL2Ahead * static_cast<int64_t>(gridDim.x);
    const bool ahead_on =
        l2_prefetch && vec4 && threadIdx.x == 0 && kLseL2Ahead > 0 && first_ahead < n_rows * units_per_row;
    int64_t ahead_row = n_rows, ahead_cb = 0;
    if (ahead_on) {
        ahead_row = first_ahead / units_per_row;
        ahead_cb = first_ahead - ahead_row * units_per_row;
    }
    for (; row < n_rows; row += step_rows) {
        if (ahead_on) {
            if (ahead_row < n_rows && ahead_cb * span + span <= n_cols) {
                prefetch_l2(a + ahead_row * a_stride + ahead_cb * span, static_cast<uint32_t>(span * 4));
                prefetch_l2(b + ahead_row * b_stride + ahead_cb * span, static_cast<uint32_t>(span * 4));
            }
            ahead_row += step_rows;
            ahead_cb += step_cb;
            if (ahead_cb >= units_per_row) {
                ahead_cb -= units_per_row;
                ++ahead_row;
            }
        }
        const int64_t base = cb * span;
        const float* ar = a + row * a_stride + base;
        const float* br = b + row * b_stride + base;
        float* orow = out + row * out_stride + base;
        if (VEC >= 4 && vec4 && base + span <= n_cols) {
            constexpr int G = VEC >= 4 ? VEC / 4 : 1;
            float4 va[G], vb[G];
#pragma unroll
            for (int k = 0; k < G; ++k) {
                va[k] = __ldcs(reinterpret_cast<const float4*>(ar) + threadIdx.x + k * blockDim.x);
                vb[k] = __ldcs(reinterpret_cast<const float4*>(br) + threadIdx.x + k * blockDim.x);
            }
#pragma unroll
            for (int k = 0; k < G; ++k) {
                float4 r;
                lse_merge2(va[k].x, va[k].y, vb[k].x, vb[k].y, r.x, r.y);
                lse_merge2(va[k].z, va[k].w, vb[k].z, vb[k].w, r.z, r.w);
                __stcs(reinterpret_cast<float4*>(orow) + threadIdx.x + k * blockDim.x, r);
            }
        } else {
            const int64_t lim = n_cols - base;
            float va[VEC], vb[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const int64_t c = threadIdx.x + static_cast<int64_t>(v) * blockDim.x;
                if (c < lim) {
                    va[v] = __ldcs(ar + c);
                    vb[v] = __ldcs(br + c);
                }
            }
            if constexpr (VEC == 1) {
                if (threadIdx.x < lim)
                    __stcs(orow + threadIdx.x, lse_merge1(va[0], vb[0]));
            } else {
#pragma unroll
                for (int v = 0; v < VEC; v += 2) {
                    const int64_t c = threadIdx.x + static_cast<int64_t>(v) * blockDim.x;
                    const int64_t c1 = c + blockDim.x;
                    float r0, r1;
                    lse_merge2(va[v], va[v + 1], vb[v], vb[v + 1], r0, r1);
                    if (c < lim)
                        __stcs(orow + c, r0);
                    if (c1 < lim)
                        __stcs(orow + c1, r1);
                }
            }
        }
        cb += step_cb;
        if (cb >= units_per_row) {
            cb -= units_per_row;
            ++row;
        }
    }
}

// The same unit walk over one flat array (vec4: both base addresses 16-byte
// aligned).
template <int VEC>
__global__ void __launch_bounds__(1024) unary_kernel(float* out, const float* x, int64_t n, int op, int vec4,
                                                     int l2_prefetch)
{
    const int64_t span = static_cast<int64_t>(blockDim.x) * VEC;
    if (l2_prefetch && vec4 && threadIdx.x == 0) {
        const int64_t base = static_cast<int64_t>(blockIdx.x) * span;
        const int64_t end = base + span < n ? base + span : n;
        if (base < n) {
            const uint32_t bytes = static_cast<uint32_t>(((end - base) * 4) & ~int64_t{15});
            if (bytes > 0)
                prefetch_l2(x + base, bytes);
        }
    }
    wait_prior_grids();
    allow_next_grid();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * span;
    // As in the merge: thread 0 prefetches the whole unit kLseL2Ahead grid
    // strides ahead into L2.
    const bool ahead_on = l2_prefetch && vec4 && threadIdx.x == 0 && kLseL2Ahead > 0;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * span; base < n; base += stride) {
        if (ahead_on) {
            const int64_t ahead = base + kLseL2Ahead * stride;
            if (ahead < n && span <= n - ahead)
                prefetch_l2(x + ahead, static_cast<uint32_t>(span * 4));
        }
        const float* xr = x + base;
        float* orow = out + base;
        if (VEC >= 4 && vec4 && base + span <= n) {
            constexpr int G = VEC >= 4 ? VEC / 4 : 1;
            float4 vx[G];
#pragma unroll
            for (int k = 0; k < G; ++k)
                vx[k] = __ldcs(reinterpret_cast<const float4*>(xr) + threadIdx.x + k * blockDim.x);
#pragma unroll
            for (int k = 0; k < G; ++k) {
                const float4 r = make_float4(unary1(vx[k].x, op), unary1(vx[k].y, op), unary1(vx[k].z, op),
                                             unary1(vx[k].w, op));
                __stcs(reinterpret_cast<float4*>(orow) + threadIdx.x + k * blockDim.x, r);
            }
        } else {
            const int64_t lim = n - base;
            float vx[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const int64_t i = threadIdx.x + static_cast<int64_t>(v) * blockDim.x;
                if (i < lim)
                    vx[v] = __ldcs(xr + i);
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const int64_t i = threadIdx.x + static_cast<int64_t>(v) * blockDim.x;
                if (i < lim)
                    __stcs(orow + i, unary1(vx[v], op));
            }
        }
    }
}

cudaError_t launch_lse_merge(float* out, int64_t out_stride, const float* a, int64_t a_stride, const float* b,
                             int64_t b_stride, int64_t n_rows, int64_t n_cols, int vec, bool vec4,
                             bool l2_prefetch, int grid, int threads, bool serialize, cudaStream_t stream)
{
    void (*fn)(float*, int64_t, const float*, int64_t, const float*, int64_t, int64_t, int64_t, int, int) =
        vec == 1 ? lse_merge_kernel<1> : vec == 2 ? lse_merge_kernel<2> : vec == 4 ? lse_merge_kernel<4>
        : vec == 8 ? lse_merge_kernel<8> : nullptr;
    if (!fn)
        return cudaErrorInvalidValue;
    return launch(fn, grid, threads, 0, serialize, stream, out, out_stride, a, a_stride, b, b_stride, n_rows,
                  n_cols, vec4 ? 1 : 0, l2_prefetch ? 1 : 0);
}

cudaError_t launch_unary(float* out, const float* x, int64_t n, int op, int vec, bool vec4, bool l2_prefetch,
                         int grid, int threads, bool serialize, cudaStream_t stream)
{
    void (*fn)(float*, const float*, int64_t, int, int, int) = vec == 1 ? unary_kernel<1> : vec == 2 ? unary_kernel<2>
                                                     : vec == 4 ? unary_kernel<4> : vec == 8 ? unary_kernel<8>
                                                                                             : nullptr;
    if (!fn)
        return cudaErrorInvalidValue;
    return launch(fn, grid, threads, 0, serialize, stream, out, x, n, op, vec4 ? 1 : 0, l2_prefetch ? 1 : 0);
}

}  // namespace dradd
