// dradd_kernels.cuh -- the kernel templates for the fused residual-add +
// RMSNorm forward (bf16 out and per-row int8 out) and for plain RMSNorm, on
// sm_103a.  Instantiated by the dradd_*.cu translation units.
//
// The operation (ROCm/aiter issue #5151, "Steps to Reproduce", reference()):
//   acc = fp32(x) + fp32(residual); residual_out = bf16_rne(acc);
//   out = bf16_rne((acc * (1 / sqrt(S / hidden + eps))) * fp32(weight)),
// where S is the canonical pairwise sum of acc^2 over the row zero-padded to
// P = next power of two >= hidden.  With ADD = false the residual is absent:
// acc = fp32(x) (exact) and there is no residual_out (plain RMSNorm).
//
// Work layout shared by both kernels.  A row is split into 8-element blocks
// (one 16-byte vector each), P / 8 of them counting the padding.  The T
// threads of a row own K = P / (8 T) blocks each, thread t holding blocks
// t, t + T, ..., t + (K - 1) T, so consecutive threads touch consecutive
// 16-byte vectors (fully coalesced for every K).  The canonical tree then
// factors exactly:
//   levels 1-3   inside each 8-block, in registers            (fold8_squares)
//   next log2 T  across the T threads for each j: lanes by xor butterfly,
//                then warps through shared memory and a second butterfly
//   top log2 K   across the K subtrees a thread holds          (fold_k)
// Each stage adds adjacent aligned blocks, lower + upper, so the sum equals
// the tree over the padded row whatever T, K, rows per CTA or grid are; the
// padding blocks contribute +0 and adding +0 to a sum of squares is exact.
//
// Kernels:
//   rows_kernel    rows are loaded straight into registers with streaming
//                  16-byte loads; a CTA handles rows_per_cta rows side by side
//                  and loops over the rows with a grid stride.
// The fused q/k kernels (dradd_qk.cuh) and the split-row cluster kernel
// (dradd_split.cuh) build on the helpers here.
//   staged_kernel  persistent CTAs stage whole rows of x (and residual) into
//                  shared memory with 1-D bulk asynchronous copies (TMA
//                  engine), `stages` rows ahead of the compute; the copy for
//                  row i + stages is issued as soon as row i has been read.
//                  Every wait on a copy is bounded: past the limit the CTA
//                  records a timeout in the device status word, waits (again
//                  bounded) for its other copies and returns.
#pragma once

#include "dradd_device.cuh"
#include "dradd_internal.h"

namespace dradd {

// ------------------------------------------------------------------ helpers
// Sum of one row across its T threads for each of the K subtrees: lanes
// first, then (T > 32) each warp's lane 0 publishes its sums in `red` (W * K
// floats for this row); the caller puts a CTA-wide barrier between this and
// gather_warps.
template <int K>
__device__ __forceinline__ void lanes_then_publish(float (&part)[K], int T, int lane, int warp_in_row,
                                                   float* red)
{
    const int width = T < 32 ? T : 32;
#pragma unroll
    for (int j = 0; j < K; ++j)
        part[j] = butterfly_sum(part[j], width);
    if (T > 32 && lane == 0) {
#pragma unroll
        for (int j = 0; j < K; ++j)
            red[warp_in_row * K + j] = part[j];
    }
}

template <int K>
__device__ __forceinline__ void gather_warps(float (&part)[K], int T, int lane, const float* red)
{
    if (T <= 32)
        return;
    const int W = T >> 5;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const float v = red[(lane & (W - 1)) * K + j];
        part[j] = butterfly_sum(v, W);
    }
}

// Row epilogue after inv is known: bf16 store, or the per-row int8 / e4m3
// codes (which need their own CTA-wide max).  Called by every thread of the
// CTA.
template <int K, int OUT>
__device__ __forceinline__ void finish_row(const Params& p, float (&acc)[K][8], const uint4 (&w)[K],
                                           float inv, int64_t row, bool active, int t, int T, int lane,
                                           int warp_in_row, int nblocks, float* red_max)
{
    // Padding blocks (t + jT >= nblocks) keep acc = 0 and are never stored;
    // a warp whose blocks for some j are all padding skips that j.
#pragma unroll
    for (int j = 0; j < K; ++j) {
        if (t + j * T >= nblocks)
            continue;
        scale8(acc[j], inv, w[j]);
    }
    if constexpr (OUT == kOutBf16) {
        if (active) {
            uint4* orow = reinterpret_cast<uint4*>(p.out + row * p.hidden);
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = t + j * T;
                if (b < nblocks)
                    st_stream(orow + b, pack8_rne(acc[j]));
            }
        }
    } else if constexpr (OUT == kOutE4m3Group) {
        // A group is gb consecutive blocks, gb a power of two <= min(T, 32)
        // that divides nblocks.  Block t + jT belongs to group (t + jT) / gb,
        // and since gb divides T the gb lanes of an aligned lane group hold
        // one group for every j: its amax is their butterfly max (exact,
        // so independent of the order).  Padding blocks form whole groups
        // of their own and are never stored.
        const int gb = p.group_blocks;
        const int gshift = p.group_shift;
        const int64_t groups = nblocks >> gshift;
        uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            // with T >= 32 a warp lies inside one row: warp-uniform skip
            if (T >= 32 && (t & ~31) + j * T >= nblocks)
                continue;
            float m = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                m = fmaxf(m, fabsf(acc[j][e]));
            m = butterfly_max(m, gb);
            const float scale = div448_rn(m);
            const int b = t + j * T;
            if (active && b < nblocks) {
                if ((b & (gb - 1)) == 0)
                    p.scale[row * groups + (b >> gshift)] = scale;
                st_stream(qrow + b, quantize8_e4m3(acc[j], make_e4m3_scale(scale)));
            }
        }
    } else {
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                m = fmaxf(m, fabsf(acc[j][e]));
        }
        m = butterfly_max(m, T < 32 ? T : 32);
        if (T > 32) {
            if (lane == 0)
                red_max[warp_in_row] = m;
            __syncthreads();
            m = butterfly_max(red_max[lane & ((T >> 5) - 1)], T >> 5);
        }
        const float scale = div_const_rn<quant_divisor(OUT)>(m);
        if (active) {
            if (t == 0)
                p.scale[row] = scale;
            uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
            if constexpr (OUT == kOutE2m1) {
                // two codes per byte: a row is hidden / 2 bytes, a block 4 bytes
                uint32_t* prow = reinterpret_cast<uint32_t*>(p.out_q + row * (p.hidden / 2));
                const E4m3Scale qs = make_e4m3_scale(scale);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const int b = t + j * T;
                    if (b < nblocks)
                        __stcs(prow + b, quantize8_e2m1(acc[j], qs));
                }
            } else if constexpr (OUT == kOutInt8) {
                const QuantScale qs = make_quant_scale(scale);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const int b = t + j * T;
                    if (b < nblocks)
                        st_stream(qrow + b, quantize8(acc[j], qs));
                }
            } else {
                const E4m3Scale qs = make_e4m3_scale(scale);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const int b = t + j * T;
                    if (b < nblocks)
                        st_stream(qrow + b, quantize8_e4m3(acc[j], qs));
                }
            }
        }
    }
}

// The weight blocks a thread needs, kept as packed bf16 (4 registers per
// 8 weights) for the whole life of the CTA.
template <int K>
__device__ __forceinline__ void load_weights(const Params& p, uint4 (&w)[K], int t, int T, int nblocks)
{
    const uint4* wrow = reinterpret_cast<const uint4*>(p.weight);
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int b = t + j * T;
        w[j] = b < nblocks ? __ldg(wrow + b) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Whether block b = t + j * T (j unrolled) of a thread lies in the row, for
// a kernel whose T threads of K blocks cover the padded row exactly (T * K =
// P / 8 blocks).  P is the next power of two >= hidden, so nblocks > P / 16
// = T * K / 2: blocks j < K / 2 (b <= T * K / 2 - 1) always lie in the row
// and only the others need the test (with K = 1, every block does).
template <int K>
__device__ __forceinline__ bool block_in_row(int j, int b, int nblocks)
{
    return 2 * (j + 1) <= K || b < nblocks;
}

// acc for K blocks from already loaded vectors (x + residual with ADD, x
// alone otherwise); with ADD residual_out is stored in the same pass.
// Returns the per-block partial sums of squares.  COVERS: the caller's T
// threads of K blocks cover the padded row exactly (block_in_row applies).
template <int K, bool ADD, bool COVERS = false>
__device__ __forceinline__ void row_accumulate(const Params& p, const uint4 (&xv)[K], const uint4 (&rv)[K],
                                               float (&acc)[K][8], float (&part)[K], int64_t row,
                                               bool active, int t, int T, int nblocks)
{
    uint4* rorow = ADD ? reinterpret_cast<uint4*>(p.residual_out + row * p.hidden) : nullptr;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int b = t + j * T;
        if (active && (COVERS ? block_in_row<K>(j, b, nblocks) : b < nblocks)) {
            if constexpr (ADD) {
                add8(xv[j], rv[j], acc[j]);
                st_stream(rorow + b, pack8_rne(acc[j]));
            } else {
                unpack8(xv[j], acc[j]);
            }
            part[j] = fold8_squares(acc[j]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[j][e] = 0.0f;
            part[j] = 0.0f;
        }
    }
}

__device__ __forceinline__ void record_timeout(const Params& p)
{
    atomicOr(p.status, kDeviceStatusTimeout);
}

// After an expired wait, thread 0 of a staged CTA waits for every bulk copy
// the CTA has issued and not yet consumed: iterations i .. i + stages - 1
// (stage s onwards, phase parity `parity`) whose unit first + i2 * stride
// is below n_units; with fault_inject the copy of iteration 0 was never
// issued.  A copy that has not landed within the wait limit gets up to
// kDrainRounds limits in all, so that none lands in shared memory after
// the CTA has exited; one still missing then is recorded as
// kDeviceStatusUndrained (every wait stays bounded).
constexpr int kDrainRounds = 8;

__device__ __forceinline__ void drain_issued_copies(const Params& p, uint64_t* bars, int s, uint32_t parity,
                                                    int64_t i, int stages, int64_t first, int64_t stride,
                                                    int64_t n_units)
{
    for (int64_t i2 = i; i2 < i + stages; ++i2) {
        if (first + i2 * stride >= n_units)
            break;
        if (!(p.fault_inject && i2 == 0)) {
            bool landed = false;
            for (int r = 0; r < kDrainRounds && !landed; ++r)
                landed = mbar_wait_bounded(&bars[s], parity, p.wait_limit_ns);
            if (!landed)
                atomicOr(p.status, kDeviceStatusUndrained);
        }
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
}

// ---------------------------------------------------------------- rows_kernel
// The CTA numbered `cta` of `n_ctas` handles row groups cta, cta + n_ctas, ...
template <int K, int OUT, bool ADD>
__device__ __forceinline__ void rows_body(const Params& p, int64_t cta, int64_t n_ctas)
{
    __shared__ float s_sum[2][32 * K];
    __shared__ float s_max[2][32];
    const int T = p.threads_per_row;
    const int tid = threadIdx.x;
    const int r_local = tid / T;
    const int t = tid - r_local * T;
    const int lane = tid & 31;
    const int warp_in_row = t >> 5;
    const int warps_per_row = T > 32 ? T >> 5 : 1;
    const int nblocks = p.hidden >> 3;

    wait_prior_grids();
    allow_next_grid();
    uint4 w[K];
    load_weights<K>(p, w, t, T, nblocks);

    const int64_t rows_per_step = n_ctas * p.rows_per_cta;
    int buf = 0;
    for (int64_t base = cta * p.rows_per_cta; base < p.n_rows;
         base += rows_per_step) {
        const int64_t row = base + r_local;
        const bool active = row < p.n_rows;
        uint4 xv[K], rv[K];
        if (active) {
            const uint4* xrow = reinterpret_cast<const uint4*>(p.x + row * p.hidden);
            const uint4* rrow = ADD ? reinterpret_cast<const uint4*>(p.residual + row * p.hidden) : nullptr;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = t + j * T;
                if (b < nblocks) {
                    xv[j] = ld_stream(xrow + b);
                    if constexpr (ADD)
                        rv[j] = ld_stream(rrow + b);
                }
            }
        }
        float acc[K][8], part[K];
        row_accumulate<K, ADD>(p, xv, rv, acc, part, row, active, t, T, nblocks);

        float* red = &s_sum[buf][r_local * warps_per_row * K];
        lanes_then_publish<K>(part, T, lane, warp_in_row, red);
        if (T > 32)
            __syncthreads();
        gather_warps<K>(part, T, lane, red);
        const float inv = inv_rms(fold_k<K>(part), p.hidden, p.inv_hidden, p.eps);
        finish_row<K, OUT>(p, acc, w, inv, row, active, t, T, lane, warp_in_row, nblocks,
                             &s_max[buf][r_local * warps_per_row]);
        buf ^= 1;
    }
}

template <int K, int OUT, bool ADD>
__global__ void __launch_bounds__(max_threads_for(K)) rows_kernel(const Params p)
{
    rows_body<K, OUT, ADD>(p, blockIdx.x, gridDim.x);
}

// Input bytes per CTA prefetched into L2 before the wait for the previous
// grid (whole rows, at least one): with 4 CTAs per SM about 10 MB per
// launch, what the previous grid's last rows leave room for.  Measured on
// GB300 at 4096 x 4096: one row of x and residual per CTA (16 KiB) gave
// 5708 -> 6405 GB/s with 2 stages at 2048 rows, 5715 -> 6810 GB/s for the
// plain RMSNorm with two rows of x; deeper prefetches slowed the calls.
constexpr uint32_t kL2PrefetchBytes = 16384;

// -------------------------------------------------------------- staged_kernel
// This thread's part of a row's amax, reduced over its warp: int8 with NaN
// propagation (a row holding a NaN y shows as a NaN amax and takes the exact
// path, whose amax ignores NaN); the other formats ignore NaN, as a running
// max from 0.
template <int K, int OUT>
__device__ __forceinline__ float quant_warp_amax(const float (&y)[K][8])
{
    if constexpr (OUT == kOutInt8)
        return warp_max_nan(tree_max_abs<K, true>(y));
    else
        return warp_max(fmaxf(0.0f, tree_max_abs<K, false>(y)));
}

// The CTA-wide amax from the W warps' values in red (lane l reads warp
// l mod W; with W == 1, m is already the row's).
template <int W, int OUT>
__device__ __forceinline__ float quant_cta_amax(float m, const float* red, int lane)
{
    if constexpr (W > 1)
        return OUT == kOutInt8 ? warp_max_nan(red[lane & (W - 1)]) : warp_max(red[lane & (W - 1)]);
    else
        return m;
}

// Per-row scale and codes of the quantised outputs (one row per T threads,
// compile-time; T threads of K blocks cover the padded row), given the
// row's amax m over the CTA.  Called by every thread of the CTA: an int8
// row whose amax is NaN takes a second, NaN-ignoring amax through red_max2
// (W floats of its own) and a barrier.
template <int T, int K, int OUT>
__device__ __forceinline__ void quant_row_finish(const Params& p, const float (&y)[K][8], float m, int64_t row,
                                                 int tid, int lane, int warp, int nblocks, float* red_max2)
{
    constexpr int W = T / 32;
    if constexpr (OUT == kOutInt8) {
        uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
        if (!isnan(m)) {
            const float scale = div_const_rn<127>(m);
            if (tid == 0)
                p.scale[row] = scale;
            const Int8Bracket qs = make_int8_bracket(scale);
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = tid + j * T;
                if (block_in_row<K>(j, b, nblocks)) {
                    uint32_t differ = 0u;
                    uint2 code = quantize8_bracket(y[j], qs, differ);
                    if (!qs.fast || differ != 0u)
                        code = quantize8_exact(y[j], scale);
                    st_stream(qrow + b, code);
                }
            }
        } else {
            // uniform over the CTA: every thread holds the same m
            float m2 = warp_max(fmaxf(0.0f, tree_max_abs<K, false>(y)));  // NaN ignored, as a running max from 0
            if constexpr (W > 1) {
                if (lane == 0)
                    red_max2[warp] = m2;
                __syncthreads();
                m2 = warp_max(red_max2[lane & (W - 1)]);
            }
            const float scale = div_const_rn<127>(m2);
            if (tid == 0)
                p.scale[row] = scale;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = tid + j * T;
                if (block_in_row<K>(j, b, nblocks))
                    st_stream(qrow + b, quantize8_exact(y[j], scale));
            }
        }
    } else {
        const float scale = div_const_rn<quant_divisor(OUT)>(m);
        if (tid == 0)
            p.scale[row] = scale;
        const E4m3Scale qs = make_e4m3_scale(scale);
        if constexpr (OUT == kOutE2m1) {
            // two codes per byte: a row is hidden / 2 bytes, a block 4 bytes
            uint32_t* prow = reinterpret_cast<uint32_t*>(p.out_q + row * (p.hidden / 2));
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = tid + j * T;
                if (block_in_row<K>(j, b, nblocks))
                    __stcs(prow + b, quantize8_e2m1(y[j], qs));
            }
        } else {
            uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = tid + j * T;
                if (block_in_row<K>(j, b, nblocks))
                    st_stream(qrow + b, quantize8_e4m3(y[j], qs));
            }
        }
    }
}

// Per-row scale and codes of the quantised outputs in the staged kernel
// (one row per CTA, T threads, compile-time): the row's amax over the CTA,
// then the codes of each of the thread's blocks.
template <int T, int K, int OUT>
__device__ __forceinline__ void staged_quant_row(const Params& p, const float (&y)[K][8], int64_t row, int tid,
                                                 int lane, int warp, int nblocks, float* red_max,
                                                 float* red_max2)
{
    constexpr int W = T / 32;
    float m = quant_warp_amax<K, OUT>(y);
    if constexpr (W > 1) {
        if (lane == 0)
            red_max[warp] = m;
        __syncthreads();
    }
    m = quant_cta_amax<W, OUT>(m, red_max, lane);
    quant_row_finish<T, K, OUT>(p, y, m, row, tid, lane, warp, nblocks, red_max2);
}

// T (threads per row = threads per CTA) is a compile-time constant so that
// every (T, K) pair gets its own register budget (staged_min_blocks) and the
// reduction widths fold away.  A stage holds one row of x, then (with ADD)
// one row of residual.  The row's sum of squares: each thread's K block sums
// go through warp_halving_sum, then (T > 32) lanes 0 .. K - 1 of each warp
// publish their subtree sums and cross_warp_sum finishes the tree.  The
// quantised outputs read their weights as fp32 from shared memory (widened
// once per CTA, each thread its own blocks: w_lo holds elements 0-3 of
// every block, w_hi elements 4-7, so a warp's 16-byte reads are
// consecutive); bf16 out keeps them packed in registers.
template <int T, int K, int OUT, bool ADD>
__global__ void __launch_bounds__(T, staged_min_blocks(T, K)) staged_kernel(const Params p)
{
    static_assert(T >= 32 && T <= 1024 && (T & (T - 1)) == 0, "T: a power of two, 32..1024");
    constexpr int W = T / 32;
    constexpr bool kWsm = OUT != kOutBf16;
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ float s_sum[2][K * W];
    __shared__ float s_max[2][W];
    __shared__ float s_max2[W];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nblocks = p.hidden >> 3;
    const int stages = p.stages;
    const uint32_t row_bytes = static_cast<uint32_t>(p.hidden) * 2u;
    const uint32_t stage_bytes = (ADD ? 2u : 1u) * row_bytes;
    unsigned char* const after_stages = stage_mem + static_cast<size_t>(stages) * stage_bytes;
    float4* const w_lo = reinterpret_cast<float4*>(after_stages);
    float4* const w_hi = w_lo + nblocks;
    uint64_t* bars = reinterpret_cast<uint64_t*>(after_stages + staged_weight_bytes(OUT, p.hidden));
    const int64_t stride = gridDim.x;

    if (tid == 0) {
        // While the previous grid finishes: L2 prefetches of this CTA's
        // first rows.  The copies that consume them are issued after the
        // wait below, and read what the memory holds then.
        const uint32_t ahead =
            !p.l2_prefetch ? 0u : (stage_bytes < kL2PrefetchBytes ? kL2PrefetchBytes / stage_bytes : 1u);
        for (uint32_t s = 0; s < ahead; ++s) {
            const int64_t row = blockIdx.x + static_cast<int64_t>(s) * stride;
            if (row >= p.n_rows)
                break;
            prefetch_l2(p.x + row * p.hidden, row_bytes);
            if constexpr (ADD)
                prefetch_l2(p.residual + row * p.hidden, row_bytes);
        }
        for (int s = 0; s < stages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    wait_prior_grids();
    allow_next_grid();

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int s, int64_t row) {
        unsigned char* dst = stage_mem + static_cast<size_t>(s) * stage_bytes;
        mbar_arrive_expect_tx(&bars[s], stage_bytes);
        bulk_copy_g2s(dst, p.x + row * p.hidden, row_bytes, &bars[s], policy);
        if constexpr (ADD)
            bulk_copy_g2s(dst + row_bytes, p.residual + row * p.hidden, row_bytes, &bars[s], policy);
    };
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t row = blockIdx.x + s * stride;
            if (row >= p.n_rows)
                break;
            if (p.fault_inject && s == 0)
                continue;  // test hook: this copy never comes, so its wait expires
            issue(s, row);
        }
    }

    uint4 w[kWsm ? 1 : K];
    if constexpr (kWsm) {
        // each thread widens the weights of its own blocks (and only it
        // reads them, so no barrier is needed)
        const uint4* wrow = reinterpret_cast<const uint4*>(p.weight);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = tid + j * T;
            if (block_in_row<K>(j, b, nblocks)) {
                float f[8];
                unpack8(__ldg(wrow + b), f);
                w_lo[b] = make_float4(f[0], f[1], f[2], f[3]);
                w_hi[b] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    } else {
        load_weights<K>(p, w, tid, T, nblocks);
    }

    int buf = 0;
    // Iteration i of this CTA uses stage s = i mod stages and waits for phase
    // parity floor(i / stages) mod 2; both are kept incrementally.
    int64_t i = 0;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t row = blockIdx.x; row < p.n_rows; row += stride, ++i) {
        // A thread whose wait gives up goes on with whatever the stage holds
        // (outputs are unspecified after a timeout); the CTA learns of it at
        // the barrier below and stops there, before refilling any stage.
        const bool ok = mbar_wait_bounded(&bars[s], parity, p.wait_limit_ns);
        const unsigned char* sbase = stage_mem + static_cast<size_t>(s) * stage_bytes;
        const uint4* xs = reinterpret_cast<const uint4*>(sbase);
        const uint4* rs = reinterpret_cast<const uint4*>(sbase + row_bytes);
        uint4 xv[K], rv[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = tid + j * T;
            if (block_in_row<K>(j, b, nblocks)) {
                xv[j] = xs[b];
                if constexpr (ADD)
                    rv[j] = rs[b];
            }
        }
        float acc[K][8], part[K];
        row_accumulate<K, ADD, true>(p, xv, rv, acc, part, row, true, tid, T, nblocks);

        int jsub;
        float v = warp_halving_sum<K>(part, lane, jsub);
        if constexpr (W > 1) {
            if (lane < K)
                s_sum[buf][jsub * W + warp] = v;
        }
        // Every thread has read stage s (so it can be refilled) and published
        // its warp's subtree sums; any expired wait ends the CTA here.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                record_timeout(p);
                // Copies already issued must land before shared memory is released.
                drain_issued_copies(p, bars, s, parity, i, stages, blockIdx.x, stride, p.n_rows);
            }
            return;
        }
        if (tid == 0) {
            const int64_t next = row + static_cast<int64_t>(stages) * stride;
            if (next < p.n_rows) {
                fence_proxy_async_smem();
                issue(s, next);
            }
        }
        float sum;
        if constexpr (W > 1)
            sum = cross_warp_sum<K, W>(s_sum[buf], lane);
        else
            sum = fold_lane_subtrees<K>(v);
        const float inv = inv_rms(sum, p.hidden, p.inv_hidden, p.eps);
        if constexpr (kWsm) {
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = tid + j * T;
                if (block_in_row<K>(j, b, nblocks))
                    scale8_f32(acc[j], inv, w_lo[b], w_hi[b]);
            }
            staged_quant_row<T, K, OUT>(p, acc, row, tid, lane, warp, nblocks, s_max[buf], s_max2);
        } else {
            finish_row<K, OUT>(p, acc, w, inv, row, true, tid, T, lane, warp, nblocks, &s_max[buf][0]);
        }
        buf ^= 1;
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
}

// ---------------------------------------------------------- staged_pair_kernel
// The plain RMSNorm with quantised out, two rows per thread: a unit is the
// pair of adjacent rows 2u, 2u + 1 (the last alone when n_rows is odd),
// staged by one bulk copy, and every thread carries both rows through the
// same steps as staged_kernel, so one barrier serves both rows' sums and one
// both rows' amax, and the two rows' dependent chains interleave.  Each row
// gets exactly the arithmetic of staged_kernel (same tree, same epilogue).
template <int T, int K, int OUT>
__global__ void __launch_bounds__(T, staged_min_blocks(T, 2 * K)) staged_pair_kernel(const Params p)
{
    static_assert(T >= 32 && T <= 1024 && (T & (T - 1)) == 0, "T: a power of two, 32..1024");
    static_assert(OUT != kOutBf16, "quantised outputs only");
    constexpr int W = T / 32;
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ float s_sum[2][2][K * W];
    __shared__ float s_max[2][2][W];
    __shared__ float s_max2[2][W];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nblocks = p.hidden >> 3;
    const int stages = p.stages;
    const uint32_t row_bytes = static_cast<uint32_t>(p.hidden) * 2u;
    const uint32_t stage_bytes = 2u * row_bytes;
    unsigned char* const after_stages = stage_mem + static_cast<size_t>(stages) * stage_bytes;
    float4* const w_lo = reinterpret_cast<float4*>(after_stages);
    float4* const w_hi = w_lo + nblocks;
    uint64_t* bars = reinterpret_cast<uint64_t*>(after_stages + staged_weight_bytes(OUT, p.hidden));
    const int64_t stride = gridDim.x;
    const int64_t n_units = (p.n_rows + 1) / 2;

    // bytes of unit u: one or two rows
    auto unit_bytes = [&](int64_t u) -> uint32_t {
        return 2 * u + 1 < p.n_rows ? stage_bytes : row_bytes;
    };
    if (tid == 0) {
        if (p.l2_prefetch && static_cast<int64_t>(blockIdx.x) < n_units)
            prefetch_l2(p.x + 2 * static_cast<int64_t>(blockIdx.x) * p.hidden, unit_bytes(blockIdx.x));
        for (int s = 0; s < stages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    wait_prior_grids();
    allow_next_grid();

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int s, int64_t u) {
        const uint32_t bytes = unit_bytes(u);
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_copy_g2s(stage_mem + static_cast<size_t>(s) * stage_bytes, p.x + 2 * u * p.hidden, bytes, &bars[s],
                      policy);
    };
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t u = blockIdx.x + s * stride;
            if (u >= n_units)
                break;
            if (p.fault_inject && s == 0)
                continue;  // test hook: this copy never comes, so its wait expires
            issue(s, u);
        }
    }
    {
        // each thread widens the weights of its own blocks (only it reads them)
        const uint4* wrow = reinterpret_cast<const uint4*>(p.weight);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = tid + j * T;
            if (block_in_row<K>(j, b, nblocks)) {
                float f[8];
                unpack8(__ldg(wrow + b), f);
                w_lo[b] = make_float4(f[0], f[1], f[2], f[3]);
                w_hi[b] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    }

    int buf = 0;
    int64_t i = 0;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t u = blockIdx.x; u < n_units; u += stride, ++i) {
        const bool ok = mbar_wait_bounded(&bars[s], parity, p.wait_limit_ns);
        const int64_t row0 = 2 * u;
        const bool two = row0 + 1 < p.n_rows;  // uniform over the CTA
        const uint4* xs0 = reinterpret_cast<const uint4*>(stage_mem + static_cast<size_t>(s) * stage_bytes);
        const uint4* xs1 = xs0 + (row_bytes >> 4);
        float a0[K][8], a1[K][8], part0[K], part1[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = tid + j * T;
            if (block_in_row<K>(j, b, nblocks)) {
                unpack8(xs0[b], a0[j]);
                part0[j] = fold8_squares(a0[j]);
                if (two) {
                    unpack8(xs1[b], a1[j]);
                    part1[j] = fold8_squares(a1[j]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        a1[j][e] = 0.0f;
                    part1[j] = 0.0f;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    a0[j][e] = 0.0f;
                    a1[j][e] = 0.0f;
                }
                part0[j] = 0.0f;
                part1[j] = 0.0f;
            }
        }
        int jsub0, jsub1;
        const float v0 = warp_halving_sum<K>(part0, lane, jsub0);
        const float v1 = warp_halving_sum<K>(part1, lane, jsub1);
        if constexpr (W > 1) {
            if (lane < K) {
                s_sum[buf][0][jsub0 * W + warp] = v0;
                s_sum[buf][1][jsub1 * W + warp] = v1;
            }
        }
        // Every thread has read stage s (so it can be refilled) and published
        // its warps' subtree sums; any expired wait ends the CTA here.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                record_timeout(p);
                drain_issued_copies(p, bars, s, parity, i, stages, blockIdx.x, stride, n_units);
            }
            return;
        }
        if (tid == 0) {
            const int64_t next = u + static_cast<int64_t>(stages) * stride;
            if (next < n_units) {
                fence_proxy_async_smem();
                issue(s, next);
            }
        }
        float sum0, sum1;
        if constexpr (W > 1) {
            sum0 = cross_warp_sum<K, W>(s_sum[buf][0], lane);
            sum1 = cross_warp_sum<K, W>(s_sum[buf][1], lane);
        } else {
            sum0 = fold_lane_subtrees<K>(v0);
            sum1 = fold_lane_subtrees<K>(v1);
        }
        const float inv0 = inv_rms(sum0, p.hidden, p.inv_hidden, p.eps);
        const float inv1 = inv_rms(sum1, p.hidden, p.inv_hidden, p.eps);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = tid + j * T;
            if (block_in_row<K>(j, b, nblocks)) {
                const float4 wl = w_lo[b], wh = w_hi[b];
                scale8_f32(a0[j], inv0, wl, wh);
                scale8_f32(a1[j], inv1, wl, wh);
            }
        }
        float m0 = quant_warp_amax<K, OUT>(a0);
        float m1 = quant_warp_amax<K, OUT>(a1);
        if constexpr (W > 1) {
            if (lane == 0) {
                s_max[buf][0][warp] = m0;
                s_max[buf][1][warp] = m1;
            }
            __syncthreads();
        }
        m0 = quant_cta_amax<W, OUT>(m0, s_max[buf][0], lane);
        m1 = quant_cta_amax<W, OUT>(m1, s_max[buf][1], lane);
        quant_row_finish<T, K, OUT>(p, a0, m0, row0, tid, lane, warp, nblocks, s_max2[0]);
        if (two)
            quant_row_finish<T, K, OUT>(p, a1, m1, row0 + 1, tid, lane, warp, nblocks, s_max2[1]);
        buf ^= 1;
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
}

template <int T, int K, int OUT>
KernelFn staged_pair_pick()
{
    if constexpr (T <= max_threads_for(2 * K))
        return staged_pair_kernel<T, K, OUT>;
    else
        return nullptr;
}

// Pair kernels for T = 32..512 and K in {1, 2, 4} (two rows' accumulators
// per thread, so the register budget of 2 K blocks).
template <int OUT>
KernelFn staged_pair_table(int T, int K)
{
#define DRADD_PAIR_K(TT)                                   \
    switch (K) {                                           \
    case 1: return staged_pair_pick<TT, 1, OUT>();         \
    case 2: return staged_pair_pick<TT, 2, OUT>();         \
    case 4: return staged_pair_pick<TT, 4, OUT>();         \
    default: return nullptr;                               \
    }
    switch (T) {
    case 32: DRADD_PAIR_K(32)
    case 64: DRADD_PAIR_K(64)
    case 128: DRADD_PAIR_K(128)
    case 256: DRADD_PAIR_K(256)
    case 512: DRADD_PAIR_K(512)
    default: return nullptr;
    }
#undef DRADD_PAIR_K
}

// ------------------------------------------------------- staged kernel table
// Staged kernels exist for T = 32..1024 and K in {1, 2, 4, 8} with
// T <= max_threads_for(K); each translation unit instantiates one (OUT, ADD).
template <int T, int K, int OUT, bool ADD>
KernelFn staged_pick()
{
    if constexpr (T <= max_threads_for(K))
        return staged_kernel<T, K, OUT, ADD>;
    else
        return nullptr;
}

template <int T, int OUT, bool ADD>
KernelFn staged_by_k(int K)
{
    switch (K) {
    case 1: return staged_pick<T, 1, OUT, ADD>();
    case 2: return staged_pick<T, 2, OUT, ADD>();
    case 4: return staged_pick<T, 4, OUT, ADD>();
    case 8: return staged_pick<T, 8, OUT, ADD>();
    default: return nullptr;
    }
}

template <int OUT, bool ADD>
KernelFn staged_table(int T, int K)
{
    switch (T) {
    case 32: return staged_by_k<32, OUT, ADD>(K);
    case 64: return staged_by_k<64, OUT, ADD>(K);
    case 128: return staged_by_k<128, OUT, ADD>(K);
    case 256: return staged_by_k<256, OUT, ADD>(K);
    case 512: return staged_by_k<512, OUT, ADD>(K);
    case 1024: return staged_by_k<1024, OUT, ADD>(K);
    default: return nullptr;
    }
}

}  // namespace dradd
