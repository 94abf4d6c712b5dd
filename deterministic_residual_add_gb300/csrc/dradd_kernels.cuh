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
//   qk_kernel      fused q/k RMSNorm: two row sets in one launch, the q side
//                  optionally with per-group e4m3 out; each side runs either
//                  the rows_kernel body or tile_body, which stages groups of
//                  rows_per_cta adjacent rows into shared memory with one
//                  bulk copy per tensor.
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
        const float scale = __fdiv_rn(m, OUT == kOutInt8 ? 127.0f : OUT == kOutE4m3 ? 448.0f : 6.0f);
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

// acc for K blocks from already loaded vectors (x + residual with ADD, x
// alone otherwise); with ADD residual_out is stored in the same pass.
// Returns the per-block partial sums of squares.
template <int K, bool ADD>
__device__ __forceinline__ void row_accumulate(const Params& p, const uint4 (&xv)[K], const uint4 (&rv)[K],
                                               float (&acc)[K][8], float (&part)[K], int64_t row,
                                               bool active, int t, int T, int nblocks)
{
    uint4* rorow = ADD ? reinterpret_cast<uint4*>(p.residual_out + row * p.hidden) : nullptr;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int b = t + j * T;
        if (active && b < nblocks) {
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

// -------------------------------------------------------------- staged_kernel
// T (threads per row = threads per CTA) is a compile-time constant so that
// every (T, K) pair gets its own register budget (staged_min_blocks) and the
// reduction widths fold away.  A stage holds one row of x, then (with ADD)
// one row of residual.
template <int T, int K, int OUT, bool ADD>
__global__ void __launch_bounds__(T, staged_min_blocks(T, K)) staged_kernel(const Params p)
{
    static_assert(T >= 32 && T <= 1024 && (T & (T - 1)) == 0, "T: a power of two, 32..1024");
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ float s_sum[2][32 * K];
    __shared__ float s_max[2][32];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp_in_row = tid >> 5;
    const int nblocks = p.hidden >> 3;
    const int stages = p.stages;
    const uint32_t row_bytes = static_cast<uint32_t>(p.hidden) * 2u;
    const uint32_t stage_bytes = (ADD ? 2u : 1u) * row_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage_mem + static_cast<size_t>(stages) * stage_bytes);
    const int64_t stride = gridDim.x;

    if (tid == 0) {
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

    uint4 w[K];
    load_weights<K>(p, w, tid, T, nblocks);

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
            if (b < nblocks) {
                xv[j] = xs[b];
                if constexpr (ADD)
                    rv[j] = rs[b];
            }
        }
        float acc[K][8], part[K];
        row_accumulate<K, ADD>(p, xv, rv, acc, part, row, true, tid, T, nblocks);

        float* red = &s_sum[buf][0];
        lanes_then_publish<K>(part, T, lane, warp_in_row, red);
        // Every thread has read stage s (so it can be refilled) and published
        // its warp's partial sums; any expired wait ends the CTA here.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                record_timeout(p);
                // Copies already issued must land before shared memory is released.
                int s2 = s;
                uint32_t parity2 = parity;
                for (int64_t i2 = i; i2 < i + stages; ++i2) {
                    if (blockIdx.x + i2 * stride >= p.n_rows)
                        break;
                    if (!(p.fault_inject && i2 == 0))
                        mbar_wait_bounded(&bars[s2], parity2, p.wait_limit_ns);
                    if (++s2 == stages) {
                        s2 = 0;
                        parity2 ^= 1u;
                    }
                }
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
        gather_warps<K>(part, T, lane, red);
        const float inv = inv_rms(fold_k<K>(part), p.hidden, p.inv_hidden, p.eps);
        finish_row<K, OUT>(p, acc, w, inv, row, true, tid, T, lane, warp_in_row, nblocks,
                             &s_max[buf][0]);
        buf ^= 1;
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
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

// --------------------------------------------------------------- split_kernel
// A cluster of C CTAs shares each row: CTA rank r of the cluster owns the
// r-th of C equal slices of the padded row (P / C elements, an aligned
// subtree of the canonical tree), stages its slice of x (and residual) with
// 1-D bulk copies `stages` rows ahead, and reduces it as staged_kernel
// reduces a whole row (T threads, K blocks of 8 per thread).  The C slice
// sums meet through distributed shared memory after a cluster barrier and
// are folded as the top levels of the tree ((S0 + S1) for C = 2,
// (S0 + S1) + (S2 + S3) for C = 4), so the bits equal every other variant's.
// Rows go round-robin over the clusters.  A timed-out wait is made known to
// the whole cluster at that barrier, and every CTA then drains its copies
// and leaves after one more cluster barrier: every CTA of a cluster always
// runs the same number of cluster barriers.  bf16 output.
template <int T, int K, int C, bool ADD>
__global__ void __launch_bounds__(T, staged_min_blocks(T, K)) split_kernel(const Params p)
{
    static_assert(C == 2 || C == 4, "cluster of 2 or 4 CTAs");
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ float s_sum[2][32 * K];
    __shared__ float s_max[2][32];
    __shared__ float s_part[2][2];  // [buffer][slice sum, timeout flag]
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp_in_row = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const int64_t first_row = cluster_id_x();
    const int64_t n_clusters = cluster_count_x();
    constexpr int kSliceElems = 8 * T * K;
    const int slice_off = static_cast<int>(rank) * kSliceElems;
    int valid = p.hidden - slice_off;
    valid = valid < 0 ? 0 : (valid > kSliceElems ? kSliceElems : valid);
    const int nblocks = valid >> 3;
    const int stages = p.stages;
    const uint32_t slice_bytes = static_cast<uint32_t>(valid) * 2u;
    constexpr uint32_t kStageBytes = (ADD ? 2u : 1u) * kSliceElems * 2u;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage_mem + static_cast<size_t>(stages) * kStageBytes);
    // this slice's view of the outputs and the weight
    Params ps = p;
    ps.out = p.out + slice_off;
    ps.weight = p.weight + slice_off;
    if constexpr (ADD)
        ps.residual_out = p.residual_out + slice_off;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    wait_prior_grids();
    allow_next_grid();

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int s, int64_t row) {
        unsigned char* dst = stage_mem + static_cast<size_t>(s) * kStageBytes;
        mbar_arrive_expect_tx(&bars[s], (ADD ? 2u : 1u) * slice_bytes);
        if (slice_bytes) {
            bulk_copy_g2s(dst, p.x + row * p.hidden + slice_off, slice_bytes, &bars[s], policy);
            if constexpr (ADD)
                bulk_copy_g2s(dst + kSliceElems * 2, p.residual + row * p.hidden + slice_off, slice_bytes, &bars[s],
                              policy);
        }
    };
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t row = first_row + s * n_clusters;
            if (row >= p.n_rows)
                break;
            if (p.fault_inject && s == 0)
                continue;  // test hook: this copy never comes, so its wait expires
            issue(s, row);
        }
    }

    uint4 w[K];
    load_weights<K>(ps, w, tid, T, nblocks);

    int buf = 0;
    int64_t i = 0;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t row = first_row; row < p.n_rows; row += n_clusters, ++i) {
        const bool ok = mbar_wait_bounded(&bars[s], parity, p.wait_limit_ns);
        const unsigned char* sbase = stage_mem + static_cast<size_t>(s) * kStageBytes;
        const uint4* xs = reinterpret_cast<const uint4*>(sbase);
        const uint4* rs = reinterpret_cast<const uint4*>(sbase + kSliceElems * 2);
        uint4 xv[K], rv[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = tid + j * T;
            if (b < nblocks) {
                xv[j] = xs[b];
                if constexpr (ADD)
                    rv[j] = rs[b];
            }
        }
        float acc[K][8], part[K];
        row_accumulate<K, ADD>(ps, xv, rv, acc, part, row, true, tid, T, nblocks);

        float* red = &s_sum[buf][0];
        lanes_then_publish<K>(part, T, lane, warp_in_row, red);
        const bool bad = __syncthreads_or(!ok);
        gather_warps<K>(part, T, lane, red);
        const float slice_sum = fold_k<K>(part);
        if (tid == 0) {
            s_part[buf][0] = slice_sum;
            s_part[buf][1] = bad ? 1.0f : 0.0f;
        }
        cluster_sync_all();
        float sums[C];
        float flags = 0.0f;
#pragma unroll
        for (int r = 0; r < C; ++r) {
            sums[r] = ld_cluster_f32(&s_part[buf][0], static_cast<uint32_t>(r));
            flags = __fadd_rn(flags, ld_cluster_f32(&s_part[buf][1], static_cast<uint32_t>(r)));
        }
        if (flags != 0.0f) {
            // some CTA of the cluster gave up waiting: all of them leave here
            if (tid == 0) {
                if (bad)
                    record_timeout(p);
                // Copies already issued (rows i .. i + stages - 1; none was
                // issued for a stage after its wait) must land before shared
                // memory is released.
                int s2 = s;
                uint32_t parity2 = parity;
                for (int64_t i2 = i; i2 < i + stages; ++i2) {
                    if (first_row + i2 * n_clusters >= p.n_rows)
                        break;
                    if (!(p.fault_inject && i2 == 0))
                        mbar_wait_bounded(&bars[s2], parity2, p.wait_limit_ns);
                    if (++s2 == stages) {
                        s2 = 0;
                        parity2 ^= 1u;
                    }
                }
            }
            cluster_sync_all();  // no CTA leaves while another may read its shared memory
            return;
        }
        // every CTA has read stage s and every wait succeeded: refill it
        if (tid == 0) {
            const int64_t next = row + static_cast<int64_t>(stages) * n_clusters;
            if (next < p.n_rows) {
                fence_proxy_async_smem();
                issue(s, next);
            }
        }
        float total;
        if constexpr (C == 2)
            total = __fadd_rn(sums[0], sums[1]);
        else
            total = __fadd_rn(__fadd_rn(sums[0], sums[1]), __fadd_rn(sums[2], sums[3]));
        const float inv = inv_rms(total, p.hidden, p.inv_hidden, p.eps);
        finish_row<K, kOutBf16>(ps, acc, w, inv, row, true, tid, T, lane, warp_in_row, nblocks, &s_max[buf][0]);
        buf ^= 1;
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
    cluster_sync_all();  // the last row's slice sums may still be read by other CTAs
}

template <int T, int K, int C, bool ADD>
KernelFn split_pick()
{
    if constexpr (T <= max_threads_for(K))
        return split_kernel<T, K, C, ADD>;
    else
        return nullptr;
}

template <int T, int C, bool ADD>
KernelFn split_by_k(int K)
{
    switch (K) {
    case 1: return split_pick<T, 1, C, ADD>();
    case 2: return split_pick<T, 2, C, ADD>();
    case 4: return split_pick<T, 4, C, ADD>();
    case 8: return split_pick<T, 8, C, ADD>();
    default: return nullptr;
    }
}

template <int C, bool ADD>
KernelFn split_table(int T, int K)
{
    switch (T) {
    case 32: return split_by_k<32, C, ADD>(K);
    case 64: return split_by_k<64, C, ADD>(K);
    case 128: return split_by_k<128, C, ADD>(K);
    case 256: return split_by_k<256, C, ADD>(K);
    case 512: return split_by_k<512, C, ADD>(K);
    case 1024: return split_by_k<1024, C, ADD>(K);
    default: return nullptr;
    }
}

// ----------------------------------------------------------------- tile_body
// Staged body for rows of any width: R = rows_per_cta consecutive rows form
// a group, T = threads_per_row threads per row (T x R = the CTA), K blocks
// of 8 per thread.  A stage holds one group: its R rows of x (and then its
// R rows of residual) arrive by one 1-D bulk copy each, since the rows of
// a group are adjacent in memory; the last group of the tensor may be
// short, and its copies carry only the rows that exist.  Groups cta,
// cta + n_ctas, ... are this CTA's; the copy for the group `stages` ahead
// is issued as soon as every thread has read the current stage.  Waits are
// bounded as in staged_kernel.
template <int K, int OUT, bool ADD>
__device__ __forceinline__ void tile_body(const Params& p, int64_t cta, int64_t n_ctas,
                                          unsigned char* stage_mem)
{
    __shared__ float s_sum[2][32 * K];
    __shared__ float s_max[2][32];
    const int T = p.threads_per_row;
    const int R = p.rows_per_cta;
    const int tid = threadIdx.x;
    const int r_local = tid / T;
    const int t = tid - r_local * T;
    const int lane = tid & 31;
    const int warp_in_row = t >> 5;
    const int warps_per_row = T > 32 ? T >> 5 : 1;
    const int nblocks = p.hidden >> 3;
    const int stages = p.stages;
    const uint32_t row_bytes = static_cast<uint32_t>(p.hidden) * 2u;
    const uint32_t tile_bytes = row_bytes * static_cast<uint32_t>(R);
    const uint32_t stage_bytes = (ADD ? 2u : 1u) * tile_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage_mem + static_cast<size_t>(stages) * stage_bytes);
    const int64_t n_groups = (p.n_rows + R - 1) / R;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    wait_prior_grids();
    allow_next_grid();

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int s, int64_t g) {
        const int64_t row0 = g * R;
        const int64_t left = p.n_rows - row0;
        const uint32_t bytes = row_bytes * static_cast<uint32_t>(left < R ? left : R);
        unsigned char* dst = stage_mem + static_cast<size_t>(s) * stage_bytes;
        mbar_arrive_expect_tx(&bars[s], (ADD ? 2u : 1u) * bytes);
        bulk_copy_g2s(dst, p.x + row0 * p.hidden, bytes, &bars[s], policy);
        if constexpr (ADD)
            bulk_copy_g2s(dst + tile_bytes, p.residual + row0 * p.hidden, bytes, &bars[s], policy);
    };
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t g = cta + s * n_ctas;
            if (g >= n_groups)
                break;
            if (p.fault_inject && s == 0)
                continue;  // test hook: this copy never comes, so its wait expires
            issue(s, g);
        }
    }

    uint4 w[K];
    load_weights<K>(p, w, t, T, nblocks);

    int buf = 0;
    int64_t i = 0;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t g = cta; g < n_groups; g += n_ctas, ++i) {
        const bool ok = mbar_wait_bounded(&bars[s], parity, p.wait_limit_ns);
        const int64_t row = g * R + r_local;
        const bool active = row < p.n_rows;
        const unsigned char* sbase =
            stage_mem + static_cast<size_t>(s) * stage_bytes + static_cast<size_t>(r_local) * row_bytes;
        const uint4* xs = reinterpret_cast<const uint4*>(sbase);
        const uint4* rs = reinterpret_cast<const uint4*>(sbase + tile_bytes);
        uint4 xv[K], rv[K];
        if (active) {
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = t + j * T;
                if (b < nblocks) {
                    xv[j] = xs[b];
                    if constexpr (ADD)
                        rv[j] = rs[b];
                }
            }
        }
        float acc[K][8], part[K];
        row_accumulate<K, ADD>(p, xv, rv, acc, part, row, active, t, T, nblocks);

        float* red = &s_sum[buf][r_local * warps_per_row * K];
        lanes_then_publish<K>(part, T, lane, warp_in_row, red);
        // Every thread has read stage s and published its warp's partial
        // sums; any expired wait ends the CTA here.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                record_timeout(p);
                // Copies already issued must land before shared memory is released.
                int s2 = s;
                uint32_t parity2 = parity;
                for (int64_t i2 = i; i2 < i + stages; ++i2) {
                    if (cta + i2 * n_ctas >= n_groups)
                        break;
                    if (!(p.fault_inject && i2 == 0))
                        mbar_wait_bounded(&bars[s2], parity2, p.wait_limit_ns);
                    if (++s2 == stages) {
                        s2 = 0;
                        parity2 ^= 1u;
                    }
                }
            }
            return;
        }
        if (tid == 0) {
            const int64_t next = g + static_cast<int64_t>(stages) * n_ctas;
            if (next < n_groups) {
                fence_proxy_async_smem();
                issue(s, next);
            }
        }
        gather_warps<K>(part, T, lane, red);
        const float inv = inv_rms(fold_k<K>(part), p.hidden, p.inv_hidden, p.eps);
        finish_row<K, OUT>(p, acc, w, inv, row, active, t, T, lane, warp_in_row, nblocks,
                             &s_max[buf][r_local * warps_per_row]);
        buf ^= 1;
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
}

// ----------------------------------------------------------- rows_body_contig
// The register-load body with the contiguous mapping: thread t of a row owns
// the K adjacent blocks tK .. tK + K - 1, an aligned subtree of 8K elements
// of the canonical tree.  The thread folds its K block sums first (fold_k
// pairs adjacent blocks), then one butterfly over the row's lanes and, past
// 32 threads, one over its warps: the same tree, so the same bits as the
// strided mapping.  A lane's 16-byte loads stride K x 16 bytes across the
// warp; the neighbouring halves of each 32-byte sector arrive with the
// thread's next block.  Each thread loads its blocks of the next row while
// it computes the current one.  For the per-group e4m3 output a group (gb blocks,
// gb >= K, both powers of two) is held whole by gb / K adjacent lanes, so
// its max takes log2(gb / K) shuffles and its scale is computed once per
// thread rather than once per block.  bf16 or per-group e4m3 out.
template <int K, int OUT, bool ADD>
__device__ __forceinline__ void rows_body_contig(const Params& p, int64_t cta, int64_t n_ctas)
{
    static_assert(OUT == kOutBf16 || OUT == kOutE4m3Group, "bf16 or per-group e4m3 out");
    __shared__ float s_sum[2][32];
    const int T = p.threads_per_row;
    const int tid = threadIdx.x;
    const int r_local = tid / T;
    const int t = tid - r_local * T;
    const int lane = tid & 31;
    const int warp_in_row = t >> 5;
    const int warps_per_row = T > 32 ? T >> 5 : 1;
    const int nblocks = p.hidden >> 3;
    const int b0 = t * K;

    wait_prior_grids();
    allow_next_grid();
    uint4 w[K];
    {
        const uint4* wrow = reinterpret_cast<const uint4*>(p.weight);
#pragma unroll
        for (int j = 0; j < K; ++j)
            w[j] = b0 + j < nblocks ? __ldg(wrow + b0 + j) : make_uint4(0u, 0u, 0u, 0u);
    }

    const int64_t rows_per_step = n_ctas * p.rows_per_cta;
    // The next row's vectors are loaded while this row is computed (one
    // row of prefetch in registers).
    auto load_row = [&](int64_t row, uint4 (&xv)[K], uint4 (&rv)[K]) {
        if (row >= p.n_rows)
            return;
        const uint4* xrow = reinterpret_cast<const uint4*>(p.x + row * p.hidden);
        const uint4* rrow = ADD ? reinterpret_cast<const uint4*>(p.residual + row * p.hidden) : nullptr;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (b0 + j < nblocks) {
                xv[j] = ld_stream(xrow + b0 + j);
                if constexpr (ADD)
                    rv[j] = ld_stream(rrow + b0 + j);
            }
        }
    };
    uint4 xv[K], rv[K], nxv[K], nrv[K];
    load_row(cta * p.rows_per_cta + r_local, nxv, nrv);
    int buf = 0;
    for (int64_t base = cta * p.rows_per_cta; base < p.n_rows; base += rows_per_step) {
        const int64_t row = base + r_local;
        const bool active = row < p.n_rows;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            xv[j] = nxv[j];
            rv[j] = nrv[j];
        }
        load_row(row + rows_per_step, nxv, nrv);
        float acc[K][8], part[K];
        uint4* rorow = ADD ? reinterpret_cast<uint4*>(p.residual_out + row * p.hidden) : nullptr;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (active && b0 + j < nblocks) {
                if constexpr (ADD) {
                    add8(xv[j], rv[j], acc[j]);
                    st_stream(rorow + b0 + j, pack8_rne(acc[j]));
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
        float sum = butterfly_sum(fold_k<K>(part), T < 32 ? T : 32);
        if (T > 32) {
            float* red = &s_sum[buf][r_local * warps_per_row];
            if (lane == 0)
                red[warp_in_row] = sum;
            __syncthreads();
            sum = butterfly_sum(red[lane & (warps_per_row - 1)], warps_per_row);
        }
        const float inv = inv_rms(sum, p.hidden, p.inv_hidden, p.eps);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (b0 + j >= nblocks)
                continue;
            scale8(acc[j], inv, w[j]);
        }
        if constexpr (OUT == kOutBf16) {
            if (active) {
                uint4* orow = reinterpret_cast<uint4*>(p.out + row * p.hidden);
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (b0 + j < nblocks)
                        st_stream(orow + b0 + j, pack8_rne(acc[j]));
            }
        } else {
            const int lanes = p.group_blocks / K;  // lanes per group, a power of two >= 1
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < K; ++j) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    m = fmaxf(m, fabsf(acc[j][e]));
            }
            m = butterfly_max(m, lanes);
            const float scale = div448_rn(m);
            if (active && b0 < nblocks) {
                const int64_t groups = nblocks >> p.group_shift;
                if ((t & (lanes - 1)) == 0)
                    p.scale[row * groups + (b0 >> p.group_shift)] = scale;
                const E4m3Scale qs = make_e4m3_scale(scale);
                uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (b0 + j < nblocks)
                        st_stream(qrow + b0 + j, quantize8_e4m3(acc[j], qs));
            }
        }
        buf ^= 1;
    }
}

// ------------------------------------------------------------------ qk_kernel
// Fused q/k RMSNorm in one launch: CTAs [0, q_ctas) run the q rows (residual
// add with QADD; per-group e4m3 out with QQUANT, else bf16), the rest the k
// rows (plain, bf16).  Both sides use the CTA's threads, each with its own
// threads per row, rows per CTA and blocks per thread; STAGED selects
// tile_body (bulk copies into shared memory, `stages` groups ahead) over
// rows_body_contig (loads straight into registers, contiguous mapping).
template <int KQ, int KK, bool QQUANT, bool QADD, bool STAGED>
__global__ void __launch_bounds__(qk_max_threads(KQ > KK ? KQ : KK))
    qk_kernel(const Params pq, const Params pk, int q_ctas)
{
    extern __shared__ __align__(128) unsigned char stage_mem[];
    constexpr int QOUT = QQUANT ? kOutE4m3Group : kOutBf16;
    const int cta = static_cast<int>(blockIdx.x);
    const int k_ctas = static_cast<int>(gridDim.x) - q_ctas;
    if constexpr (STAGED) {
        if (cta < q_ctas)
            tile_body<KQ, QOUT, QADD>(pq, cta, q_ctas, stage_mem);
        else
            tile_body<KK, kOutBf16, false>(pk, cta - q_ctas, k_ctas, stage_mem);
    } else {
        if (cta < q_ctas)
            rows_body_contig<KQ, QOUT, QADD>(pq, cta, q_ctas);
        else
            rows_body_contig<KK, kOutBf16, false>(pk, cta - q_ctas, k_ctas);
    }
}

template <int KQ, bool QQUANT, bool QADD, bool STAGED>
QkKernelFn qk_by_kk(int kk)
{
    switch (kk) {
    case 1: return qk_kernel<KQ, 1, QQUANT, QADD, STAGED>;
    case 2: return qk_kernel<KQ, 2, QQUANT, QADD, STAGED>;
    case 4: return qk_kernel<KQ, 4, QQUANT, QADD, STAGED>;
    case 8: return qk_kernel<KQ, 8, QQUANT, QADD, STAGED>;
    default: return nullptr;
    }
}

template <bool QQUANT, bool QADD, bool STAGED>
QkKernelFn qk_table(int kq, int kk)
{
    switch (kq) {
    case 1: return qk_by_kk<1, QQUANT, QADD, STAGED>(kk);
    case 2: return qk_by_kk<2, QQUANT, QADD, STAGED>(kk);
    case 4: return qk_by_kk<4, QQUANT, QADD, STAGED>(kk);
    case 8: return qk_by_kk<8, QQUANT, QADD, STAGED>(kk);
    default: return nullptr;
    }
}

}  // namespace dradd
