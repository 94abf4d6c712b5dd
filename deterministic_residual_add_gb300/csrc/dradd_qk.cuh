// dradd_qk.cuh -- the fused q/k RMSNorm kernel templates: two row sets in
// one launch, the q side optionally with per-group e4m3 out; each side runs
// either tile_body, which stages groups of rows_per_cta adjacent rows into
// shared memory with one bulk copy per tensor, or rows_body_contig, which
// loads rows straight into registers with the contiguous thread-to-block
// mapping.  Instantiated by the dradd_qk_<out>_<variant>.cu translation
// units.
#pragma once

#include "dradd_kernels.cuh"
#include "dradd_warp.cuh"

namespace dradd {

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
        // While the previous grid finishes: L2 prefetches of this CTA's
        // first groups (about 16 KiB of input); the copies that consume
        // them come after the wait and read what the memory holds then.
        if (p.l2_prefetch) {
            const uint32_t ahead = stage_bytes < kL2PrefetchBytes ? kL2PrefetchBytes / stage_bytes : 1u;
            for (uint32_t a = 0; a < ahead; ++a) {
                const int64_t row0 = (cta + static_cast<int64_t>(a) * n_ctas) * R;
                if (row0 >= p.n_rows)
                    break;
                const int64_t left = p.n_rows - row0;
                const uint32_t bytes = row_bytes * static_cast<uint32_t>(left < R ? left : R);
                prefetch_l2(p.x + row0 * p.hidden, bytes);
                if constexpr (ADD)
                    prefetch_l2(p.residual + row0 * p.hidden, bytes);
            }
        }
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
                drain_issued_copies(p, bars, s, parity, i, stages, cta, n_ctas, n_groups);
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

// Row steps ahead of its loads at which a register-variant CTA prefetches
// its rows into L2.
constexpr int64_t kQkL2Ahead = 4;

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

    if (p.l2_prefetch && tid == 0) {
        // The CTA's first rows (about 16 KiB of input; adjacent rows), into
        // L2 while the previous grid finishes; the loads come after the wait.
        const uint32_t row_bytes = static_cast<uint32_t>(p.hidden) * 2u;
        const uint32_t step_bytes = (ADD ? 2u : 1u) * row_bytes * static_cast<uint32_t>(p.rows_per_cta);
        const uint32_t ahead = step_bytes < kL2PrefetchBytes ? kL2PrefetchBytes / step_bytes : 1u;
        for (uint32_t a = 0; a < ahead; ++a) {
            const int64_t row0 = (cta + static_cast<int64_t>(a) * n_ctas) * p.rows_per_cta;
            if (row0 >= p.n_rows)
                break;
            const int64_t left = p.n_rows - row0;
            const uint32_t bytes = row_bytes * static_cast<uint32_t>(left < p.rows_per_cta ? left : p.rows_per_cta);
            prefetch_l2(p.x + row0 * p.hidden, bytes);
            if constexpr (ADD)
                prefetch_l2(p.residual + row0 * p.hidden, bytes);
        }
    }
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
        if (p.l2_prefetch && tid == 0) {
            // the CTA's rows kQkL2Ahead steps ahead, into L2 (a hint: the
            // registers already hold the next step's rows)
            const int64_t ahead = base + kQkL2Ahead * rows_per_step;
            if (ahead < p.n_rows) {
                const int64_t left = p.n_rows - ahead;
                const uint32_t bytes = static_cast<uint32_t>(p.hidden) * 2u *
                                       static_cast<uint32_t>(left < p.rows_per_cta ? left : p.rows_per_cta);
                prefetch_l2(p.x + ahead * p.hidden, bytes);
                if constexpr (ADD)
                    prefetch_l2(p.residual + ahead * p.hidden, bytes);
            }
        }
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

// ------------------------------------------------------------- qk_warp_kernel
// Fused q/k RMSNorm, one warp per row (warp_ring_body): CTAs [0, q_ctas)
// take the q rows, the rest the k rows, each side with its own rings and
// weights (dynamic shared memory: the larger side's warp_smem_bytes).
template <int KQ, int KK, bool QQUANT, bool QADD>
__global__ void __launch_bounds__(256, 1) qk_warp_kernel(const Params pq, const Params pk, int q_ctas)
{
    extern __shared__ __align__(128) unsigned char wsm[];
    constexpr int QOUT = QQUANT ? kOutE4m3Group : kOutBf16;
    const int cta = static_cast<int>(blockIdx.x);
    if (cta < q_ctas)
        warp_ring_body<KQ, QOUT, QADD>(pq, cta, q_ctas, wsm);
    else
        warp_ring_body<KK, kOutBf16, false>(pk, cta - q_ctas, static_cast<int64_t>(gridDim.x) - q_ctas, wsm);
}

template <bool QQUANT, bool QADD>
QkKernelFn qk_warp_table(int kq, int kk)
{
#define DRADD_QK_WARP_KK(KQV)                                         \
    switch (kk) {                                                     \
    case 1: return qk_warp_kernel<KQV, 1, QQUANT, QADD>;              \
    case 2: return qk_warp_kernel<KQV, 2, QQUANT, QADD>;              \
    case 4: return qk_warp_kernel<KQV, 4, QQUANT, QADD>;              \
    case 8: return qk_warp_kernel<KQV, 8, QQUANT, QADD>;              \
    default: return nullptr;                                          \
    }
    switch (kq) {
    case 1: DRADD_QK_WARP_KK(1)
    case 2: DRADD_QK_WARP_KK(2)
    case 4: DRADD_QK_WARP_KK(4)
    case 8: DRADD_QK_WARP_KK(8)
    default: return nullptr;
    }
#undef DRADD_QK_WARP_KK
}

// ----------------------------------------------------------- qk_chunk_kernel
// Fused q/k RMSNorm with the q rows in 512-element chunks (chunk_row_body,
// one warp a chunk, a CTA a row) and the k rows one warp each
// (warp_ring_body): CTAs [0, q_ctas) take the q rows, the rest the k rows;
// both kinds have the q row's chunk count of warps.  Compiled for at least
// three resident CTAs of up to 256 threads (72 registers, no spills:
// 4096 x 3072 q + 1024 k 25.39 -> 23.13 us against the unbounded 86).
template <int KK, bool QQUANT, bool QADD>
__global__ void __launch_bounds__(256, 3) qk_chunk_kernel(const Params pq, const Params pk, int q_ctas)
{
    extern __shared__ __align__(128) unsigned char wsm[];
    constexpr int QOUT = QQUANT ? kOutE4m3Group : kOutBf16;
    const int cta = static_cast<int>(blockIdx.x);
    if (cta < q_ctas)
        chunk_row_body<QOUT, QADD>(pq, cta, q_ctas, wsm);
    else
        warp_ring_body<KK, kOutBf16, false>(pk, cta - q_ctas, static_cast<int64_t>(gridDim.x) - q_ctas, wsm);
}

template <bool QQUANT, bool QADD>
QkKernelFn qk_chunk_table(int kk)
{
    switch (kk) {
    case 1: return qk_chunk_kernel<1, QQUANT, QADD>;
    case 2: return qk_chunk_kernel<2, QQUANT, QADD>;
    case 4: return qk_chunk_kernel<4, QQUANT, QADD>;
    case 8: return qk_chunk_kernel<8, QQUANT, QADD>;
    default: return nullptr;
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
