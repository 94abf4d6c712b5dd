// dradd_split.cuh -- the split-row kernel template: a thread-block cluster
// of 2 or 4 CTAs shares each row, the slice sums meeting in distributed
// shared memory.  Instantiated by dradd_split_<mode>.cu.
#pragma once

#include "dradd_kernels.cuh"

namespace dradd {

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
                drain_issued_copies(p, bars, s, parity, i, stages, first_row, n_clusters, p.n_rows);
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

}  // namespace dradd
