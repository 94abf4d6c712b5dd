// dradd_warp.cuh -- the warp-per-row kernels: one warp owns a whole row at a
// time, so a row's reductions never leave the warp; the rows reach shared
// memory through the TMA engine, a group of R adjacent rows (one per warp
// of the CTA) per stage, `stages` groups ahead of the compute.
//
// Lane l of a row owns the 8-element blocks l, l + 32, ..., l + 32 (K - 1)
// (K = P / 256 blocks per lane, P = next power of two >= hidden) and reads
// them from the stage with 16-byte loads (a warp's loads for one j are 512
// consecutive bytes, free of bank conflicts).  The row's sum of squares
// follows the canonical tree exactly as in the other kernels: each block
// folded in registers, then warp_halving_sum across the lanes for all K
// subtrees at once, then fold_lane_subtrees for the top log2 K levels.
//
// Without a residual, acc = fp32(x) is exact, so x is read again from the
// stage wherever y is needed and no copy of the row is held in registers;
// with one, acc = fp32(x) + fp32(residual) is kept in fp32 registers
// (K <= 8).  The quantised outputs with a per-row scale compute y twice,
// once for the row's amax and once for the codes; both passes perform the
// same operations, so they give the same bits.  The per-group e4m3 output
// needs y only within a block's group, which lies in one j-slice of the
// warp, so it computes y once.
//
// Int8 codes take the bracket of quantize8_bracket on rows where the sum,
// the inverse RMS and every weight are finite: then |acc * inv| stays
// below about sqrt(hidden), so no y is NaN (a y that overflows to infinity
// makes the scale infinite, which the bracket does not take).  Other rows,
// and blocks whose bracket ends differ, use the correctly rounded division.
//
// warp_body's CTA meets at a barrier once per group, after every warp has
// finished with the stage, and thread 0 then refills that stage with the
// group `stages` ahead; warp_ring_body's warps share only the weights and
// never wait for one another.  Every wait on a copy is bounded, as in
// staged_kernel.
#pragma once

#include "dradd_kernels.cuh"

namespace dradd {

// The row's weights widened to fp32 once per CTA: w_lo[b] holds elements
// 0-3 of block b, w_hi[b] elements 4-7, so a warp's 16-byte reads of one
// j-slice are consecutive.  Ends with a CTA-wide barrier; returns whether
// every weight is finite.
__device__ __forceinline__ bool widen_weights_to_smem(const uint16_t* weight, int nblocks, float4* w_lo,
                                                      float4* w_hi)
{
    const uint4* wv = reinterpret_cast<const uint4*>(weight);
    bool finite = true;
    for (int b = threadIdx.x; b < nblocks; b += blockDim.x) {
        float f[8];
        unpack8(__ldg(wv + b), f);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            finite = finite && fabsf(f[e]) <= 3.40282347e38f;
        w_lo[b] = make_float4(f[0], f[1], f[2], f[3]);
        w_hi[b] = make_float4(f[4], f[5], f[6], f[7]);
    }
    return __syncthreads_and(finite) != 0;
}

// max |y| of one block as a balanced tree (exact; NaN ignored).
__device__ __forceinline__ float block_max_abs(const float (&y)[8])
{
    float a[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        a[e] = fabsf(y[e]);
    return max_tree<8, false>(a);
}

// One row by one warp: xs (and rs) its x (and residual) in shared memory.
template <int K, int OUT, bool ADD>
__device__ __forceinline__ void warp_row(const Params& p, int64_t row, const uint4* xs, const uint4* rs,
                                         const float4* w_lo, const float4* w_hi, bool w_finite)
{
    static_assert(K >= 1 && K <= 16 && (K & (K - 1)) == 0, "K: a power of two up to 16");
    static_assert(!ADD || K <= 8, "with a residual, acc stays in fp32 registers: K <= 8");
    const int lane = threadIdx.x & 31;
    const int nblocks = p.hidden >> 3;
    float part[K];
    float acc[ADD ? K : 1][8];
    if constexpr (ADD) {
        uint4* rorow = reinterpret_cast<uint4*>(p.residual_out + row * p.hidden);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = lane + 32 * j;
            if (b < nblocks) {
                add8(xs[b], rs[b], acc[j]);
                st_stream(rorow + b, pack8_rne(acc[j]));
                part[j] = fold8_squares(acc[j]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[j][e] = 0.0f;
                part[j] = 0.0f;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = lane + 32 * j;
            part[j] = 0.0f;
            if (b < nblocks) {
                float f[8];
                unpack8(xs[b], f);
                part[j] = fold8_squares(f);
            }
        }
    }
    int jsub;
    const float sum = fold_lane_subtrees<K>(warp_halving_sum<K>(part, lane, jsub));
    const float inv = inv_rms(sum, p.hidden, p.inv_hidden, p.eps);

    // y of this lane's block j (valid blocks only)
    auto y_of = [&](int j, float (&y)[8]) {
        const int b = lane + 32 * j;
        if constexpr (ADD) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                y[e] = acc[j][e];
        } else {
            unpack8(xs[b], y);
        }
        scale8_f32(y, inv, w_lo[b], w_hi[b]);
    };

    if constexpr (OUT == kOutBf16) {
        uint4* orow = reinterpret_cast<uint4*>(p.out + row * p.hidden);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = lane + 32 * j;
            if (b < nblocks) {
                float y[8];
                y_of(j, y);
                st_stream(orow + b, pack8_rne(y));
            }
        }
    } else if constexpr (OUT == kOutE4m3Group) {
        // A group is gb consecutive blocks (gb a power of two <= 32 that
        // divides nblocks): for each j, an aligned group of gb lanes.
        const int gb = p.group_blocks;
        const int64_t groups = nblocks >> p.group_shift;
        uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (32 * j >= nblocks)
                continue;  // the whole j-slice is padding (warp-uniform)
            const int b = lane + 32 * j;
            float y[8];
            float m = 0.0f;
            if (b < nblocks) {
                y_of(j, y);
                m = block_max_abs(y);
            }
            m = butterfly_max(m, gb);
            const float scale = div448_rn(m);
            if (b < nblocks) {
                if ((b & (gb - 1)) == 0)
                    p.scale[row * groups + (b >> p.group_shift)] = scale;
                st_stream(qrow + b, quantize8_e4m3(y, make_e4m3_scale(scale)));
            }
        }
    } else {
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int b = lane + 32 * j;
            if (b < nblocks) {
                float y[8];
                y_of(j, y);
                m = fmaxf(m, block_max_abs(y));
            }
        }
        m = warp_max(m);
        const float scale = div_const_rn<quant_divisor(OUT)>(m);
        if (lane == 0)
            p.scale[row] = scale;
        if constexpr (OUT == kOutInt8) {
            uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
            const Int8Bracket qs = make_int8_bracket(scale);
            const bool fast =
                qs.fast && w_finite && fabsf(sum) <= 3.40282347e38f && fabsf(inv) <= 3.40282347e38f;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int b = lane + 32 * j;
                if (b < nblocks) {
                    float y[8];
                    y_of(j, y);
                    uint32_t differ = 0u;
                    uint2 code = quantize8_bracket(y, qs, differ);
                    if (!fast || differ != 0u)
                        code = quantize8_exact(y, scale);
                    st_stream(qrow + b, code);
                }
            }
        } else {
            const E4m3Scale qs = make_e4m3_scale(scale);
            if constexpr (OUT == kOutE2m1) {
                uint32_t* prow = reinterpret_cast<uint32_t*>(p.out_q + row * (p.hidden / 2));
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const int b = lane + 32 * j;
                    if (b < nblocks) {
                        float y[8];
                        y_of(j, y);
                        __stcs(prow + b, quantize8_e2m1(y, qs));
                    }
                }
            } else {
                uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const int b = lane + 32 * j;
                    if (b < nblocks) {
                        float y[8];
                        y_of(j, y);
                        st_stream(qrow + b, quantize8_e4m3(y, qs));
                    }
                }
            }
        }
    }
}

// Groups cta, cta + n_ctas, ... of R = warps-per-CTA adjacent rows of p.
template <int K, int OUT, bool ADD>
__device__ __forceinline__ void warp_body(const Params& p, int64_t cta, int64_t n_ctas, unsigned char* smem)
{
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int R = blockDim.x >> 5;
    const int nblocks = p.hidden >> 3;
    const int stages = p.stages;
    const uint32_t row_bytes = static_cast<uint32_t>(p.hidden) * 2u;
    const uint32_t tile_bytes = row_bytes * static_cast<uint32_t>(R);
    const uint32_t stage_bytes = (ADD ? 2u : 1u) * tile_bytes;
    unsigned char* const after_stages = smem + static_cast<size_t>(stages) * stage_bytes;
    float4* const w_lo = reinterpret_cast<float4*>(after_stages);
    float4* const w_hi = w_lo + nblocks;
    uint64_t* const bars = reinterpret_cast<uint64_t*>(after_stages + 4u * static_cast<uint32_t>(p.hidden));
    const int64_t n_groups = (p.n_rows + R - 1) / R;

    if (tid == 0) {
        // While the previous grid finishes: L2 prefetches of this CTA's
        // first group (the copies that consume them are issued after the
        // wait below, and read what the memory holds then).
        if (p.l2_prefetch && cta < n_groups) {
            const int64_t row0 = cta * R;
            const int64_t left = p.n_rows - row0;
            const uint32_t bytes = row_bytes * static_cast<uint32_t>(left < R ? left : R);
            prefetch_l2(p.x + row0 * p.hidden, bytes);
            if constexpr (ADD)
                prefetch_l2(p.residual + row0 * p.hidden, bytes);
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
        unsigned char* dst = smem + static_cast<size_t>(s) * stage_bytes;
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
    const bool w_finite = widen_weights_to_smem(p.weight, nblocks, w_lo, w_hi);

    int64_t i = 0;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t g = cta; g < n_groups; g += n_ctas, ++i) {
        const bool ok = mbar_wait_bounded(&bars[s], parity, p.wait_limit_ns);
        const int64_t row = g * R + warp;
        if (ok && row < p.n_rows) {
            const unsigned char* sbase = smem + static_cast<size_t>(s) * stage_bytes +
                                         static_cast<size_t>(warp) * row_bytes;
            warp_row<K, OUT, ADD>(p, row, reinterpret_cast<const uint4*>(sbase),
                                  reinterpret_cast<const uint4*>(sbase + tile_bytes), w_lo, w_hi, w_finite);
        }
        // Every warp is done with stage s (so it can be refilled); any
        // expired wait ends the CTA here (that warp skipped its row, whose
        // outputs are then unspecified).
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                record_timeout(p);
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
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
}

// Rows of p for the warps of CTAs cta, cta + n_ctas, ...: warp w of the CTA
// (W warps) takes rows gw, gw + GW, ... with gw = cta * W + w and GW =
// n_ctas * W, each through a ring of `stages` row slots of its own in shared
// memory, filled by bulk copies that its lane 0 issues `stages` rows ahead
// and waited on through the warp's own mbarriers.  No barrier joins the
// warps once the weights are widened, so a warp never waits for another.
template <int K, int OUT, bool ADD>
__device__ __forceinline__ void warp_ring_body(const Params& p, int64_t cta, int64_t n_ctas, unsigned char* smem)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int W = blockDim.x >> 5;
    const int nblocks = p.hidden >> 3;
    const int stages = p.stages;
    const uint32_t row_bytes = static_cast<uint32_t>(p.hidden) * 2u;
    const uint32_t slot_bytes = (ADD ? 2u : 1u) * row_bytes;
    unsigned char* const ring = smem + static_cast<size_t>(warp) * stages * slot_bytes;
    unsigned char* const after_rings = smem + static_cast<size_t>(W) * stages * slot_bytes;
    float4* const w_lo = reinterpret_cast<float4*>(after_rings);
    float4* const w_hi = w_lo + nblocks;
    uint64_t* const bars =
        reinterpret_cast<uint64_t*>(after_rings + 4u * static_cast<uint32_t>(p.hidden)) + warp * stages;
    const int64_t first = cta * W + warp;
    const int64_t stride = n_ctas * W;

    if (lane == 0) {
        // While the previous grid finishes: an L2 prefetch of this warp's
        // first row (the copy that consumes it is issued after the wait
        // below, and reads what the memory holds then).
        if (p.l2_prefetch && first < p.n_rows) {
            prefetch_l2(p.x + first * p.hidden, row_bytes);
            if constexpr (ADD)
                prefetch_l2(p.residual + first * p.hidden, row_bytes);
        }
        for (int s = 0; s < stages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    wait_prior_grids();
    allow_next_grid();

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int s, int64_t row) {
        unsigned char* dst = ring + static_cast<size_t>(s) * slot_bytes;
        mbar_arrive_expect_tx(&bars[s], slot_bytes);
        bulk_copy_g2s(dst, p.x + row * p.hidden, row_bytes, &bars[s], policy);
        if constexpr (ADD)
            bulk_copy_g2s(dst + row_bytes, p.residual + row * p.hidden, row_bytes, &bars[s], policy);
    };
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t row = first + s * stride;
            if (row >= p.n_rows)
                break;
            if (p.fault_inject && s == 0)
                continue;  // test hook: this copy never comes, so its wait expires
            issue(s, row);
        }
    }
    const bool w_finite = widen_weights_to_smem(p.weight, nblocks, w_lo, w_hi);

    int64_t i = 0;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t row = first; row < p.n_rows; row += stride, ++i) {
        const bool ok = mbar_wait_bounded(&bars[s], parity, p.wait_limit_ns);
        if (__any_sync(0xFFFFFFFFu, !ok)) {
            // this warp stops; its issued copies land before it leaves
            if (lane == 0) {
                record_timeout(p);
                drain_issued_copies(p, bars, s, parity, i, stages, first, stride, p.n_rows);
            }
            return;
        }
        const unsigned char* slot = ring + static_cast<size_t>(s) * slot_bytes;
        warp_row<K, OUT, ADD>(p, row, reinterpret_cast<const uint4*>(slot),
                              reinterpret_cast<const uint4*>(slot + row_bytes), w_lo, w_hi, w_finite);
        __syncwarp();  // every lane is done with the slot
        if (lane == 0) {
            const int64_t next = row + static_cast<int64_t>(stages) * stride;
            if (next < p.n_rows) {
                fence_proxy_async_smem();
                issue(s, next);
            }
        }
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
}

// ------------------------------------------------------------ chunked rows
// Rows of kChunkElems-element chunks, one warp per chunk: a CTA of NW
// warps (NW = the chunks that hold data, hidden / kChunkElems rounded up)
// takes whole rows, rows cta, cta + n_ctas, ...  Warp c owns the blocks
// 64 c .. 64 c + 63 of every row, lane l the blocks 64 c + l and 64 c + l
// + 32, so within its chunk the warp computes exactly what warp_row
// computes for a 512-element row: the chunk's subtree of the canonical
// tree.  The P / 512 chunk sums (zero for the chunks past the data) then
// fold pairwise, adjacent first: the top levels of the same tree, so the
// row's sum is bit for bit the one-warp (and the oracle's) value.  One CTA
// barrier per row exchanges the chunk sums; each warp has its own ring of
// `stages` chunk slots in shared memory, filled by bulk copies that its
// lane 0 issues `stages` rows ahead.  The chunk's fp32 weights are widened
// into shared memory once by the warp that reads them.  Outputs: bf16, or
// per-group e4m3 (a group, gb <= 32 aligned blocks, lies inside one
// j-slice of a chunk).
template <int OUT, bool ADD>
__device__ __forceinline__ void chunk_row_body(const Params& p, int64_t cta, int64_t n_ctas, unsigned char* smem)
{
    static_assert(OUT == kOutBf16 || OUT == kOutE4m3Group, "bf16 or per-group e4m3 out");
    constexpr int K = kChunkBlocks / 32;  // blocks per lane in a chunk
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int NW = blockDim.x >> 5;
    const int nblocks = p.hidden >> 3;
    int Q = 1;  // chunks of the padded row (P / 512)
    while (Q * kChunkBlocks < nblocks)
        Q <<= 1;
    const int stages = p.stages;
    const int first_block = warp * kChunkBlocks;
    const int cblocks = nblocks - first_block < kChunkBlocks ? nblocks - first_block : kChunkBlocks;
    const uint32_t chunk_bytes = static_cast<uint32_t>(cblocks) * 16u;
    constexpr uint32_t slot_bytes = chunk_slot_bytes(ADD);
    unsigned char* const ring = smem + static_cast<size_t>(warp) * stages * slot_bytes;
    unsigned char* const after_rings = smem + static_cast<size_t>(NW) * stages * slot_bytes;
    float4* const w_lo = reinterpret_cast<float4*>(after_rings);
    float4* const w_hi = w_lo + nblocks;
    float* const s_chunk = reinterpret_cast<float*>(after_rings + 4u * static_cast<uint32_t>(p.hidden));  // [2][8]
    uint64_t* const bars = reinterpret_cast<uint64_t*>(s_chunk + 16) + warp * stages;

    if (lane == 0) {
        if (p.l2_prefetch && cta < p.n_rows) {
            prefetch_l2(p.x + cta * p.hidden + first_block * 8, chunk_bytes);
            if constexpr (ADD)
                prefetch_l2(p.residual + cta * p.hidden + first_block * 8, chunk_bytes);
        }
        for (int s = 0; s < stages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    wait_prior_grids();
    allow_next_grid();

    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int s, int64_t row) {
        unsigned char* dst = ring + static_cast<size_t>(s) * slot_bytes;
        const int64_t off = row * p.hidden + first_block * 8;
        mbar_arrive_expect_tx(&bars[s], (ADD ? 2u : 1u) * chunk_bytes);
        bulk_copy_g2s(dst, p.x + off, chunk_bytes, &bars[s], policy);
        if constexpr (ADD)
            bulk_copy_g2s(dst + kChunkElems * 2, p.residual + off, chunk_bytes, &bars[s], policy);
    };
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t row = cta + s * n_ctas;
            if (row >= p.n_rows)
                break;
            if (p.fault_inject && s == 0)
                continue;  // test hook: this copy never comes, so its wait expires
            issue(s, row);
        }
    }
    {
        // this warp's chunk of the weights, widened once (only this lane reads them)
        const uint4* wrow = reinterpret_cast<const uint4*>(p.weight);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int bl = lane + 32 * j;
            if (bl < cblocks) {
                float f[8];
                unpack8(__ldg(wrow + first_block + bl), f);
                w_lo[first_block + bl] = make_float4(f[0], f[1], f[2], f[3]);
                w_hi[first_block + bl] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    }

    int buf = 0;
    int64_t i = 0;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t row = cta; row < p.n_rows; row += n_ctas, ++i) {
        const bool ok = mbar_wait_bounded(&bars[s], parity, p.wait_limit_ns);
        const unsigned char* slot = ring + static_cast<size_t>(s) * slot_bytes;
        const uint4* xs = reinterpret_cast<const uint4*>(slot);
        const uint4* rs = reinterpret_cast<const uint4*>(slot + kChunkElems * 2);
        float part[K];
        float acc[ADD ? K : 1][8];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int bl = lane + 32 * j;
            part[j] = 0.0f;
            if constexpr (ADD) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[j][e] = 0.0f;
            }
            if (bl < cblocks) {
                if constexpr (ADD) {
                    add8(xs[bl], rs[bl], acc[j]);
                    st_stream(reinterpret_cast<uint4*>(p.residual_out + row * p.hidden) + first_block + bl,
                              pack8_rne(acc[j]));
                    part[j] = fold8_squares(acc[j]);
                } else {
                    float f[8];
                    unpack8(xs[bl], f);
                    part[j] = fold8_squares(f);
                }
            }
        }
        int jsub;
        const float v = fold_lane_subtrees<K>(warp_halving_sum<K>(part, lane, jsub));
        if (lane == 0)
            s_chunk[buf * 8 + warp] = v;
        // every warp has published its chunk's sum; any expired wait ends
        // the CTA here (each warp's lane 0 first waits for its own copies)
        if (__syncthreads_or(!ok)) {
            if (lane == 0) {
                record_timeout(p);
                drain_issued_copies(p, bars, s, parity, i, stages, cta, n_ctas, p.n_rows);
            }
            return;
        }
        if constexpr (ADD) {
            // acc holds the row: the slot can be refilled now
            if (lane == 0) {
                const int64_t next = row + static_cast<int64_t>(stages) * n_ctas;
                if (next < p.n_rows) {
                    fence_proxy_async_smem();
                    issue(s, next);
                }
            }
        }
        float c[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            c[q] = q < NW ? s_chunk[buf * 8 + q] : 0.0f;
        // the chunk sums, adjacent pairs first, up to the Q chunks of P
#pragma unroll
        for (int width = 1; width < 8; width *= 2) {
#pragma unroll
            for (int q = 0; q < 8; q += 2 * width) {
                if (width < Q)
                    c[q] = __fadd_rn(c[q], c[q + width]);
            }
        }
        const float inv = inv_rms(c[0], p.hidden, p.inv_hidden, p.eps);

        auto y_of = [&](int j, float (&y)[8]) {
            const int bl = lane + 32 * j;
            if constexpr (ADD) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    y[e] = acc[j][e];
            } else {
                unpack8(xs[bl], y);
            }
            scale8_f32(y, inv, w_lo[first_block + bl], w_hi[first_block + bl]);
        };
        if constexpr (OUT == kOutBf16) {
            uint4* orow = reinterpret_cast<uint4*>(p.out + row * p.hidden);
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int bl = lane + 32 * j;
                if (bl < cblocks) {
                    float y[8];
                    y_of(j, y);
                    st_stream(orow + first_block + bl, pack8_rne(y));
                }
            }
        } else {
            const int gb = p.group_blocks;
            const int64_t groups = nblocks >> p.group_shift;
            uint2* qrow = reinterpret_cast<uint2*>(p.out_q + row * p.hidden);
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (32 * j >= cblocks)
                    continue;  // the whole j-slice is past the data (warp-uniform)
                const int bl = lane + 32 * j;
                const int b = first_block + bl;
                float y[8];
                float m = 0.0f;
                if (bl < cblocks) {
                    y_of(j, y);
                    m = block_max_abs(y);
                }
                m = butterfly_max(m, gb);
                const float scale = div448_rn(m);
                if (bl < cblocks) {
                    if ((b & (gb - 1)) == 0)
                        p.scale[row * groups + (b >> p.group_shift)] = scale;
                    st_stream(qrow + b, quantize8_e4m3(y, make_e4m3_scale(scale)));
                }
            }
        }
        if constexpr (!ADD) {
            __syncwarp();  // every lane is done with the slot
            if (lane == 0) {
                const int64_t next = row + static_cast<int64_t>(stages) * n_ctas;
                if (next < p.n_rows) {
                    fence_proxy_async_smem();
                    issue(s, next);
                }
            }
        }
        buf ^= 1;
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
}

// The warp-per-row kernel of the main op (up to kWarpMaxRows warps a CTA;
// shared memory layout as warp_smem_bytes).
template <int K, int OUT, bool ADD>
__global__ void __launch_bounds__(32 * kWarpMaxRows, 1) warp_kernel(const Params p)
{
    extern __shared__ __align__(128) unsigned char wsm[];
    warp_body<K, OUT, ADD>(p, blockIdx.x, gridDim.x, wsm);
}

template <int OUT, bool ADD>
KernelFn warp_table(int K)
{
    switch (K) {
    case 1: return warp_kernel<1, OUT, ADD>;
    case 2: return warp_kernel<2, OUT, ADD>;
    case 4: return warp_kernel<4, OUT, ADD>;
    case 8: return warp_kernel<8, OUT, ADD>;
    case 16:
        if constexpr (!ADD)
            return warp_kernel<16, OUT, ADD>;
        else
            return nullptr;
    default: return nullptr;
    }
}

}  // namespace dradd
