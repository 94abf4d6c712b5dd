// dradd_internal.h -- what the C-ABI layer and the kernels share: the kernel
// parameter block and the launchers.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dradd {

struct Params {
    uint16_t* out;            // bf16 out (bf16 variant)
    int8_t* out_q;            // int8, e4m3 or packed e2m1 codes (quantised variants)
    float* scale;             // per-row (or per-group) scale (quantised variants)
    uint16_t* residual_out;
    const uint16_t* x;
    const uint16_t* residual;
    const uint16_t* weight;
    float eps;
    int hidden;
    float inv_hidden;         // 1 / hidden if hidden is a power of two, else 0
    int64_t n_rows;
    int threads_per_row;      // T
    int rows_per_cta;         // rows kernel only
    int stages;               // staged kernel only
    int fault_inject;         // staged kernel only
    uint64_t wait_limit_ns;   // staged kernel only
    unsigned* status;         // device status word (set on an expired wait)
    int group_blocks;         // per-group e4m3 out: 8-element blocks per group (a power of two)
    int group_shift;          // log2(group_blocks)
    int l2_prefetch;          // 1: device memory; first rows may be prefetched into L2 before the dependency wait
};

constexpr unsigned kDeviceStatusTimeout = 1u;
// A bulk copy issued before a timeout had still not landed when the CTA gave
// up waiting for it (after several wait limits).
constexpr unsigned kDeviceStatusUndrained = 2u;

// What a normalised row is stored as.
enum OutKind : int { kOutBf16 = 0, kOutInt8 = 1, kOutE4m3 = 2, kOutE2m1 = 3, kOutE4m3Group = 4 };

// The largest code magnitude of a quantised output: its scale is
// RN(amax / quant_divisor(out)).
__host__ __device__ constexpr int quant_divisor(int out)
{
    return out == kOutInt8 ? 127 : out == kOutE2m1 ? 6 : 448;
}

// Shared memory the staged kernel keeps besides its stages: for the
// quantised outputs the row's weights, widened to fp32 once per CTA (4
// bytes per element of the row, 16-byte aligned).
__host__ __device__ constexpr uint32_t staged_weight_bytes(int out, int hidden)
{
    return out == kOutBf16 ? 0u : 4u * static_cast<uint32_t>(hidden);
}

using KernelFn = void (*)(Params);
// Fused q/k RMSNorm: (q rows, k rows, number of CTAs given to the q rows).
using QkKernelFn = void (*)(Params, Params, int);

// Largest CTA for K blocks per thread: the register budget of the bigger
// tiles (K * 8 accumulators per thread) needs the smaller CTA.
constexpr int max_threads_for(int K) { return K <= 2 ? 1024 : 512; }

// Largest CTA of the fused q/k kernel whose larger side has K blocks per
// thread: 128 registers per thread up to K = 4, 255 at K = 8, no spills.
constexpr int qk_max_threads(int K) { return K <= 4 ? 512 : 256; }

// Resident CTAs per SM the staged kernel with T threads and K blocks per
// thread is compiled for: the register budget per thread is about 40 for
// K = 1 (three 512-thread CTAs per SM), 64 for K = 2, 128 for K = 4 and 255
// for K = 8, capped at 2048 threads and 32 CTAs per SM.
constexpr int staged_reg_target(int K) { return K == 1 ? 40 : K == 2 ? 64 : K == 4 ? 128 : 255; }
constexpr int staged_min_blocks(int T, int K)
{
    int by_regs = 65536 / (T * staged_reg_target(K));
    int by_threads = 2048 / T;
    int b = by_regs < by_threads ? by_regs : by_threads;
    b = b > 32 ? 32 : b;
    return b < 1 ? 1 : b;
}

// add = true: residual-add + RMSNorm (reads x and residual, writes
// residual_out); false: plain RMSNorm of x.
cudaError_t launch_rows(const Params& p, int K, int out, bool add, int grid, int threads, bool serialize,
                        cudaStream_t stream);
cudaError_t launch_staged(const Params& p, int K, int out, bool add, int grid, int threads,
                          size_t dyn_smem, bool serialize, cudaStream_t stream);
cudaError_t staged_occupancy(int K, int out, bool add, int threads, size_t dyn_smem, int* blocks_per_sm,
                             bool pair = false);
size_t staged_static_smem(int K, bool pair = false);
// One function per (mode, output kind), each in its own translation unit.
KernelFn staged_fn_add_bf16(int T, int K);
KernelFn staged_fn_add_int8(int T, int K);
KernelFn staged_fn_add_e4m3(int T, int K);
KernelFn staged_fn_add_e2m1(int T, int K);
KernelFn staged_fn_norm_bf16(int T, int K);
KernelFn staged_fn_norm_int8(int T, int K);
KernelFn staged_pair_fn_norm_int8(int T, int K);
KernelFn staged_pair_fn_norm_e4m3(int T, int K);
KernelFn staged_pair_fn_norm_e2m1(int T, int K);
KernelFn staged_fn_norm_e4m3(int T, int K);
KernelFn staged_fn_norm_e2m1(int T, int K);
// Warp-per-row kernels: K = P / 256 blocks of 8 per lane (1..16; with a
// residual 1..8), one warp per row, R warps per CTA (at most kWarpMaxRows),
// `stages` groups of R rows (the main op) or a ring of `stages` row slots
// per warp (the fused q/k call).  Dynamic shared memory: the row slots, the
// fp32 weights and the mbarriers (one per slot at most).
constexpr int kWarpMaxRows = 16;
constexpr size_t warp_smem_bytes(int stages, int rows, int hidden, bool add)
{
    return static_cast<size_t>(stages) * (add ? 2u : 1u) * static_cast<size_t>(rows) * 2u *
               static_cast<size_t>(hidden) +
           4u * static_cast<size_t>(hidden) + 8u * static_cast<size_t>(stages) * static_cast<size_t>(rows);
}

// Chunked rows (the fused q/k call's CHUNK variant): kChunkElems elements
// a warp.  Dynamic shared memory of a CTA of nw chunk warps: the rings of
// `stages` chunk slots per warp, the row's fp32 weights, the chunk sums
// (2 x 8 floats) and the mbarriers.
constexpr int kChunkElems = 512;
constexpr int kChunkBlocks = kChunkElems / 8;

__host__ __device__ constexpr uint32_t chunk_slot_bytes(bool add)
{
    return (add ? 2u : 1u) * kChunkElems * 2u;
}

__host__ __device__ constexpr size_t chunk_smem_bytes(int stages, int nw, int hidden, bool add)
{
    return static_cast<size_t>(nw) * stages * chunk_slot_bytes(add) + 4u * static_cast<size_t>(hidden) + 64u +
           8u * static_cast<size_t>(nw) * stages;
}
KernelFn warp_fn_add(int out, int K);
KernelFn warp_fn_norm(int out, int K);
cudaError_t launch_warp(const Params& p, int K, int out, bool add, int grid, int threads, size_t dyn_smem,
                        bool serialize, cudaStream_t stream);
cudaError_t warp_occupancy(int K, int out, bool add, int threads, size_t dyn_smem, int* blocks_per_sm);
// Split-row kernels (bf16 out): clusters of C CTAs (2 or 4), each CTA a
// slice of every row of its cluster; grid a multiple of C.
KernelFn split_fn_add(int T, int K, int C);
KernelFn split_fn_norm(int T, int K, int C);
cudaError_t launch_split(const Params& p, int K, int C, bool add, int grid, int threads, size_t dyn_smem,
                         bool serialize, cudaStream_t stream);
cudaError_t split_max_clusters(int K, int C, bool add, int threads, size_t dyn_smem, int* clusters);
size_t split_static_smem(int K);
// Fused q/k RMSNorm: CTAs [0, q_ctas) take the q rows, the next k_ctas the
// k rows; kq / kk blocks of 8 per thread on each side.  quant: per-group
// e4m3 q out (else bf16); add: q has a residual; staged: rows staged
// through dyn_smem bytes of shared memory (else loaded into registers).
// mode: how each side's rows reach the registers.
enum QkMode : int { kQkRows = 0, kQkStaged = 1, kQkWarp = 2, kQkChunk = 3 };
cudaError_t launch_qk(const Params& pq, const Params& pk, int kq, int kk, bool quant, bool add, int mode,
                      int q_ctas, int k_ctas, int threads, size_t dyn_smem, bool serialize, cudaStream_t stream);
cudaError_t qk_occupancy(int kq, int kk, bool quant, bool add, int mode, int threads, size_t dyn_smem,
                         int* blocks_per_sm);
QkKernelFn qk_fn_bf16_rows(int kq, int kk, bool add);
QkKernelFn qk_fn_bf16_staged(int kq, int kk, bool add);
QkKernelFn qk_fn_e4m3_rows(int kq, int kk, bool add);
QkKernelFn qk_fn_e4m3_staged(int kq, int kk, bool add);
QkKernelFn qk_fn_bf16_warp(int kq, int kk, bool add);
QkKernelFn qk_fn_e4m3_warp(int kq, int kk, bool add);
QkKernelFn qk_fn_bf16_chunk(int kk, bool add);
QkKernelFn qk_fn_e4m3_chunk(int kk, bool add);
// Static shared memory of a qk kernel whose sides have kq / kk blocks per thread.
size_t qk_static_smem(int kq, int kk);
// l2_prefetch: all three are device memory (each CTA's first vectors are
// then prefetched into L2 before the dependency wait).
cudaError_t launch_residual_add(uint16_t* residual_out, const uint16_t* x, const uint16_t* residual,
                                int64_t n_vec, int sm_count, bool l2_prefetch, bool serialize,
                                cudaStream_t stream);
cudaError_t launch_convert(uint16_t* out, uint64_t first, int64_t count, int method, cudaStream_t stream);
cudaError_t read_device_status(unsigned* status, bool clear, cudaStream_t stream);
cudaError_t device_status_ptr(unsigned** ptr);

// Launch with programmatic stream serialization unless `serialize`: the
// kernel may then be scheduled while the previous kernel in the stream is
// still draining, and waits for it (griddepcontrol.wait) before touching
// global memory.
template <typename... Args>
inline cudaError_t launch(void (*fn)(Args...), int grid, int threads, size_t dyn_smem, bool serialize,
                          cudaStream_t stream, Args... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = dyn_smem;
    cfg.stream = stream;
    cfg.attrs = serialize ? nullptr : attr;
    cfg.numAttrs = serialize ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, fn, args...);
}

// Log-sum-exp merge and launch-invariant elementwise functions
// (dradd_lse.cu).  Rows of n_cols elements, row strides in elements; a flat
// array is one row.  vec: elements per thread per pass (1, 2, 4, 8); vec4:
// every base address is 16-byte aligned and every row stride a multiple of
// 4 elements (whole units then move as 16-byte vectors); l2_prefetch (with
// vec4): the inputs are device memory, and each CTA's first unit is
// prefetched into L2 before the dependency wait.
cudaError_t launch_lse_merge(float* out, int64_t out_stride, const float* a, int64_t a_stride, const float* b,
                             int64_t b_stride, int64_t n_rows, int64_t n_cols, int vec, bool vec4,
                             bool l2_prefetch, int grid, int threads, bool serialize, cudaStream_t stream);
cudaError_t launch_unary(float* out, const float* x, int64_t n, int op, int vec, bool vec4, bool l2_prefetch,
                         int grid, int threads, bool serialize, cudaStream_t stream);

}  // namespace dradd
