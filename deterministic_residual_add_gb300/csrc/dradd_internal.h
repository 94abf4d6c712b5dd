// dradd_internal.h -- what the C-ABI layer and the kernels share: the kernel
// parameter block and the launchers.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dradd {

struct Params {
    uint16_t* out;            // bf16 out (bf16 variant)
    int8_t* out_q;            // int8 out (quant variant)
    float* scale;             // per-row scale (quant variant)
    uint16_t* residual_out;
    const uint16_t* x;
    const uint16_t* residual;
    const uint16_t* weight;
    float eps;
    int hidden;
    int64_t n_rows;
    int threads_per_row;      // T
    int rows_per_cta;         // rows kernel only
    int stages;               // staged kernel only
    int fault_inject;         // staged kernel only
    uint64_t wait_limit_ns;   // staged kernel only
};

// Largest CTA for K blocks per thread: the register budget of the bigger
// tiles (K * 8 accumulators per thread) needs the smaller CTA.
constexpr int max_threads_for(int K) { return K <= 2 ? 1024 : 512; }
#ifndef DRADD_MINB1
#define DRADD_MINB1 1
#endif
#ifndef DRADD_MINB2
#define DRADD_MINB2 1
#endif
constexpr int min_blocks_for(int K) { return K == 1 ? DRADD_MINB1 : K == 2 ? DRADD_MINB2 : 1; }

cudaError_t launch_rows(const Params& p, int K, bool quant, int grid, int threads, bool serialize,
                        cudaStream_t stream);
cudaError_t launch_staged(const Params& p, int K, bool quant, int grid, int threads, size_t dyn_smem,
                          bool serialize, cudaStream_t stream);
size_t staged_static_smem(int K);
cudaError_t staged_occupancy(int K, bool quant, int threads, size_t dyn_smem, int* blocks_per_sm);
cudaError_t launch_convert(uint16_t* out, uint64_t first, int64_t count, int method, cudaStream_t stream);
cudaError_t read_device_status(unsigned* status, bool clear, cudaStream_t stream);

}  // namespace dradd
