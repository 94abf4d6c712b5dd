// dradd_kernels.cu -- the rows kernels, the residual-add kernel, the
// conversion test kernel, the device status word and every launcher.  The
// staged kernels are instantiated in dradd_staged_<mode>_<out>.cu (one
// translation unit per mode and output kind, compiled in parallel) and
// reached through staged_fn_<mode>_<out>; the fused q/k kernels likewise in
// dradd_qk_<out>_<variant>.cu through qk_fn_<out>_<variant>.
#include <atomic>

#include <cuda_bf16.h>

#include "dradd_kernels.cuh"

namespace dradd {

// Written by a kernel only when a bounded wait expires (kernels reach it
// through Params::status); read and cleared by the host through
// dradd_device_status().
__device__ unsigned int g_device_status;

// ------------------------------------------------------------ residual add
// residual_out = bf16_rne(fp32(x) + fp32(residual)) over n_vec 16-byte
// vectors (8 elements each).  Thread t handles vectors t, t + stride, ...
// (stride = the grid's threads), kResidualAddInFlight of them per pass with
// all their loads issued before the first use, the last pass masked, so a
// thread's vectors are never fetched one round trip at a time.
constexpr int kResidualAddInFlight = 4;

__global__ void __launch_bounds__(256) residual_add_kernel(uint16_t* residual_out, const uint16_t* x,
                                                           const uint16_t* residual, int64_t n_vec,
                                                           int l2_prefetch)
{
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    const uint4* rv = reinterpret_cast<const uint4*>(residual);
    uint4* ov = reinterpret_cast<uint4*>(residual_out);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x;
    if (l2_prefetch && threadIdx.x == 0 && first < n_vec) {
        // the CTA's first vectors of x and residual, into L2 while the
        // previous grid finishes (a hint; the loads come after the wait)
        const int64_t left = n_vec - first;
        const uint32_t bytes = 16u * static_cast<uint32_t>(left < blockDim.x ? left : blockDim.x);
        prefetch_l2(xv + first, bytes);
        prefetch_l2(rv + first, bytes);
    }
    wait_prior_grids();
    allow_next_grid();
    constexpr int U = kResidualAddInFlight;
    for (int64_t i = first + threadIdx.x; i < n_vec; i += U * stride) {
        uint4 a[U], b[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (i + u * stride < n_vec) {
                a[u] = ld_stream(xv + i + u * stride);
                b[u] = ld_stream(rv + i + u * stride);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (i + u * stride < n_vec) {
                float acc[8];
                add8(a[u], b[u], acc);
                st_stream(ov + i + u * stride, pack8_rne(acc));
            }
        }
    }
}

// ---------------------------------------------------------- conversion hook
__global__ void convert_kernel(uint16_t* out, uint64_t first, int64_t count, int method)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += stride) {
        const float f = __uint_as_float(static_cast<uint32_t>(first + static_cast<uint64_t>(i)));
        uint32_t b;
        if (method == 1)
            b = rne_bits_int(f);
        else if (method == 2)
            b = pack_rne_cvt(f, f) & 0xFFFFu;
        else if (method == 3)
            b = e4m3x2(f, f) & 0xFFu;
        else if (method == 4)
            b = e2m1x2(f, f) & 0xFu;
        else if (method == 5)
            b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
        else
            b = pack_rne(f, f) & 0xFFFFu;
        out[i] = static_cast<uint16_t>(b);
    }
}

// ------------------------------------------------------------------ launchers
namespace {

KernelFn rows_fn(int K, int out, bool add)
{
#define DRADD_ROWS_OUT(KK, OO) \
    return add ? rows_kernel<KK, OO, true> : rows_kernel<KK, OO, false>
#define DRADD_ROWS(KK)                                                  \
    switch (out) {                                                      \
    case kOutBf16: DRADD_ROWS_OUT(KK, kOutBf16);                        \
    case kOutInt8: DRADD_ROWS_OUT(KK, kOutInt8);                        \
    case kOutE4m3: DRADD_ROWS_OUT(KK, kOutE4m3);                        \
    case kOutE2m1: DRADD_ROWS_OUT(KK, kOutE2m1);                        \
    default: return nullptr;                                            \
    }
    switch (K) {
    case 1: DRADD_ROWS(1)
    case 2: DRADD_ROWS(2)
    case 4: DRADD_ROWS(4)
    case 8: DRADD_ROWS(8)
    default: return nullptr;
    }
#undef DRADD_ROWS
#undef DRADD_ROWS_OUT
}

KernelFn staged_fn(int T, int K, int out, bool add, bool pair = false)
{
    if (pair) {
        if (add)
            return nullptr;
        switch (out) {
        case kOutInt8: return staged_pair_fn_norm_int8(T, K);
        case kOutE4m3: return staged_pair_fn_norm_e4m3(T, K);
        case kOutE2m1: return staged_pair_fn_norm_e2m1(T, K);
        default: return nullptr;
        }
    }
    switch (out) {
    case kOutBf16: return add ? staged_fn_add_bf16(T, K) : staged_fn_norm_bf16(T, K);
    case kOutInt8: return add ? staged_fn_add_int8(T, K) : staged_fn_norm_int8(T, K);
    case kOutE4m3: return add ? staged_fn_add_e4m3(T, K) : staged_fn_norm_e4m3(T, K);
    case kOutE2m1: return add ? staged_fn_add_e2m1(T, K) : staged_fn_norm_e2m1(T, K);
    default: return nullptr;
    }
}

int log2i(int v)
{
    int l = 0;
    while ((1 << l) < v)
        ++l;
    return l;
}

// One bit per staged kernel: (add, out = 0..3, T = 32..1024, K = 1..8); the
// plain quantised pair kernels (out = 1..3) follow from 288.
int staged_index(int T, int K, int out, bool add, bool pair = false)
{
    if (pair)
        return 288 + (out - 1) * 24 + (log2i(T) - 5) * 4 + log2i(K);
    return ((add ? 4 : 0) + out) * 24 + (log2i(T) - 5) * 4 + log2i(K);
}

constexpr int kMaxDevices = 64;
// Per device: bit k of word k / 64 set once staged kernel k (8 x 24 of them),
// split kernel k - 192 (4 x 24) or pair kernel k - 288 (3 x 24) has been
// allowed its full dynamic shared memory.
std::atomic<uint64_t> g_smem_attr_done[kMaxDevices][6];
std::atomic<unsigned*> g_status_ptr[kMaxDevices];

cudaError_t ensure_smem_attr(KernelFn fn, int index, int dev)
{
    const uint64_t bit = 1ull << (index % 64);
    std::atomic<uint64_t>* word = dev >= 0 && dev < kMaxDevices ? &g_smem_attr_done[dev][index / 64] : nullptr;
    if (word && (word->load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return e;
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, fn);
    if (e != cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(attr.sharedSizeBytes));
    if (e != cudaSuccess)
        return e;
    if (word)
        word->fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

}  // namespace

cudaError_t device_status_ptr(unsigned** ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < kMaxDevices) {
        unsigned* cached = g_status_ptr[dev].load(std::memory_order_acquire);
        if (cached) {
            *ptr = cached;
            return cudaSuccess;
        }
    }
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_device_status);
    if (e != cudaSuccess)
        return e;
    *ptr = static_cast<unsigned*>(addr);
    if (dev >= 0 && dev < kMaxDevices)
        g_status_ptr[dev].store(*ptr, std::memory_order_release);
    return cudaSuccess;
}

cudaError_t launch_rows(const Params& p, int K, int out, bool add, int grid, int threads, bool serialize,
                        cudaStream_t stream)
{
    KernelFn fn = rows_fn(K, out, add);
    if (!fn)
        return cudaErrorInvalidValue;
    return launch(fn, grid, threads, 0, serialize, stream, p);
}

cudaError_t launch_staged(const Params& p, int K, int out, bool add, int grid, int threads,
                          size_t dyn_smem, bool serialize, cudaStream_t stream)
{
    const bool pair = p.rows_per_cta == 2;
    KernelFn fn = staged_fn(threads, K, out, add, pair);
    if (!fn)
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = ensure_smem_attr(fn, staged_index(threads, K, out, add, pair), dev);
    if (e != cudaSuccess)
        return e;
    return launch(fn, grid, threads, dyn_smem, serialize, stream, p);
}

namespace {

KernelFn split_fn(int T, int K, int C, bool add)
{
    return add ? split_fn_add(T, K, C) : split_fn_norm(T, K, C);
}

int split_index(int T, int K, int C, bool add)
{
    return 192 + ((add ? 2 : 0) + (C == 4 ? 1 : 0)) * 24 + (log2i(T) - 5) * 4 + log2i(K);
}

cudaLaunchConfig_t split_config(int grid, int threads, size_t dyn_smem, bool serialize, cudaStream_t stream,
                                int C, cudaLaunchAttribute (&attr)[2])
{
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = dyn_smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = serialize ? 1 : 2;
    return cfg;
}

}  // namespace

cudaError_t launch_split(const Params& p, int K, int C, bool add, int grid, int threads, size_t dyn_smem,
                         bool serialize, cudaStream_t stream)
{
    KernelFn fn = split_fn(threads, K, C, add);
    if (!fn || grid % C != 0)
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = ensure_smem_attr(fn, split_index(threads, K, C, add), dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = split_config(grid, threads, dyn_smem, serialize, stream, C, attr);
    return cudaLaunchKernelEx(&cfg, fn, p);
}

cudaError_t split_max_clusters(int K, int C, bool add, int threads, size_t dyn_smem, int* clusters)
{
    KernelFn fn = split_fn(threads, K, C, add);
    if (!fn)
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = ensure_smem_attr(fn, split_index(threads, K, C, add), dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = split_config(C, threads, dyn_smem, true, 0, C, attr);
    return cudaOccupancyMaxActiveClusters(clusters, fn, &cfg);
}

// One bit per warp kernel (add, out = 0..3, K = 1..16): its dynamic shared
// memory limit has been raised to the device's opt-in maximum.
std::atomic<uint64_t> g_warp_smem_done[kMaxDevices];

cudaError_t warp_prepare(KernelFn fn, int K, int out, bool add)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (((add ? 4 : 0) + out) * 5 + log2i(K));
    std::atomic<uint64_t>* word = dev >= 0 && dev < kMaxDevices ? &g_warp_smem_done[dev] : nullptr;
    if (word && (word->load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return e;
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, fn);
    if (e != cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(attr.sharedSizeBytes));
    if (e != cudaSuccess)
        return e;
    if (word)
        word->fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

cudaError_t launch_warp(const Params& p, int K, int out, bool add, int grid, int threads, size_t dyn_smem,
                        bool serialize, cudaStream_t stream)
{
    KernelFn fn = add ? warp_fn_add(out, K) : warp_fn_norm(out, K);
    if (!fn)
        return cudaErrorInvalidValue;
    cudaError_t e = warp_prepare(fn, K, out, add);
    if (e != cudaSuccess)
        return e;
    return launch(fn, grid, threads, dyn_smem, serialize, stream, p);
}

cudaError_t warp_occupancy(int K, int out, bool add, int threads, size_t dyn_smem, int* blocks_per_sm)
{
    KernelFn fn = add ? warp_fn_add(out, K) : warp_fn_norm(out, K);
    if (!fn)
        return cudaErrorInvalidValue;
    cudaError_t e = warp_prepare(fn, K, out, add);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, threads, dyn_smem);
}

cudaError_t staged_occupancy(int K, int out, bool add, int threads, size_t dyn_smem, int* blocks_per_sm,
                             bool pair)
{
    KernelFn fn = staged_fn(threads, K, out, add, pair);
    if (!fn)
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = ensure_smem_attr(fn, staged_index(threads, K, out, add, pair), dev);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, threads, dyn_smem);
}

size_t split_static_smem(int K)
{
    // s_sum[2][32 * K] + s_max[2][32] + s_part[2][2], as declared in split_kernel
    return sizeof(float) * (2 * 32 * static_cast<size_t>(K) + 2 * 32 + 4);
}

size_t staged_static_smem(int K, bool pair)
{
    // at most s_sum[2][K * 32] + s_max[2][32] + s_max2[32] (32 warps), as
    // declared in staged_kernel; twice each for staged_pair_kernel
    const size_t one = 2 * 32 * static_cast<size_t>(K) + 3 * 32;
    return sizeof(float) * (pair ? 2 * one : one);
}

namespace {

QkKernelFn qk_fn(int kq, int kk, bool quant, bool add, int mode)
{
    if (mode == kQkChunk)
        return quant ? qk_fn_e4m3_chunk(kk, add) : qk_fn_bf16_chunk(kk, add);
    if (mode == kQkWarp)
        return quant ? qk_fn_e4m3_warp(kq, kk, add) : qk_fn_bf16_warp(kq, kk, add);
    const bool staged = mode == kQkStaged;
    if (quant)
        return staged ? qk_fn_e4m3_staged(kq, kk, add) : qk_fn_e4m3_rows(kq, kk, add);
    return staged ? qk_fn_bf16_staged(kq, kk, add) : qk_fn_bf16_rows(kq, kk, add);
}

// One bit per staged (word 0), warp-per-row (word 1) or chunked-q (word 2)
// qk kernel (kq, kk, quant, add): its dynamic shared memory limit has been
// raised to the device's opt-in maximum.
std::atomic<uint64_t> g_qk_smem_done[kMaxDevices][3];

cudaError_t qk_prepare(QkKernelFn fn, int kq, int kk, bool quant, bool add, int mode)
{
    if (mode == kQkRows)
        return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const int kq_bits = mode == kQkChunk ? 0 : log2i(kq);  // the chunked kernels have no kq
    const uint64_t bit = 1ull << (((kq_bits * 4 + log2i(kk)) * 2 + (quant ? 1 : 0)) * 2 + (add ? 1 : 0));
    const int w = mode == kQkChunk ? 2 : mode == kQkWarp ? 1 : 0;
    std::atomic<uint64_t>* word = dev >= 0 && dev < kMaxDevices ? &g_qk_smem_done[dev][w] : nullptr;
    if (word && (word->load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return e;
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, fn);
    if (e != cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(attr.sharedSizeBytes));
    if (e != cudaSuccess)
        return e;
    if (word)
        word->fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

}  // namespace

size_t qk_static_smem(int kq, int kk)
{
    // s_sum[2][32 * K] + s_max[2][32] of each side's body, as declared
    return sizeof(float) * (2 * 32 * static_cast<size_t>(kq + kk) + 4 * 32);
}

cudaError_t launch_qk(const Params& pq, const Params& pk, int kq, int kk, bool quant, bool add, int mode,
                      int q_ctas, int k_ctas, int threads, size_t dyn_smem, bool serialize, cudaStream_t stream)
{
    QkKernelFn fn = qk_fn(kq, kk, quant, add, mode);
    if (!fn)
        return cudaErrorInvalidValue;
    cudaError_t e = qk_prepare(fn, kq, kk, quant, add, mode);
    if (e != cudaSuccess)
        return e;
    return launch(fn, q_ctas + k_ctas, threads, dyn_smem, serialize, stream, pq, pk, q_ctas);
}

cudaError_t qk_occupancy(int kq, int kk, bool quant, bool add, int mode, int threads, size_t dyn_smem,
                         int* blocks_per_sm)
{
    QkKernelFn fn = qk_fn(kq, kk, quant, add, mode);
    if (!fn)
        return cudaErrorInvalidValue;
    cudaError_t e = qk_prepare(fn, kq, kk, quant, add, mode);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, threads, dyn_smem);
}

cudaError_t launch_residual_add(uint16_t* residual_out, const uint16_t* x, const uint16_t* residual,
                                int64_t n_vec, int sm_count, bool l2_prefetch, bool serialize,
                                cudaStream_t stream)
{
    const int threads = 256;
    int64_t blocks = (n_vec + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count) * (2048 / threads);
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    return launch(residual_add_kernel, static_cast<int>(blocks), threads, 0, serialize, stream, residual_out, x,
                  residual, n_vec, l2_prefetch ? 1 : 0);
}

cudaError_t launch_convert(uint16_t* out, uint64_t first, int64_t count, int method, cudaStream_t stream)
{
    if (count <= 0)
        return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (count + threads - 1) / threads;
    if (blocks > 65536)
        blocks = 65536;
    convert_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(out, first, count, method);
    return cudaGetLastError();
}

// The status word is read (and with `clear` reset) by one atomic exchange in
// a one-thread kernel on the caller's stream, so a timeout that a kernel on
// another stream records at the same moment is either in the value read or
// stays in the word for the next read; never lost.  The value travels back
// through a result slot of its own per call (a ring of kStatusSlots, picked
// by a host counter), so reads from several host threads at once do not
// overwrite each other's results.
constexpr unsigned kStatusSlots = 64;
__device__ unsigned int g_status_taken[kStatusSlots];

__global__ void status_take_kernel(unsigned slot, int clear)
{
    g_status_taken[slot] = clear ? atomicExch(&g_device_status, 0u) : atomicOr(&g_device_status, 0u);
}

cudaError_t read_device_status(unsigned* status, bool clear, cudaStream_t stream)
{
    static std::atomic<unsigned> next_slot{0};
    const unsigned slot = next_slot.fetch_add(1, std::memory_order_relaxed) % kStatusSlots;
    status_take_kernel<<<1, 1, 0, stream>>>(slot, clear ? 1 : 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    unsigned value = 0;
    e = cudaMemcpyFromSymbolAsync(&value, g_status_taken, sizeof(unsigned), slot * sizeof(unsigned),
                                  cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess)
        return e;
    e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess)
        *status = value;
    return e;
}

}  // namespace dradd
