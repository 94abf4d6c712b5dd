// dradd_abi.cu -- the C entry points declared in include/dradd.h: argument
// validation, launch-configuration choice, and dispatch to the kernels.
//
// Nothing here changes a result bit: the configuration only decides how rows
// and blocks are spread over threads, CTAs and SMs, and the kernels combine
// the partial sums in the same canonical pairwise order for every choice.
#include <atomic>
#include <cmath>
#include <initializer_list>
#include <cstdint>
#include <cstring>

#include "dradd.h"
#include "dradd_internal.h"

namespace {

using dradd::Params;

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // 1 s

// Shared-memory and thread limits used to size grids and stages.  Defaults
// are GB300's; with a live device they come from the device.
struct DeviceLimits {
    int sm_count = 152;
    int smem_per_block_optin = 232448;  // 227 KiB
    int smem_per_sm = 233472;           // 228 KiB
    int max_threads_per_sm = 2048;
    int max_blocks_per_sm = 32;
};

std::atomic<int> g_limits_ready[kMaxDevices];
DeviceLimits g_limits[kMaxDevices];

dradd_status query_limits(DeviceLimits* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DRADD_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices && g_limits_ready[dev].load(std::memory_order_acquire)) {
        *out = g_limits[dev];
        return DRADD_OK;
    }
    DeviceLimits L;
    if (cudaDeviceGetAttribute(&L.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&L.smem_per_block_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&L.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&L.max_threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&L.max_blocks_per_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev) !=
            cudaSuccess)
        return DRADD_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) {
        g_limits[dev] = L;  // identical values if two threads race here
        g_limits_ready[dev].store(1, std::memory_order_release);
    }
    *out = L;
    return DRADD_OK;
}

// True when every non-NULL pointer is device memory.  Other memory the GPU
// can address (pinned or registered host memory, memory the GPU reaches
// through the host link, managed memory) is served by the register-load
// variant only: the staged variant's bulk copies are used on device memory.
bool all_device_memory(std::initializer_list<const void*> ptrs)
{
    for (const void* p : ptrs) {
        if (!p)
            continue;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
            cudaGetLastError();  // not a sticky error; the pointer is simply not device memory
            return false;
        }
        if (a.type != cudaMemoryTypeDevice)
            return false;
    }
    return true;
}

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

int64_t next_pow2(int64_t v)
{
    int64_t p = 1;
    while (p < v)
        p *= 2;
    return p;
}

// Byte ranges of the buffers of one call, for the overlap rules.
struct Range {
    uintptr_t lo = 0, hi = 0;  // [lo, hi)
    bool overlaps(const Range& o) const { return lo < o.hi && o.lo < hi; }
    bool same(const Range& o) const { return lo == o.lo && hi == o.hi; }
};

Range range_of(const void* p, int64_t bytes)
{
    Range r;
    r.lo = reinterpret_cast<uintptr_t>(p);
    r.hi = r.lo + static_cast<uintptr_t>(bytes);
    return r;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Outputs must not overlap one another.  A bf16 output may coincide exactly
// with x or residual (inputs 0 and 2: each element is read by the thread that
// later writes it, before it writes it); any other overlap with an input is
// rejected.
dradd_status check_overlaps(const Range* inputs, int n_in, const Range* outs, const bool* bf16_out, int n_out)
{
    for (int a = 0; a < n_out; ++a)
        for (int b = a + 1; b < n_out; ++b)
            if (outs[a].overlaps(outs[b]))
                return DRADD_ERR_ALIAS;
    for (int a = 0; a < n_out; ++a) {
        for (int b = 0; b < n_in; ++b) {
            if (!outs[a].overlaps(inputs[b]))
                continue;
            if (bf16_out[a] && b != 1 && outs[a].same(inputs[b]))
                continue;
            return DRADD_ERR_ALIAS;
        }
    }
    return DRADD_OK;
}

// Shape, pointers, eps and overlaps.  out/out_q/scale: whichever the variant
// writes (the others NULL).  Returns DRADD_OK with *noop set for n_rows == 0.
// add = false (plain RMSNorm): residual and residual_out are not used.
// out_kind: dradd::kOutBf16 writes out; the others write 1-byte codes to
// out_q (two e2m1 codes per byte) and a per-row scale.
dradd_status validate(int out_kind, bool add, const void* out, const void* out_q, const void* scale,
                      const void* residual_out, const void* x, const void* residual, const void* weight,
                      float eps, int64_t n_rows, int64_t hidden, bool* noop)
{
    const bool quant = out_kind != dradd::kOutBf16;
    *noop = false;
    if (n_rows < 0 || hidden <= 0)
        return DRADD_ERR_BAD_SHAPE;
    if (hidden % 8 != 0 || hidden > DRADD_MAX_HIDDEN)
        return DRADD_ERR_UNSUPPORTED_HIDDEN;
    if (n_rows > (INT64_MAX / 4) / hidden)
        return DRADD_ERR_BAD_SHAPE;
    if (n_rows == 0) {
        *noop = true;
        return DRADD_OK;
    }
    const void* primary_out = quant ? out_q : out;
    if (!primary_out || !x || !weight || (quant && !scale) || (add && (!residual_out || !residual)))
        return DRADD_ERR_NULL_PTR;
    if (!aligned(primary_out, 16) || !aligned(x, 16) || !aligned(weight, 16) ||
        (quant && !aligned(scale, 4)) || (add && (!aligned(residual_out, 16) || !aligned(residual, 16))))
        return DRADD_ERR_MISALIGNED;
    if (!std::isfinite(eps) || eps < 0.0f)
        return DRADD_ERR_BAD_EPS;

    const int64_t elems = n_rows * hidden;
    // inputs: x, weight[, residual]; outputs: the bf16 ones first.
    Range inputs[3];
    int n_in = 0;
    inputs[n_in++] = range_of(x, elems * 2);
    inputs[n_in++] = range_of(weight, hidden * 2);
    if (add)
        inputs[n_in++] = range_of(residual, elems * 2);
    Range outs[3];
    bool bf16_out[3] = {false, false, false};
    int n_out = 0;
    if (add) {
        bf16_out[n_out] = true;
        outs[n_out++] = range_of(residual_out, elems * 2);
    }
    if (quant) {
        outs[n_out++] = range_of(out_q, out_kind == dradd::kOutE2m1 ? elems / 2 : elems);
        outs[n_out++] = range_of(scale, n_rows * 4);
    } else {
        bf16_out[n_out] = true;
        outs[n_out++] = range_of(out, elems * 2);
    }
    return check_overlaps(inputs, n_in, outs, bf16_out, n_out);
}

// The split-row variant: a cluster of C CTAs per row (bf16 out only), each
// CTA a slice of P / C elements with T threads and K blocks of 8 per thread.
// Automatic: C = 2, T = slice blocks / 4 (at least 32, K at most 8), 2
// stages, as many clusters as fit.
dradd_status resolve_split(int64_t n_rows, int64_t hidden, bool quant, bool add, const DeviceLimits& L,
                           dradd_launch_cfg* cfg)
{
    const int64_t P = next_pow2(hidden);
    if (quant)
        return DRADD_ERR_BAD_CONFIG;
    const int C = cfg->cluster_ctas ? cfg->cluster_ctas : 2;
    if (C != 2 && C != 4)
        return DRADD_ERR_BAD_CONFIG;
    const int64_t slice_blocks = P / 8 / C;
    if (slice_blocks < 32)
        return DRADD_ERR_BAD_CONFIG;
    if (cfg->threads_per_row == 0) {
        int64_t T;
        if (cfg->blocks_per_thread != 0) {
            if (!is_pow2(cfg->blocks_per_thread) || slice_blocks % cfg->blocks_per_thread != 0)
                return DRADD_ERR_BAD_CONFIG;
            T = slice_blocks / cfg->blocks_per_thread;
        } else {
            T = slice_blocks / 4 < 32 ? 32 : slice_blocks / 4;
            while (slice_blocks / T > 8)
                T *= 2;
            if (T > slice_blocks)
                T = slice_blocks;
        }
        cfg->threads_per_row = static_cast<int>(T);
    }
    const int T = cfg->threads_per_row;
    if (!is_pow2(T) || T < 32 || T > 1024 || slice_blocks % T != 0)
        return DRADD_ERR_BAD_CONFIG;
    const int64_t K = slice_blocks / T;
    if ((K != 1 && K != 2 && K != 4 && K != 8) || T > dradd::max_threads_for(static_cast<int>(K)) ||
        (cfg->blocks_per_thread != 0 && cfg->blocks_per_thread != K))
        return DRADD_ERR_BAD_CONFIG;
    cfg->blocks_per_thread = static_cast<int>(K);
    if (cfg->rows_per_cta == 0)
        cfg->rows_per_cta = 1;
    if (cfg->rows_per_cta != 1 || cfg->wait_limit_us < 0 || (cfg->serialize != 0 && cfg->serialize != 1) ||
        cfg->fault_inject < 0)
        return DRADD_ERR_BAD_CONFIG;
    const int64_t stage_bytes = (add ? 4 : 2) * (P / C);
    const int64_t static_smem = static_cast<int64_t>(dradd::split_static_smem(static_cast<int>(K)));
    const int64_t avail = L.smem_per_block_optin - static_smem - 8 * 8;
    if (cfg->stages == 0) {
        const int64_t S = avail / stage_bytes;
        cfg->stages = static_cast<int>(S > 2 ? 2 : S);
    }
    const int S = cfg->stages;
    if (S < 1 || S > 8 || S * stage_bytes > avail)
        return DRADD_ERR_BAD_CONFIG;
    if (cfg->grid_ctas == 0) {
        int ctas_per_sm = L.max_threads_per_sm / T;
        if (ctas_per_sm > L.max_blocks_per_sm)
            ctas_per_sm = L.max_blocks_per_sm;
        const int64_t per_cta = S * stage_bytes + static_smem + 8 * S + 1024;
        if (L.smem_per_sm / per_cta < ctas_per_sm)
            ctas_per_sm = static_cast<int>(L.smem_per_sm / per_cta);
        int64_t clusters = static_cast<int64_t>(L.sm_count) * (ctas_per_sm > 0 ? ctas_per_sm : 1) / C;
        if (clusters > n_rows)
            clusters = n_rows;
        if (clusters < 1)
            clusters = 1;
        if (clusters * C > 0x7FFFFFFF)
            clusters = 0x7FFFFFFF / C;
        cfg->grid_ctas = static_cast<int>(clusters * C);
    }
    if (cfg->grid_ctas < C || cfg->grid_ctas % C != 0)
        return DRADD_ERR_BAD_CONFIG;
    cfg->cluster_ctas = C;
    return DRADD_OK;
}

// The warp-per-row variant: K = P / 256 blocks per lane, one warp a row,
// rows_per_cta warps (and rows per stage) per CTA, `stages` stages.
// Automatic: the most warps (up to kWarpMaxRows) for which 2 stages fit in
// one CTA's shared memory, 2 stages.
dradd_status resolve_warp(int64_t n_rows, int64_t hidden, bool add, const DeviceLimits& L,
                           dradd_launch_cfg* cfg)
{
    const int64_t blocks = next_pow2(hidden) / 8;
    if (blocks < 32 || blocks / 32 > 16 || (add && blocks / 32 > 8))
        return DRADD_ERR_BAD_CONFIG;
    const int K = static_cast<int>(blocks / 32);
    if (cfg->threads_per_row == 0)
        cfg->threads_per_row = 32;
    if (cfg->blocks_per_thread == 0)
        cfg->blocks_per_thread = K;
    if (cfg->threads_per_row != 32 || cfg->blocks_per_thread != K || cfg->cluster_ctas != 0 ||
        cfg->wait_limit_us < 0 || (cfg->serialize != 0 && cfg->serialize != 1) || cfg->grid_ctas < 0 ||
        cfg->fault_inject < 0 || cfg->rows_per_cta < 0 || cfg->rows_per_cta > dradd::kWarpMaxRows ||
        cfg->stages < 0 || cfg->stages > 8)
        return DRADD_ERR_BAD_CONFIG;
    const int64_t limit = L.smem_per_block_optin - 1024;
    const int S0 = cfg->stages != 0 ? cfg->stages : 2;
    if (cfg->rows_per_cta == 0) {
        int R = dradd::kWarpMaxRows;
        while (R > 1 && static_cast<int64_t>(dradd::warp_smem_bytes(S0, R, static_cast<int>(hidden), add)) > limit)
            --R;
        cfg->rows_per_cta = R;
    }
    if (cfg->stages == 0)
        cfg->stages = S0;
    const int64_t smem = static_cast<int64_t>(
        dradd::warp_smem_bytes(cfg->stages, cfg->rows_per_cta, static_cast<int>(hidden), add));
    if (smem > limit)
        return DRADD_ERR_BAD_CONFIG;
    if (cfg->grid_ctas == 0) {
        // as many CTAs as fit at once (the launch refines this with the
        // kernel's occupancy), at most one per group of rows
        int64_t per_sm = L.smem_per_sm / (smem + 1024);
        const int64_t by_threads = L.max_threads_per_sm / (32 * cfg->rows_per_cta);
        if (by_threads < per_sm)
            per_sm = by_threads;
        const int64_t groups = (n_rows + cfg->rows_per_cta - 1) / cfg->rows_per_cta;
        int64_t grid = static_cast<int64_t>(L.sm_count) * (per_sm > 0 ? per_sm : 1);
        if (grid > groups)
            grid = groups;
        cfg->grid_ctas = static_cast<int>(grid < 1 ? 1 : grid);
    }
    return DRADD_OK;
}

// Fill the automatic fields of *cfg and check the explicit ones.
dradd_status resolve(int64_t n_rows, int64_t hidden, bool quant, bool add, const DeviceLimits& L,
                     dradd_launch_cfg* cfg)
{
    if (n_rows < 0 || hidden <= 0)
        return DRADD_ERR_BAD_SHAPE;
    if (hidden % 8 != 0 || hidden > DRADD_MAX_HIDDEN)
        return DRADD_ERR_UNSUPPORTED_HIDDEN;
    const int64_t P = next_pow2(hidden);
    const int64_t blocks = P / 8;

    // Automatic choice, measured on GB300 (back-to-back launches over buffers
    // larger than L2, median of interleaved rounds, with the staged
    // kernel's L2 prefetch of its first rows).  Rows of up to 256
    // elements go several to a CTA in registers; longer rows are staged
    // through shared memory, mostly with K = 4 blocks of 8 per thread:
    //   P      T     K  stages (residual-add forms)   stages (plain RMSNorm)
    //   512    32    2  4                             4
    //   1024   64    2  3                             2
    //   2048   128   2  4 (64 rows per SM or more:    T = 64, K = 4: 2
    //                      T = 64, K = 4, 3 stages;
    //                      quantised: T = 64, K = 4,
    //                      1 stage below 32 rows per
    //                      SM, else 3)
    //   4096   128   4  bf16: 3 below 24 rows per SM,  bf16: 4 from 20 to 63
    //                   2 below 64, else 1;           rows per SM, else 2;
    //                   quantised: 2 below 44, else 1 quantised: 2
    //          (bf16 residual-add batches of up to 256 rows: T = 256, K = 2;
    //          quantised residual-add, int8: 48 rows per SM 33.87 us with 1
    //          stage against 34.63 with 2, 32 rows per SM 23.14 with 2 against
    //          23.62 with 1; plain quantised, 4096 x 4096: int8 13.51 us with 2
    //          stages against 13.85 with 1, e4m3 14.91 against 15.04)
    //   8192   1024  1  2                             T = 512, K = 2: 3
    //          (bf16 residual-add batches of 65..512 rows, and the quantised
    //          residual-add forms: T = 512, K = 2)
    //   16384  512   4  2                             4
    //   32768  512   8  1                             2
    //
    // These shapes go elsewhere (same measurements):
    //   - bf16 out, P = 32768 and at most 160 rows: the split-row cluster
    //     variant, 4 CTAs a row up to 64 rows, else 2 (one row: 3.2 us
    //     against 8.8 us staged; 152 rows: 10.5 against 11.4);
    //   - plain RMSNorm with quantised out, 1024 <= P <= 16384 except
    //     P = 4096 beyond 4 rows per SM: the staged pair kernel (two rows
    //     per thread), one stage, K = 2 up to P = 2048 and K = 4 beyond,
    //     K = 1 for at most 4 rows per SM (int8: 16384 x 1024 12.70
    //     against 14.61 us, 8192 x 2048 12.72 against 13.47, 2048 x 8192
    //     14.61 against 16.52, 1024 x 16384 17.51 against 17.95, 512 x 4096
    //     3.84 against 4.87; at 4096 x 4096 int8 a tie, 13.73 against
    //     13.74, and e4m3 slower, 15.47 against 14.95); at P = 512 one
    //     stage, the pair kernel with K = 1 below 8192 rows, else one row
    //     a CTA with K = 2 (below);
    //   - 512 <= P <= 2048 with enough rows: the warp-per-row variant
    //     (residual-add bf16 from 1024 rows, 4 warps and 3 stages: 4096 x
    //     1024 in 5.27 us against 6.83; quantised residual-add at P <= 1024
    //     from 2048 rows, 4 warps and 2 stages; plain bf16 from 16384 rows,
    //     8 warps and 3 stages).
    const bool auto_variant = cfg->variant == DRADD_VARIANT_AUTO;
    if (auto_variant) {
        cfg->variant = hidden > 256 ? DRADD_VARIANT_STAGED : DRADD_VARIANT_ROWS;
        const bool no_explicit = cfg->threads_per_row == 0 && cfg->rows_per_cta == 0 && cfg->stages == 0 &&
                                 cfg->blocks_per_thread == 0 && cfg->fault_inject == 0 && cfg->cluster_ctas == 0;
        if (no_explicit && !quant && P >= 32768 && n_rows <= 160) {
            cfg->variant = DRADD_VARIANT_SPLIT;
            cfg->cluster_ctas = n_rows <= 64 ? 4 : 2;
        } else if (no_explicit && !add && quant && P == 512) {
            // one stage; below 8192 rows the pair kernel with K = 1, else
            // one row a CTA with K = 2 (4096 rows: 4.29 us against 4.85 for
            // 4 stages of single rows; 16384 rows: 7.57 against 9.40 for
            // one warp a row)
            cfg->variant = DRADD_VARIANT_STAGED;
            cfg->stages = 1;
            if (n_rows < 8192) {
                cfg->rows_per_cta = 2;
                cfg->threads_per_row = 64;
            } else {
                cfg->threads_per_row = 32;
            }
        } else if (no_explicit && !add && quant && P >= 1024 && P <= 16384 &&
                   (P != 4096 || n_rows <= 4 * static_cast<int64_t>(L.sm_count))) {
            // the pair kernel, one stage: K = 1 for batches of at most 4
            // rows per SM (up to 512 threads), else K = 2 up to P = 2048
            // and K = 4 beyond (at P = 4096 only the small batches)
            const int64_t b = P / 8;
            const bool few = n_rows <= 4 * static_cast<int64_t>(L.sm_count) && b <= 512;
            const int64_t T = few ? b : P <= 2048 ? b / 2 : b / 4;
            cfg->variant = DRADD_VARIANT_STAGED;
            cfg->rows_per_cta = 2;
            cfg->threads_per_row = static_cast<int>(T);
            cfg->stages = 1;
        } else if (no_explicit && P >= 512 && P <= 2048) {
            int R = 0, S = 0;
            if (add && !quant && n_rows >= 1024) {
                R = 4;
                S = 3;
            } else if (add && quant && n_rows >= 2048 && P < 2048) {
                R = 4;
                S = 2;
            } else if (!add && !quant && n_rows >= 16384) {
                R = 8;
                S = 3;
            }
            if (R != 0) {
                cfg->variant = DRADD_VARIANT_WARP;
                cfg->rows_per_cta = R;
                cfg->stages = S;
            }
        }
    }
    if (cfg->variant == DRADD_VARIANT_SPLIT)
        return resolve_split(n_rows, hidden, quant, add, L, cfg);
    if (cfg->variant == DRADD_VARIANT_WARP)
        return resolve_warp(n_rows, hidden, add, L, cfg);
    if (cfg->cluster_ctas != 0)
        return DRADD_ERR_BAD_CONFIG;
    if (cfg->variant != DRADD_VARIANT_ROWS && cfg->variant != DRADD_VARIANT_STAGED)
        return DRADD_ERR_BAD_CONFIG;
    const bool staged = cfg->variant == DRADD_VARIANT_STAGED;

    int auto_stages = 2;
    const int64_t per_sm = n_rows / (L.sm_count > 0 ? L.sm_count : 1);  // rows per SM
    if (cfg->threads_per_row == 0 && cfg->blocks_per_thread != 0) {
        if (!is_pow2(cfg->blocks_per_thread) || cfg->blocks_per_thread > 8 || blocks % cfg->blocks_per_thread != 0)
            return DRADD_ERR_BAD_CONFIG;
        cfg->threads_per_row = static_cast<int>(blocks / cfg->blocks_per_thread);
    }
    if (cfg->threads_per_row == 0) {
        int64_t T;
        if (!staged) {
            T = blocks < 512 ? blocks : 512;
        } else if (P <= 512) {
            T = blocks / 2 < 32 ? 32 : blocks / 2;
            auto_stages = 4;
        } else if (P == 1024) {
            T = 64;
            auto_stages = add ? 3 : 2;
        } else if (P == 2048) {
            const bool wide = add && per_sm < 64;
            T = wide ? 128 : 64;
            auto_stages = wide ? 4 : (add ? 3 : 2);
            if (add && quant) {
                // quantised residual-add: 64 threads, K = 4 (2048 rows, 1
                // stage: 6.63 us against 8.37 one warp a row; 8192 rows, 3
                // stages: 19.20 against 20.72)
                T = 64;
                auto_stages = per_sm < 32 ? 1 : 3;
            }
        } else if (P == 4096) {
            // small bf16 batches (up to 256 rows): 256 threads, K = 2
            T = add && !quant && n_rows <= 256 ? 256 : 128;
            if (add && !quant)
                auto_stages = per_sm < 24 ? 3 : (per_sm < 64 ? 2 : 1);
            else if (add)
                auto_stages = per_sm < 44 ? 2 : 1;
            else if (!quant)
                auto_stages = per_sm < 20 || per_sm >= 64 ? 2 : 4;
            else
                auto_stages = 2;
        } else if (P == 8192) {
            // bf16 residual-add: 1024 threads, K = 1 (65..512-row batches:
            // 512 threads, K = 2); quantised residual-add and plain: 512
            // threads, K = 2 (int8 4096 x 8192: 38.27 us against 42.67 with
            // 1024 threads; 2048 x 8192: 19.55 against 23.04)
            T = add && !quant && (n_rows <= 64 || n_rows > 512) ? 1024 : 512;
            auto_stages = add ? 2 : 3;
        } else {
            T = 512;
            auto_stages = P == 16384 ? (add ? 2 : 4) : (add ? 1 : 2);
        }
        if (T > blocks)
            T = blocks;
        while (blocks / T > 8)
            T *= 2;
        cfg->threads_per_row = static_cast<int>(T);
    }
    const int T = cfg->threads_per_row;
    if (!is_pow2(T) || T > 1024 || blocks % T != 0)
        return DRADD_ERR_BAD_CONFIG;
    const int64_t K = blocks / T;
    if ((K != 1 && K != 2 && K != 4 && K != 8) || (cfg->blocks_per_thread != 0 && cfg->blocks_per_thread != K))
        return DRADD_ERR_BAD_CONFIG;
    cfg->blocks_per_thread = static_cast<int>(K);
    if (staged && T < 32)
        return DRADD_ERR_BAD_CONFIG;

    if (cfg->rows_per_cta == 0)
        cfg->rows_per_cta = staged ? 1 : (T < 128 ? static_cast<int>(128 / T) : 1);
    const int R = cfg->rows_per_cta;
    // staged with R = 2: the plain quantised forms' pair kernel (two rows
    // per thread, T threads a CTA, K <= 4)
    const bool pair = staged && R == 2;
    if (pair) {
        if (add || !quant || K > 4 || T > dradd::max_threads_for(static_cast<int>(2 * K)))
            return DRADD_ERR_BAD_CONFIG;
    } else if (R < 1 || static_cast<int64_t>(T) * R > dradd::max_threads_for(static_cast<int>(K)) ||
               (T * R) % 32 != 0 || (staged && R != 1)) {
        return DRADD_ERR_BAD_CONFIG;
    }

    const int threads = pair ? T : T * R;
    int ctas_per_sm = L.max_threads_per_sm / threads;
    if (ctas_per_sm > L.max_blocks_per_sm)
        ctas_per_sm = L.max_blocks_per_sm;
    if (staged) {
        const int64_t stage_bytes = (add ? 4 : 2) * hidden * R;
        const int64_t static_smem = static_cast<int64_t>(dradd::staged_static_smem(static_cast<int>(K), pair));
        // the quantised outputs keep the row's weights in fp32 beside the stages
        const int64_t weight_bytes = quant ? 4 * hidden : 0;
        const int64_t avail = L.smem_per_block_optin - static_smem - weight_bytes - 8 * 8;
        if (auto_variant && avail < stage_bytes) {
            // not even one stage fits beside the weights: registers instead
            cfg->variant = DRADD_VARIANT_ROWS;
            cfg->threads_per_row = 0;
            cfg->blocks_per_thread = 0;
            cfg->stages = 0;
            return resolve(n_rows, hidden, quant, add, L, cfg);
        }
        if (cfg->stages == 0) {
            int64_t S = avail / stage_bytes;
            cfg->stages = static_cast<int>(S > auto_stages ? auto_stages : S);
        }
        const int S = cfg->stages;
        if (S < 1 || S > 8 || S * stage_bytes > avail)
            return DRADD_ERR_BAD_CONFIG;
        const int64_t per_cta = S * stage_bytes + weight_bytes + static_smem + 8 * S + 1024;  // 1 KiB reserved per CTA
        const int64_t by_smem = L.smem_per_sm / per_cta;
        if (by_smem < ctas_per_sm)
            ctas_per_sm = static_cast<int>(by_smem);
        if (ctas_per_sm < 1)
            return DRADD_ERR_BAD_CONFIG;
    } else if (cfg->stages != 0 || cfg->fault_inject != 0) {
        return DRADD_ERR_BAD_CONFIG;
    }
    if (cfg->wait_limit_us < 0 || (cfg->serialize != 0 && cfg->serialize != 1))
        return DRADD_ERR_BAD_CONFIG;

    if (cfg->grid_ctas == 0) {
        const int64_t groups = (n_rows + R - 1) / R;
        int64_t grid;
        if (staged)
            grid = static_cast<int64_t>(L.sm_count) * ctas_per_sm;
        else
            grid = groups;
        if (grid > groups)
            grid = groups;
        if (grid > 0x7FFFFFFF)
            grid = 0x7FFFFFFF;
        if (grid < 1)
            grid = 1;
        cfg->grid_ctas = static_cast<int>(grid);
    }
    if (cfg->grid_ctas < 1)
        return DRADD_ERR_BAD_CONFIG;
    return DRADD_OK;
}

// out_kind: dradd::kOutBf16 (writes out), kOutInt8 or kOutE4m3 (writes the
// 1-byte codes to out_q and the per-row scale).
dradd_status run(int out_kind, bool add, dradd_bf16* out, int8_t* out_q, float* scale,
                 dradd_bf16* residual_out, const dradd_bf16* x, const dradd_bf16* residual,
                 const dradd_bf16* weight, float eps, int64_t n_rows, int64_t hidden, cudaStream_t stream,
                 const dradd_launch_cfg* user_cfg)
{
    const bool quant = out_kind != dradd::kOutBf16;
    bool noop = false;
    dradd_status st = validate(out_kind, add, out, out_q, scale, residual_out, x, residual, weight, eps, n_rows,
                               hidden, &noop);
    if (st != DRADD_OK || noop)
        return st;
    DeviceLimits L;
    st = query_limits(&L);
    if (st != DRADD_OK)
        return st;
    dradd_launch_cfg cfg = {};
    if (user_cfg)
        cfg = *user_cfg;
    const bool auto_grid = cfg.grid_ctas == 0;
    const bool device_memory = all_device_memory({out, out_q, scale, residual_out, x, residual, weight});
    if (!device_memory) {
        // host memory (read and written over the host link): register loads
        // only, so no variant that stages rows with bulk copies
        if (cfg.variant == DRADD_VARIANT_STAGED || cfg.variant == DRADD_VARIANT_SPLIT)
            return DRADD_ERR_BAD_CONFIG;
        if (cfg.variant == DRADD_VARIANT_WARP)
            return DRADD_ERR_BAD_CONFIG;
        cfg.variant = DRADD_VARIANT_ROWS;
    }
    st = resolve(n_rows, hidden, quant, add, L, &cfg);
    if (st != DRADD_OK)
        return st;
    if (cfg.variant == DRADD_VARIANT_WARP) {
        if (!device_memory)
            return DRADD_ERR_BAD_CONFIG;  // bulk copies read device memory only
        const int Kw = cfg.blocks_per_thread;
        const int threads = 32 * cfg.rows_per_cta;
        const size_t dyn_w = dradd::warp_smem_bytes(cfg.stages, cfg.rows_per_cta, static_cast<int>(hidden), add);
        int grid = cfg.grid_ctas;
        const int64_t groups = (n_rows + cfg.rows_per_cta - 1) / cfg.rows_per_cta;
        if (auto_grid) {
            int per_sm = 0;
            if (dradd::warp_occupancy(Kw, out_kind, add, threads, dyn_w, &per_sm) != cudaSuccess)
                return DRADD_ERR_CUDA;
            int64_t g = static_cast<int64_t>(L.sm_count) * (per_sm > 0 ? per_sm : 1);
            if (g > groups)
                g = groups;
            grid = static_cast<int>(g);
        }
        Params p = {};
        p.out = out;
        p.out_q = out_q;
        p.scale = scale;
        p.residual_out = residual_out;
        p.x = x;
        p.residual = residual;
        p.weight = weight;
        p.eps = eps;
        p.hidden = static_cast<int>(hidden);
        p.inv_hidden = is_pow2(hidden) ? 1.0f / static_cast<float>(hidden) : 0.0f;
        p.n_rows = n_rows;
        p.threads_per_row = 32;
        p.rows_per_cta = cfg.rows_per_cta;
        p.stages = cfg.stages;
        p.fault_inject = cfg.fault_inject;
        p.wait_limit_ns = cfg.wait_limit_us > 0 ? static_cast<uint64_t>(cfg.wait_limit_us) * 1000ull
                                                : kDefaultWaitLimitNs;
        p.l2_prefetch = 1;
        if (dradd::device_status_ptr(&p.status) != cudaSuccess)
            return DRADD_ERR_CUDA;
        return dradd::launch_warp(p, Kw, out_kind, add, grid, threads, dyn_w, cfg.serialize != 0, stream) ==
                       cudaSuccess
                   ? DRADD_OK
                   : DRADD_ERR_CUDA;
    }
    if (cfg.variant == DRADD_VARIANT_SPLIT) {
        const int C = cfg.cluster_ctas;
        const int Ks = cfg.blocks_per_thread;
        const size_t dyn_s = static_cast<size_t>(cfg.stages) *
                                 ((add ? 4 : 2) * static_cast<size_t>(next_pow2(hidden) / C) + 8);
        int grid = cfg.grid_ctas;
        if (auto_grid) {
            int clusters = 0;
            if (dradd::split_max_clusters(Ks, C, add, cfg.threads_per_row, dyn_s, &clusters) != cudaSuccess)
                return DRADD_ERR_CUDA;
            int64_t c = clusters > 0 ? clusters : 1;
            if (c > n_rows)
                c = n_rows;
            grid = static_cast<int>(c * C);
        }
        Params p = {};
        p.out = out;
        p.residual_out = residual_out;
        p.x = x;
        p.residual = residual;
        p.weight = weight;
        p.eps = eps;
        p.hidden = static_cast<int>(hidden);
        p.inv_hidden = is_pow2(hidden) ? 1.0f / static_cast<float>(hidden) : 0.0f;
        p.n_rows = n_rows;
        p.threads_per_row = cfg.threads_per_row;
        p.rows_per_cta = 1;
        p.stages = cfg.stages;
        p.fault_inject = cfg.fault_inject;
        p.wait_limit_ns = cfg.wait_limit_us > 0 ? static_cast<uint64_t>(cfg.wait_limit_us) * 1000ull
                                                : kDefaultWaitLimitNs;
        if (dradd::device_status_ptr(&p.status) != cudaSuccess)
            return DRADD_ERR_CUDA;
        return dradd::launch_split(p, Ks, C, add, grid, cfg.threads_per_row, dyn_s, cfg.serialize != 0, stream) ==
                       cudaSuccess
                   ? DRADD_OK
                   : DRADD_ERR_CUDA;
    }
    const int K = static_cast<int>(next_pow2(hidden) / 8 / cfg.threads_per_row);
    const bool pair = cfg.variant == DRADD_VARIANT_STAGED && cfg.rows_per_cta == 2;
    const size_t dyn = cfg.variant == DRADD_VARIANT_STAGED
                           ? static_cast<size_t>(cfg.stages) * (add ? 4 : 2) * static_cast<size_t>(hidden) *
                                     static_cast<size_t>(cfg.rows_per_cta) +
                                 dradd::staged_weight_bytes(out_kind, static_cast<int>(hidden)) +
                                 8 * static_cast<size_t>(cfg.stages)
                           : 0;
    if (auto_grid && cfg.variant == DRADD_VARIANT_STAGED) {
        // persistent grid: as many CTAs as fit on the device at once, at
        // most one per unit (row, or pair of rows)
        int per_sm = 0;
        if (dradd::staged_occupancy(K, out_kind, add, cfg.threads_per_row, dyn, &per_sm, pair) != cudaSuccess)
            return DRADD_ERR_CUDA;
        int64_t grid = static_cast<int64_t>(L.sm_count) * (per_sm > 0 ? per_sm : 1);
        const int64_t units = pair ? (n_rows + 1) / 2 : n_rows;
        if (grid > units)
            grid = units;
        cfg.grid_ctas = static_cast<int>(grid);
    }

    Params p = {};
    p.out = out;
    p.out_q = out_q;
    p.scale = scale;
    p.residual_out = residual_out;
    p.x = x;
    p.residual = residual;
    p.weight = weight;
    p.eps = eps;
    p.hidden = static_cast<int>(hidden);
    p.inv_hidden = is_pow2(hidden) ? 1.0f / static_cast<float>(hidden) : 0.0f;
    p.n_rows = n_rows;
    p.threads_per_row = cfg.threads_per_row;
    p.rows_per_cta = cfg.rows_per_cta;
    p.stages = cfg.stages;
    p.fault_inject = cfg.fault_inject;
    p.wait_limit_ns = cfg.wait_limit_us > 0 ? static_cast<uint64_t>(cfg.wait_limit_us) * 1000ull
                                            : kDefaultWaitLimitNs;
    p.l2_prefetch = device_memory ? 1 : 0;
    if (dradd::device_status_ptr(&p.status) != cudaSuccess)
        return DRADD_ERR_CUDA;
    cudaError_t e;
    if (cfg.variant == DRADD_VARIANT_STAGED) {
        e = dradd::launch_staged(p, K, out_kind, add, cfg.grid_ctas, cfg.threads_per_row, dyn,
                                 cfg.serialize != 0, stream);
    } else {
        e = dradd::launch_rows(p, K, out_kind, add, cfg.grid_ctas, cfg.threads_per_row * cfg.rows_per_cta,
                               cfg.serialize != 0, stream);
    }
    return e == cudaSuccess ? DRADD_OK : DRADD_ERR_CUDA;
}

// ---------------------------------------------------------- fused q/k RMSNorm
struct QkSide {
    bool active = false;
    int64_t n_rows = 0, hidden = 0;
    int K = 0, T = 0, R = 0, stages = 0;
    int64_t ctas = 0, stage_bytes = 0;
};

struct QkLaunch {
    QkSide q, k;
    int threads = 0;
    bool staged = false, warp = false, chunk = false, serialize = false;
    int64_t dyn_smem = 0;
};

constexpr int64_t kQkStageBudget = 96 * 1024;  // automatic stages: bytes per CTA

dradd_status qk_check_side(int64_t n_rows, int64_t hidden)
{
    if (hidden <= 0)
        return DRADD_ERR_BAD_SHAPE;
    if (hidden % 8 != 0 || hidden > DRADD_QK_MAX_HIDDEN)
        return DRADD_ERR_UNSUPPORTED_HIDDEN;
    if (n_rows > (INT64_MAX / 4) / hidden)
        return DRADD_ERR_BAD_SHAPE;
    return DRADD_OK;
}

// The warp-per-row plan of the fused q/k call (DRADD_VARIANT_WARP): each
// side one warp a row, K = P / 256 blocks of 8 per lane (1..8, so
// 256 <= P <= 2048 on both sides), threads_per_row read as the threads of a
// CTA (a multiple of 32 up to 256, 0 = 256: one row of each side per warp
// and stage), stages per side (0 = 2); CTAs split between the sides as in
// qk_plan.  Dynamic shared memory: the larger side's warp_smem_bytes.
dradd_status qk_plan_warp(int64_t n_q, int64_t hq, int64_t n_k, int64_t hk, bool add, int sm_count,
                          int ctas_per_sm, int smem_optin, const dradd_launch_cfg& cfg, QkLaunch* out)
{
    QkSide* q = &out->q;
    QkSide* k = &out->k;
    if (cfg.rows_per_cta != 0 || cfg.fault_inject < 0 || cfg.blocks_per_thread != 0 || cfg.cluster_ctas != 0 ||
        cfg.grid_ctas < 0 || cfg.wait_limit_us < 0 || cfg.stages < 0 || cfg.stages > 8 ||
        (cfg.serialize != 0 && cfg.serialize != 1))
        return DRADD_ERR_BAD_CONFIG;
    const int64_t B = cfg.threads_per_row != 0 ? cfg.threads_per_row : 256;
    if (B < 32 || B > 256 || B % 32 != 0)
        return DRADD_ERR_BAD_CONFIG;
    out->warp = true;
    out->staged = false;
    out->serialize = cfg.serialize != 0;
    const int S = cfg.stages != 0 ? cfg.stages : 2;
    for (QkSide* side : {q, k}) {
        if (!side->active)
            continue;
        const int64_t blocks = next_pow2(side->hidden) / 8;
        if (blocks < 32 || blocks / 32 > 8)
            return DRADD_ERR_BAD_CONFIG;
        side->K = static_cast<int>(blocks / 32);
        side->T = 32;
        side->R = static_cast<int>(B / 32);
        side->stages = S;
        const int64_t need = static_cast<int64_t>(
            dradd::warp_smem_bytes(S, side->R, static_cast<int>(side->hidden), side == q && add));
        if (need > smem_optin - 1024)
            return DRADD_ERR_BAD_CONFIG;
        if (need > out->dyn_smem)
            out->dyn_smem = need;
    }
    const int64_t need_q = q->active ? (n_q + q->R - 1) / q->R : 0;
    const int64_t need_k = k->active ? (n_k + k->R - 1) / k->R : 0;
    int64_t C = cfg.grid_ctas;
    if (C == 0)
        C = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * (ctas_per_sm > 0 ? ctas_per_sm : 2048 / B);
    if (C < (q->active ? 1 : 0) + (k->active ? 1 : 0))
        return DRADD_ERR_BAD_CONFIG;
    if (need_q + need_k <= C) {
        q->ctas = need_q;
        k->ctas = need_k;
    } else {
        const double wq = q->active ? static_cast<double>(n_q) * static_cast<double>(hq) : 0.0;
        const double wk = k->active ? static_cast<double>(n_k) * static_cast<double>(hk) : 0.0;
        int64_t cq = q->active ? static_cast<int64_t>(static_cast<double>(C) * wq / (wq + wk) + 0.5) : 0;
        if (q->active && cq < 1)
            cq = 1;
        if (k->active && cq > C - 1)
            cq = C - 1;
        if (cq > need_q)
            cq = need_q;
        int64_t ck = C - cq;
        if (ck > need_k)
            ck = need_k;
        q->ctas = cq;
        k->ctas = ck;
    }
    if (q->ctas + k->ctas > 0x7FFFFFFF)
        return DRADD_ERR_BAD_CONFIG;
    out->threads = static_cast<int>(B);
    return DRADD_OK;
}

// The chunked-q plan (DRADD_VARIANT_CHUNK): the q rows (512 < P <= 4096)
// in 512-element chunks, one warp a chunk and one CTA a row; the k rows
// one warp each (256 <= P <= 2048) in CTAs of the same number of warps.
// Both sides get `stages` ring slots per warp (0 = 2).  CTAs (grid_ctas):
// automatic SMs x ctas_per_sm (<= 0: 2048 / threads); when the two sides
// need more, they share them in proportion to their elements.
dradd_status qk_plan_chunk(int64_t n_q, int64_t hq, int64_t n_k, int64_t hk, bool add, int sm_count,
                           int ctas_per_sm, int smem_optin, const dradd_launch_cfg& cfg, QkLaunch* out)
{
    QkSide* q = &out->q;
    QkSide* k = &out->k;
    if (cfg.rows_per_cta != 0 || cfg.threads_per_row != 0 || cfg.blocks_per_thread != 0 || cfg.cluster_ctas != 0 ||
        cfg.fault_inject < 0 || cfg.grid_ctas < 0 || cfg.wait_limit_us < 0 || cfg.stages < 0 || cfg.stages > 8 ||
        (cfg.serialize != 0 && cfg.serialize != 1))
        return DRADD_ERR_BAD_CONFIG;
    if (!q->active)
        return DRADD_ERR_BAD_CONFIG;  // the variant is defined by its q rows
    const int64_t pq = next_pow2(hq);
    if (pq <= 512 || pq > 4096)
        return DRADD_ERR_BAD_CONFIG;
    const int nw = static_cast<int>((hq + dradd::kChunkElems - 1) / dradd::kChunkElems);
    const int S = cfg.stages != 0 ? cfg.stages : 2;
    out->chunk = true;
    out->staged = false;
    out->warp = false;
    out->serialize = cfg.serialize != 0;
    out->threads = 32 * nw;
    q->K = dradd::kChunkBlocks / 32;
    q->T = 32 * nw;
    q->R = 1;
    q->stages = S;
    out->dyn_smem = static_cast<int64_t>(dradd::chunk_smem_bytes(S, nw, static_cast<int>(hq), add));
    if (k->active) {
        const int64_t blocks = next_pow2(hk) / 8;
        if (blocks < 32 || blocks / 32 > 8)
            return DRADD_ERR_BAD_CONFIG;
        k->K = static_cast<int>(blocks / 32);
        k->T = 32;
        k->R = nw;
        k->stages = S;
        const int64_t need = static_cast<int64_t>(dradd::warp_smem_bytes(S, nw, static_cast<int>(hk), false));
        if (need > out->dyn_smem)
            out->dyn_smem = need;
    }
    if (out->dyn_smem > smem_optin - 1024)
        return DRADD_ERR_BAD_CONFIG;
    const int64_t need_q = n_q;
    const int64_t need_k = k->active ? (n_k + nw - 1) / nw : 0;
    int64_t C = cfg.grid_ctas;
    if (C == 0)
        C = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * (ctas_per_sm > 0 ? ctas_per_sm : 2048 / out->threads);
    if (C < 1 + (k->active ? 1 : 0))
        return DRADD_ERR_BAD_CONFIG;
    if (need_q + need_k <= C) {
        q->ctas = need_q;
        k->ctas = need_k;
    } else {
        const double wq = static_cast<double>(n_q) * static_cast<double>(hq);
        const double wk = k->active ? static_cast<double>(n_k) * static_cast<double>(hk) : 0.0;
        int64_t cq = static_cast<int64_t>(static_cast<double>(C) * wq / (wq + wk) + 0.5);
        if (cq < 1)
            cq = 1;
        if (k->active && cq > C - 1)
            cq = C - 1;
        if (cq > need_q)
            cq = need_q;
        int64_t ck = C - cq;
        if (ck > need_k)
            ck = need_k;
        q->ctas = cq;
        k->ctas = ck;
    }
    if (q->ctas + k->ctas > 0x7FFFFFFF)
        return DRADD_ERR_BAD_CONFIG;
    return DRADD_OK;
}

// Shapes and the launch plan of the fused q/k call.  A side with no rows
// takes no part.  Variant, threads per CTA B (cfg->threads_per_row) and a
// least K (cfg->blocks_per_thread) default to the table below.  Each side
// takes K = the smallest power of two with P / 8 / K <= B, raised to the
// least K if that is larger (at most P / 8 and 8); then T = P / 8 / K
// threads per row and R = B / T rows per CTA.  The staged variant gives
// each side min(S, 96 KiB / stage) stages of R rows, S = 3 for short rows
// in large batches and 2 otherwise (cfg->stages: the same
// count for both).  CTAs (cfg->grid_ctas):
// automatic SMs x ctas_per_sm (ctas_per_sm <= 0: 2048 / B); when the two
// sides need more, they share them in proportion to their elements.
dradd_status qk_plan(int64_t n_q, int64_t hq, int64_t n_k, int64_t hk, int64_t group_size, bool add,
                     int sm_count, int ctas_per_sm, int smem_optin, const dradd_launch_cfg* cfg_in, QkLaunch* out)
{
    QkSide* q = &out->q;
    QkSide* k = &out->k;
    *q = QkSide{};
    *k = QkSide{};
    out->threads = 0;
    out->dyn_smem = 0;
    if (n_q < 0 || n_k < 0 || group_size < 0)
        return DRADD_ERR_BAD_SHAPE;
    q->active = n_q > 0;
    k->active = n_k > 0;
    q->n_rows = n_q;
    k->n_rows = n_k;
    q->hidden = hq;
    k->hidden = hk;
    dradd_status st;
    if (q->active && (st = qk_check_side(n_q, hq)) != DRADD_OK)
        return st;
    if (k->active && (st = qk_check_side(n_k, hk)) != DRADD_OK)
        return st;
    if (q->active && group_size != 0 && (!is_pow2(group_size) || group_size < 8 || group_size > 256 ||
                                         hq % group_size != 0))
        return DRADD_ERR_BAD_SHAPE;
    dradd_launch_cfg cfg = {};
    if (cfg_in)
        cfg = *cfg_in;
    if (cfg.variant == DRADD_VARIANT_WARP)
        return (q->active || k->active)
                   ? qk_plan_warp(n_q, hq, n_k, hk, add, sm_count, ctas_per_sm, smem_optin, cfg, out)
                   : DRADD_OK;
    if (cfg.variant == DRADD_VARIANT_CHUNK)
        return qk_plan_chunk(n_q, hq, n_k, hk, add, sm_count, ctas_per_sm, smem_optin, cfg, out);
    if (cfg.variant < DRADD_VARIANT_AUTO || cfg.variant > DRADD_VARIANT_STAGED || cfg.rows_per_cta != 0 ||
        cfg.stages < 0 || cfg.stages > 8 || cfg.fault_inject < 0 || cfg.wait_limit_us < 0 || cfg.grid_ctas < 0 ||
        (cfg.serialize != 0 && cfg.serialize != 1) ||
        (cfg.blocks_per_thread != 0 && (!is_pow2(cfg.blocks_per_thread) || cfg.blocks_per_thread > 8)) ||
        cfg.cluster_ctas != 0)
        return DRADD_ERR_BAD_CONFIG;
    out->serialize = cfg.serialize != 0;
    int64_t max_p = 0;
    for (const QkSide* side : {q, k})
        if (side->active && next_pow2(side->hidden) > max_p)
            max_p = next_pow2(side->hidden);
    // Automatic choice by the longer side's P (and, for short rows, the row
    // count), measured on GB300 (CUDA-graph replays over rotating buffers,
    // median of interleaved rounds):
    //   P <= 256, more than 16384 rows    staged, 128 threads, K >= 4 (4 threads a row), 3 stages
    //   P <= 256, 4097..16384 rows        register variant, 128 threads, K >= 1
    //   P <= 256, up to 4096 rows         register variant, 128 threads, K >= 2
    //   256 < P <= 2048, 8192 rows or more  register variant, 256 threads, K >= 1
    //   256 < P <= 2048, fewer rows       register variant, 128 threads, K >= 2
    //   P > 2048                          staged, max(128, P / 8) threads up to 512
    // with 2 stages per side unless stated (with the L2 prefetch of each
    // CTA's first rows before the dependency wait).
    int auto_variant = DRADD_VARIANT_STAGED, auto_k = 1, auto_stages = 2;
    int64_t auto_b = max_p / 8 < 128 ? 128 : (max_p / 8 > 512 ? 512 : max_p / 8);
    const int64_t rows = n_q + n_k;
    if (max_p <= 256 && rows > 16384) {
        auto_b = 128;
        auto_k = 4;
        auto_stages = 3;
    } else if (max_p <= 256) {
        auto_variant = DRADD_VARIANT_ROWS;
        auto_b = 128;
        auto_k = rows > 4096 ? 1 : 2;
    } else if (max_p <= 2048) {
        auto_variant = DRADD_VARIANT_ROWS;
        auto_b = rows >= 8192 ? 256 : 128;
        auto_k = rows >= 8192 ? 1 : 2;
    }
    // an explicit stage count or the fault hook asks for the staged variant
    if (cfg.variant == DRADD_VARIANT_AUTO && (cfg.stages != 0 || cfg.fault_inject != 0))
        auto_variant = DRADD_VARIANT_STAGED;
    const bool auto_plain = cfg.variant == DRADD_VARIANT_AUTO && cfg.stages == 0 && cfg.fault_inject == 0 &&
                            cfg.threads_per_row == 0 && cfg.blocks_per_thread == 0;
    // q rows with 512 < P <= 4096 (k rows 256 <= P <= 2048, or none): the
    // q rows in 512-element chunks, one warp each, one stage (4096 tokens
    // of 1536 + 512: 12.41 us against 12.73 one warp a row; 2048 tokens:
    // 6.99 against 7.63; 4096 x 3072 q + 1024 k: 23.1 against 33.2 staged;
    // 4096 x 1280 q alone: 9.10 against 11.75; 16384 tokens of 1536 + 512:
    // 43.98 against 43.78, a tie).
    if (auto_plain && q->active && next_pow2(hq) > 512 && next_pow2(hq) <= 4096 &&
        (!k->active || (next_pow2(hk) >= 256 && next_pow2(hk) <= 2048))) {
        dradd_launch_cfg c = cfg;
        c.variant = DRADD_VARIANT_CHUNK;
        c.stages = 1;
        return qk_plan_chunk(n_q, hq, n_k, hk, add, sm_count, ctas_per_sm, smem_optin, c, out);
    }
    // Both sides 256 < P <= 2048 with 8192 rows or more, where the rule
    // above did not apply (q rows of P = 512): one warp a row with a ring of
    // 2 row slots per warp, 128 threads a CTA (on the low-rank layout, 4096
    // tokens of 1536 + 512, before the chunked-q kernel took it: 13.41 us
    // against 14.21 for the register variant).
    if (auto_plain && rows >= 8192 && max_p <= 2048) {
        bool fits = true;
        for (const QkSide* side : {q, k})
            if (side->active && next_pow2(side->hidden) <= 256)
                fits = false;
        if (fits) {
            dradd_launch_cfg w = cfg;
            w.variant = DRADD_VARIANT_WARP;
            w.threads_per_row = 128;
            w.stages = 2;
            return qk_plan_warp(n_q, hq, n_k, hk, add, sm_count, ctas_per_sm, smem_optin, w, out);
        }
    }
    out->staged = (cfg.variant == DRADD_VARIANT_AUTO ? auto_variant : cfg.variant) != DRADD_VARIANT_ROWS;
    if (!out->staged && (cfg.stages != 0 || cfg.fault_inject != 0))
        return DRADD_ERR_BAD_CONFIG;
    if (!q->active && !k->active)
        return DRADD_OK;
    int64_t B = cfg.threads_per_row != 0 ? cfg.threads_per_row : auto_b;
    const int64_t k_pref = cfg.blocks_per_thread != 0 ? cfg.blocks_per_thread : auto_k;
    if (!is_pow2(B) || B < 32 || B > 1024)
        return DRADD_ERR_BAD_CONFIG;
    int max_k = 1;
    for (QkSide* side : {q, k}) {
        if (!side->active)
            continue;
        const int64_t blocks = next_pow2(side->hidden) / 8;
        int64_t K = 1;
        while (blocks / K > B)
            K *= 2;
        int64_t pref = k_pref < blocks ? k_pref : blocks;
        if (side == q && group_size != 0) {
            if (pref > blocks / (group_size / 8))
                pref = blocks / (group_size / 8);  // a group's lanes stay within one row's threads
            if (!out->staged && pref > group_size / 8)
                pref = group_size / 8;  // register variant: a thread's blocks stay within one group
        }
        if (pref > K)
            K = pref;
        if (!out->staged && side == q && group_size != 0 && K > group_size / 8) {
            // the register variant cannot place this split; the staged one can
            if (cfg.variant != DRADD_VARIANT_AUTO)
                return DRADD_ERR_BAD_CONFIG;
            dradd_launch_cfg forced = cfg;
            forced.variant = DRADD_VARIANT_STAGED;
            return qk_plan(n_q, hq, n_k, hk, group_size, add, sm_count, ctas_per_sm, smem_optin, &forced, out);
        }
        if (K > 8)
            return DRADD_ERR_BAD_CONFIG;
        side->K = static_cast<int>(K);
        side->T = static_cast<int>(blocks / K);
        side->R = static_cast<int>(B / side->T);
        if (side->K > max_k)
            max_k = side->K;
    }
    if (B > dradd::qk_max_threads(max_k))
        return DRADD_ERR_BAD_CONFIG;
    if (q->active && group_size != 0 && group_size / 8 > q->T)
        return DRADD_ERR_BAD_CONFIG;

    if (out->staged) {
        const int64_t avail =
            static_cast<int64_t>(smem_optin) -
            static_cast<int64_t>(dradd::qk_static_smem(q->active ? q->K : 1, k->active ? k->K : 1)) - 1024;
        for (QkSide* side : {q, k}) {
            if (!side->active)
                continue;
            const bool side_add = side == q && add;
            side->stage_bytes = (side_add ? 4 : 2) * side->hidden * side->R;
            int64_t S = cfg.stages;
            if (S == 0) {
                S = kQkStageBudget / side->stage_bytes;
                if (S > auto_stages)
                    S = auto_stages;
                if (S < 1)
                    S = 1;
            }
            if (S * (side->stage_bytes + 8) > avail)
                return DRADD_ERR_BAD_CONFIG;
            side->stages = static_cast<int>(S);
            const int64_t need = S * (side->stage_bytes + 8);
            if (need > out->dyn_smem)
                out->dyn_smem = need;
        }
    }

    const int64_t need_q = q->active ? (n_q + q->R - 1) / q->R : 0;
    const int64_t need_k = k->active ? (n_k + k->R - 1) / k->R : 0;
    int64_t C = cfg.grid_ctas;
    if (C == 0)
        C = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * (ctas_per_sm > 0 ? ctas_per_sm : 2048 / B);
    if (C < (q->active ? 1 : 0) + (k->active ? 1 : 0))
        return DRADD_ERR_BAD_CONFIG;
    if (need_q + need_k <= C) {
        q->ctas = need_q;
        k->ctas = need_k;
    } else {
        const double wq = q->active ? static_cast<double>(n_q) * static_cast<double>(hq) : 0.0;
        const double wk = k->active ? static_cast<double>(n_k) * static_cast<double>(hk) : 0.0;
        int64_t cq = q->active ? static_cast<int64_t>(static_cast<double>(C) * wq / (wq + wk) + 0.5) : 0;
        if (q->active && cq < 1)
            cq = 1;
        if (k->active && cq > C - 1)
            cq = C - 1;
        if (cq > need_q)
            cq = need_q;
        int64_t ck = C - cq;
        if (ck > need_k)
            ck = need_k;
        q->ctas = cq;
        k->ctas = ck;
    }
    if (q->ctas + k->ctas > 0x7FFFFFFF)
        return DRADD_ERR_BAD_CONFIG;
    out->threads = static_cast<int>(B);
    return DRADD_OK;
}

int qk_mode(const QkLaunch& plan)
{
    return plan.chunk ? dradd::kQkChunk : plan.warp ? dradd::kQkWarp : plan.staged ? dradd::kQkStaged
                                                                                  : dradd::kQkRows;
}

// qk_plan on the current device (limits L): the staged and warp-per-row
// variants with an automatic grid get as many CTAs as fit on the device
// at once, from the occupancy calculator for the kernel the plan picks.
dradd_status qk_plan_on_device(int64_t n_q, int64_t hq, int64_t n_k, int64_t hk, int64_t group_size, bool add,
                               const DeviceLimits& L, const dradd_launch_cfg* cfg, QkLaunch* plan)
{
    dradd_status st = qk_plan(n_q, hq, n_k, hk, group_size, add, L.sm_count, 0, L.smem_per_block_optin, cfg, plan);
    if (st != DRADD_OK || !(plan->staged || plan->warp || plan->chunk) || (cfg && cfg->grid_ctas != 0))
        return st;
    const bool quant = group_size != 0;
    const int kq = plan->q.active ? plan->q.K : 1, kk = plan->k.active ? plan->k.K : 1;
    int per_sm = 0;
    if (dradd::qk_occupancy(kq, kk, quant, add, qk_mode(*plan), plan->threads, static_cast<size_t>(plan->dyn_smem),
                            &per_sm) != cudaSuccess)
        return DRADD_ERR_CUDA;
    return qk_plan(n_q, hq, n_k, hk, group_size, add, L.sm_count, per_sm > 0 ? per_sm : 1, L.smem_per_block_optin,
                   cfg, plan);
}

dradd_status qk_run(void* q_out, float* q_scale, dradd_bf16* q_residual_out, dradd_bf16* k_out,
                    const dradd_bf16* q, const dradd_bf16* q_residual, const dradd_bf16* q_weight,
                    const dradd_bf16* k, const dradd_bf16* k_weight, float q_eps, float k_eps, int64_t n_q,
                    int64_t hq, int64_t n_k, int64_t hk, int64_t group_size, cudaStream_t stream,
                    const dradd_launch_cfg* cfg)
{
    const bool quant = group_size != 0;
    const bool add = q_residual != nullptr;
    DeviceLimits defaults;
    QkLaunch plan;
    // shapes and configuration first, with GB300's limits; redone below
    dradd_status st = qk_plan(n_q, hq, n_k, hk, group_size, add, defaults.sm_count, 0,
                              defaults.smem_per_block_optin, cfg, &plan);
    if (st != DRADD_OK || plan.threads == 0)
        return st;
    if (plan.q.active) {
        if (!q_out || !q || !q_weight || (quant && !q_scale) || (add && !q_residual_out))
            return DRADD_ERR_NULL_PTR;
        if (!aligned(q_out, 16) || !aligned(q, 16) || !aligned(q_weight, 16) || (quant && !aligned(q_scale, 4)) ||
            (add && (!aligned(q_residual, 16) || !aligned(q_residual_out, 16))))
            return DRADD_ERR_MISALIGNED;
        if (!std::isfinite(q_eps) || q_eps < 0.0f)
            return DRADD_ERR_BAD_EPS;
    }
    if (plan.k.active) {
        if (!k_out || !k || !k_weight)
            return DRADD_ERR_NULL_PTR;
        if (!aligned(k_out, 16) || !aligned(k, 16) || !aligned(k_weight, 16))
            return DRADD_ERR_MISALIGNED;
        if (!std::isfinite(k_eps) || k_eps < 0.0f)
            return DRADD_ERR_BAD_EPS;
    }
    // Overlaps: outputs never overlap one another; an output may coincide
    // exactly with the input it replaces (q_out with q when bf16,
    // q_residual_out with q_residual, k_out with k) and overlap nothing else.
    const bool qa = plan.q.active, ka = plan.k.active;
    const int64_t eq = qa ? n_q * hq : 0, ek = ka ? n_k * hk : 0;
    const Range in[5] = {qa ? range_of(q, eq * 2) : Range{}, qa ? range_of(q_weight, hq * 2) : Range{},
                         qa && add ? range_of(q_residual, eq * 2) : Range{}, ka ? range_of(k, ek * 2) : Range{},
                         ka ? range_of(k_weight, hk * 2) : Range{}};
    const Range out[4] = {qa ? range_of(q_out, quant ? eq : eq * 2) : Range{},
                          qa && quant ? range_of(q_scale, n_q * (hq / group_size) * 4) : Range{},
                          qa && add ? range_of(q_residual_out, eq * 2) : Range{},
                          ka ? range_of(k_out, ek * 2) : Range{}};
    const int may_equal[4] = {quant ? -1 : 0, -1, 2, 3};  // input index each output may equal
    for (int a = 0; a < 4; ++a) {
        for (int b = a + 1; b < 4; ++b)
            if (out[a].overlaps(out[b]))
                return DRADD_ERR_ALIAS;
        for (int b = 0; b < 5; ++b)
            if (out[a].overlaps(in[b]) && !(b == may_equal[a] && out[a].same(in[b])))
                return DRADD_ERR_ALIAS;
    }
    DeviceLimits L;
    st = query_limits(&L);
    if (st != DRADD_OK)
        return st;
    dradd_launch_cfg eff = {};
    if (cfg)
        eff = *cfg;
    const bool device_memory =
        all_device_memory({q_out, q_scale, q_residual_out, k_out, q, q_residual, q_weight, k, k_weight});
    if (!device_memory) {
        if (eff.variant == DRADD_VARIANT_STAGED || eff.stages != 0 || eff.fault_inject != 0)
            return DRADD_ERR_BAD_CONFIG;
        if (eff.variant == DRADD_VARIANT_WARP || eff.variant == DRADD_VARIANT_CHUNK)
            return DRADD_ERR_BAD_CONFIG;  // bulk copies read device memory only
        eff.variant = DRADD_VARIANT_ROWS;
    }
    cfg = &eff;
    st = qk_plan_on_device(n_q, hq, n_k, hk, group_size, add, L, cfg, &plan);
    if (st != DRADD_OK)
        return st;
    const int kq = qa ? plan.q.K : 1, kk = ka ? plan.k.K : 1;
    const int mode = qk_mode(plan);

    unsigned* status = nullptr;
    if (dradd::device_status_ptr(&status) != cudaSuccess)
        return DRADD_ERR_CUDA;
    const uint64_t wait_ns = cfg && cfg->wait_limit_us > 0 ? static_cast<uint64_t>(cfg->wait_limit_us) * 1000ull
                                                          : kDefaultWaitLimitNs;
    auto params = [&](const QkSide& side, const dradd_bf16* x, const dradd_bf16* res, const dradd_bf16* w,
                      float eps) {
        Params p = {};
        p.x = x;
        p.residual = res;
        p.weight = w;
        p.eps = eps;
        p.hidden = static_cast<int>(side.hidden);
        p.inv_hidden = is_pow2(side.hidden) ? 1.0f / static_cast<float>(side.hidden) : 0.0f;
        p.n_rows = side.n_rows;
        p.threads_per_row = side.T;
        p.rows_per_cta = side.R;
        p.stages = side.stages;
        p.fault_inject = cfg ? cfg->fault_inject : 0;
        p.wait_limit_ns = wait_ns;
        p.status = status;
        p.l2_prefetch = device_memory ? 1 : 0;
        return p;
    };
    Params pq = params(plan.q, q, q_residual, q_weight, q_eps);
    if (quant) {
        pq.out_q = static_cast<int8_t*>(q_out);
        pq.scale = q_scale;
        pq.group_blocks = static_cast<int>(group_size / 8);
        while ((1 << pq.group_shift) < pq.group_blocks)
            ++pq.group_shift;
    } else {
        pq.out = static_cast<uint16_t*>(q_out);
    }
    pq.residual_out = q_residual_out;
    Params pk = params(plan.k, k, nullptr, k_weight, k_eps);
    pk.out = k_out;
    const cudaError_t e =
        dradd::launch_qk(pq, pk, kq, kk, quant, add, mode, static_cast<int>(plan.q.ctas),
                         static_cast<int>(plan.k.ctas), plan.threads, static_cast<size_t>(plan.dyn_smem),
                         plan.serialize, stream);
    return e == cudaSuccess ? DRADD_OK : DRADD_ERR_CUDA;
}

// ------------------------------------------- log-sum-exp merge, unary math
// Threads per CTA (cfg->threads_per_row, default 128), elements per thread
// per pass (cfg->blocks_per_thread, default 8) and CTAs (cfg->grid_ctas,
// default: threads_per_sm threads on every SM in whole CTAs, at most one
// CTA per unit).  The defaults are the fastest of sweeps on GB300 (CTA
// sizes 128-1024, 4-8 elements per thread, 1-32 CTAs per SM): the merge of
// 256 x 32768 (and of the last 16384 columns in place) with 1024 threads
// per SM, a few units per CTA (15.99 -> 15.39 and 9.45 -> 8.25 us against
// two full waves, 4096 threads per SM); log1p of 2^24 values with two full
// waves (21.2 us; 1024 threads per SM: 25.6 us).
constexpr int kMergeThreadsPerSm = 1024;
constexpr int kUnaryThreadsPerSm = 4096;

dradd_status elementwise_plan(int64_t n_rows, int64_t n_cols, const dradd_launch_cfg* cfg_in, int sm_count,
                              int threads_per_sm, int* threads, int* vec, int* grid, bool* serialize)
{
    dradd_launch_cfg cfg = {};
    if (cfg_in)
        cfg = *cfg_in;
    if (cfg.variant != DRADD_VARIANT_AUTO || cfg.rows_per_cta != 0 || cfg.stages != 0 || cfg.fault_inject != 0 ||
        cfg.wait_limit_us != 0 || cfg.grid_ctas < 0 || (cfg.serialize != 0 && cfg.serialize != 1) ||
        cfg.cluster_ctas != 0)
        return DRADD_ERR_BAD_CONFIG;
    const int T = cfg.threads_per_row ? cfg.threads_per_row : 128;
    const int V = cfg.blocks_per_thread ? cfg.blocks_per_thread : 8;
    if (!is_pow2(T) || T < 32 || T > 1024 || (V != 1 && V != 2 && V != 4 && V != 8))
        return DRADD_ERR_BAD_CONFIG;
    const int64_t span = static_cast<int64_t>(T) * V;
    const int64_t units = n_rows * ((n_cols + span - 1) / span);
    int64_t G = cfg.grid_ctas;
    if (G == 0) {
        const int per_sm = threads_per_sm > T ? threads_per_sm / T : 1;
        G = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * per_sm;
        if (G > units)
            G = units;
        if (G < 1)
            G = 1;
    }
    if (G > 0x7FFFFFFF)
        return DRADD_ERR_BAD_CONFIG;
    *threads = T;
    *vec = V;
    *grid = static_cast<int>(G);
    *serialize = cfg.serialize != 0;
    return DRADD_OK;
}

// Byte range of a row-strided fp32 tensor.
Range strided_range(const float* p, int64_t stride, int64_t n_rows, int64_t n_cols)
{
    return range_of(p, ((n_rows - 1) * stride + n_cols) * 4);
}

dradd_status lse_run(float* out, int64_t out_stride, const float* a, int64_t a_stride, const float* b,
                     int64_t b_stride, int64_t n_rows, int64_t n_cols, cudaStream_t stream,
                     const dradd_launch_cfg* cfg)
{
    if (n_rows < 0 || n_cols < 0)
        return DRADD_ERR_BAD_SHAPE;
    if (n_rows > 0 && n_cols > 0 && (out_stride < n_cols || a_stride < n_cols || b_stride < n_cols))
        return DRADD_ERR_BAD_SHAPE;
    for (int64_t stride : {out_stride, a_stride, b_stride})
        if (n_rows > 0 && n_cols > 0 && n_rows - 1 > (INT64_MAX / 8 - n_cols) / (stride > 0 ? stride : 1))
            return DRADD_ERR_BAD_SHAPE;
    int threads = 0, vec = 0, grid = 0;
    bool serialize = false;
    dradd_status st = elementwise_plan(n_rows, n_cols, cfg, 152, kMergeThreadsPerSm, &threads, &vec, &grid,
                                       &serialize);
    if (st != DRADD_OK)
        return st;
    if (n_rows == 0 || n_cols == 0)
        return DRADD_OK;
    if (!out || !a || !b)
        return DRADD_ERR_NULL_PTR;
    if (!aligned(out, 4) || !aligned(a, 4) || !aligned(b, 4))
        return DRADD_ERR_MISALIGNED;
    // out may be exactly a or b (same address and stride: each element is
    // read by the thread that then writes it); no other overlap
    const Range ro = strided_range(out, out_stride, n_rows, n_cols);
    const Range ra = strided_range(a, a_stride, n_rows, n_cols);
    const Range rb = strided_range(b, b_stride, n_rows, n_cols);
    if (ro.overlaps(ra) && !(out == a && out_stride == a_stride))
        return DRADD_ERR_ALIAS;
    if (ro.overlaps(rb) && !(out == b && out_stride == b_stride))
        return DRADD_ERR_ALIAS;
    DeviceLimits L;
    st = query_limits(&L);
    if (st != DRADD_OK)
        return st;
    st = elementwise_plan(n_rows, n_cols, cfg, L.sm_count, kMergeThreadsPerSm, &threads, &vec, &grid,
                          &serialize);
    if (st != DRADD_OK)
        return st;
    const bool vec4 = aligned(out, 16) && aligned(a, 16) && aligned(b, 16) &&
                      (n_rows == 1 || (out_stride % 4 == 0 && a_stride % 4 == 0 && b_stride % 4 == 0));
    const bool dev = all_device_memory({out, a, b});
    return dradd::launch_lse_merge(out, out_stride, a, a_stride, b, b_stride, n_rows, n_cols, vec, vec4, dev,
                                   grid, threads, serialize, stream) == cudaSuccess
               ? DRADD_OK
               : DRADD_ERR_CUDA;
}

dradd_status unary_run(float* out, const float* x, int64_t n, int op, cudaStream_t stream,
                       const dradd_launch_cfg* cfg)
{
    if (n < 0)
        return DRADD_ERR_BAD_SHAPE;
    if (n > INT64_MAX / 8)
        return DRADD_ERR_BAD_SHAPE;
    if (op < DRADD_UNARY_LOG1P || op > DRADD_UNARY_EXP)
        return DRADD_ERR_BAD_CONFIG;
    int threads = 0, vec = 0, grid = 0;
    bool serialize = false;
    dradd_status st = elementwise_plan(1, n, cfg, 152, kUnaryThreadsPerSm, &threads, &vec, &grid, &serialize);
    if (st != DRADD_OK)
        return st;
    if (n == 0)
        return DRADD_OK;
    if (!out || !x)
        return DRADD_ERR_NULL_PTR;
    if (!aligned(out, 4) || !aligned(x, 4))
        return DRADD_ERR_MISALIGNED;
    if (range_of(out, n * 4).overlaps(range_of(x, n * 4)) && out != x)
        return DRADD_ERR_ALIAS;
    DeviceLimits L;
    st = query_limits(&L);
    if (st != DRADD_OK)
        return st;
    st = elementwise_plan(1, n, cfg, L.sm_count, kUnaryThreadsPerSm, &threads, &vec, &grid, &serialize);
    if (st != DRADD_OK)
        return st;
    const bool vec4 = aligned(out, 16) && aligned(x, 16);
    const bool dev = all_device_memory({out, x});
    return dradd::launch_unary(out, x, n, op, vec, vec4, dev, grid, threads, serialize, stream) == cudaSuccess
               ? DRADD_OK
               : DRADD_ERR_CUDA;
}

}  // namespace

extern "C" {

dradd_status add_rmsnorm_fwd(dradd_bf16* out, dradd_bf16* residual_out, const dradd_bf16* x,
                             const dradd_bf16* residual, const dradd_bf16* weight, float eps,
                             int64_t n_rows, int64_t hidden, cudaStream_t stream)
{
    return run(dradd::kOutBf16, true, out, nullptr, nullptr, residual_out, x, residual, weight, eps, n_rows, hidden,
               stream, nullptr);
}

dradd_status add_rmsnorm_quant_fwd(int8_t* out_q, float* scale, dradd_bf16* residual_out,
                                   const dradd_bf16* x, const dradd_bf16* residual,
                                   const dradd_bf16* weight, float eps, int64_t n_rows,
                                   int64_t hidden, cudaStream_t stream)
{
    return run(dradd::kOutInt8, true, nullptr, out_q, scale, residual_out, x, residual, weight, eps, n_rows, hidden,
               stream, nullptr);
}

dradd_status add_rmsnorm_fwd_with_config(dradd_bf16* out, dradd_bf16* residual_out,
                                         const dradd_bf16* x, const dradd_bf16* residual,
                                         const dradd_bf16* weight, float eps, int64_t n_rows,
                                         int64_t hidden, cudaStream_t stream,
                                         const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return run(dradd::kOutBf16, true, out, nullptr, nullptr, residual_out, x, residual, weight, eps, n_rows, hidden,
               stream, cfg);
}

dradd_status add_rmsnorm_quant_fwd_with_config(int8_t* out_q, float* scale, dradd_bf16* residual_out,
                                               const dradd_bf16* x, const dradd_bf16* residual,
                                               const dradd_bf16* weight, float eps, int64_t n_rows,
                                               int64_t hidden, cudaStream_t stream,
                                               const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return run(dradd::kOutInt8, true, nullptr, out_q, scale, residual_out, x, residual, weight, eps, n_rows, hidden,
               stream, cfg);
}

dradd_status dradd_resolve_config(int64_t n_rows, int64_t hidden, int op, int sm_count,
                                  dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    if (op < DRADD_OP_ADD_RMSNORM || op > DRADD_OP_RMSNORM_FP4)
        return DRADD_ERR_BAD_CONFIG;
    DeviceLimits L;
    if (sm_count > 0) {
        L.sm_count = sm_count;
    } else {
        const dradd_status st = query_limits(&L);
        if (st != DRADD_OK)
            return st;
    }
    const bool quant = op != DRADD_OP_ADD_RMSNORM && op != DRADD_OP_RMSNORM;
    const bool add = op == DRADD_OP_ADD_RMSNORM || op == DRADD_OP_ADD_RMSNORM_QUANT ||
                     op == DRADD_OP_ADD_RMSNORM_FP8 || op == DRADD_OP_ADD_RMSNORM_FP4;
    return resolve(n_rows, hidden, quant, add, L, cfg);
}

dradd_status add_rmsnorm_fp8_fwd(uint8_t* out_q, float* scale, dradd_bf16* residual_out,
                                 const dradd_bf16* x, const dradd_bf16* residual, const dradd_bf16* weight,
                                 float eps, int64_t n_rows, int64_t hidden, cudaStream_t stream)
{
    return run(dradd::kOutE4m3, true, nullptr, reinterpret_cast<int8_t*>(out_q), scale, residual_out, x,
               residual, weight, eps, n_rows, hidden, stream, nullptr);
}

dradd_status add_rmsnorm_fp8_fwd_with_config(uint8_t* out_q, float* scale, dradd_bf16* residual_out,
                                             const dradd_bf16* x, const dradd_bf16* residual,
                                             const dradd_bf16* weight, float eps, int64_t n_rows,
                                             int64_t hidden, cudaStream_t stream,
                                             const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return run(dradd::kOutE4m3, true, nullptr, reinterpret_cast<int8_t*>(out_q), scale, residual_out, x,
               residual, weight, eps, n_rows, hidden, stream, cfg);
}

dradd_status add_rmsnorm_fp4_fwd(uint8_t* out_q, float* scale, dradd_bf16* residual_out,
                                 const dradd_bf16* x, const dradd_bf16* residual, const dradd_bf16* weight,
                                 float eps, int64_t n_rows, int64_t hidden, cudaStream_t stream)
{
    return run(dradd::kOutE2m1, true, nullptr, reinterpret_cast<int8_t*>(out_q), scale, residual_out, x,
               residual, weight, eps, n_rows, hidden, stream, nullptr);
}

dradd_status add_rmsnorm_fp4_fwd_with_config(uint8_t* out_q, float* scale, dradd_bf16* residual_out,
                                             const dradd_bf16* x, const dradd_bf16* residual,
                                             const dradd_bf16* weight, float eps, int64_t n_rows,
                                             int64_t hidden, cudaStream_t stream,
                                             const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return run(dradd::kOutE2m1, true, nullptr, reinterpret_cast<int8_t*>(out_q), scale, residual_out, x,
               residual, weight, eps, n_rows, hidden, stream, cfg);
}

dradd_status rmsnorm_fp4_fwd(uint8_t* out_q, float* scale, const dradd_bf16* x, const dradd_bf16* weight,
                             float eps, int64_t n_rows, int64_t hidden, cudaStream_t stream)
{
    return run(dradd::kOutE2m1, false, nullptr, reinterpret_cast<int8_t*>(out_q), scale, nullptr, x, nullptr,
               weight, eps, n_rows, hidden, stream, nullptr);
}

dradd_status rmsnorm_fp4_fwd_with_config(uint8_t* out_q, float* scale, const dradd_bf16* x,
                                         const dradd_bf16* weight, float eps, int64_t n_rows, int64_t hidden,
                                         cudaStream_t stream, const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return run(dradd::kOutE2m1, false, nullptr, reinterpret_cast<int8_t*>(out_q), scale, nullptr, x, nullptr,
               weight, eps, n_rows, hidden, stream, cfg);
}

dradd_status rmsnorm_fp8_fwd(uint8_t* out_q, float* scale, const dradd_bf16* x, const dradd_bf16* weight,
                             float eps, int64_t n_rows, int64_t hidden, cudaStream_t stream)
{
    return run(dradd::kOutE4m3, false, nullptr, reinterpret_cast<int8_t*>(out_q), scale, nullptr, x, nullptr,
               weight, eps, n_rows, hidden, stream, nullptr);
}

dradd_status rmsnorm_fp8_fwd_with_config(uint8_t* out_q, float* scale, const dradd_bf16* x,
                                         const dradd_bf16* weight, float eps, int64_t n_rows, int64_t hidden,
                                         cudaStream_t stream, const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return run(dradd::kOutE4m3, false, nullptr, reinterpret_cast<int8_t*>(out_q), scale, nullptr, x, nullptr,
               weight, eps, n_rows, hidden, stream, cfg);
}

dradd_status rmsnorm_fwd(dradd_bf16* out, const dradd_bf16* x, const dradd_bf16* weight, float eps,
                         int64_t n_rows, int64_t hidden, cudaStream_t stream)
{
    return run(dradd::kOutBf16, false, out, nullptr, nullptr, nullptr, x, nullptr, weight, eps, n_rows, hidden, stream,
               nullptr);
}

dradd_status rmsnorm_quant_fwd(int8_t* out_q, float* scale, const dradd_bf16* x, const dradd_bf16* weight,
                               float eps, int64_t n_rows, int64_t hidden, cudaStream_t stream)
{
    return run(dradd::kOutInt8, false, nullptr, out_q, scale, nullptr, x, nullptr, weight, eps, n_rows, hidden, stream,
               nullptr);
}

dradd_status rmsnorm_fwd_with_config(dradd_bf16* out, const dradd_bf16* x, const dradd_bf16* weight,
                                     float eps, int64_t n_rows, int64_t hidden, cudaStream_t stream,
                                     const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return run(dradd::kOutBf16, false, out, nullptr, nullptr, nullptr, x, nullptr, weight, eps, n_rows, hidden, stream,
               cfg);
}

dradd_status rmsnorm_quant_fwd_with_config(int8_t* out_q, float* scale, const dradd_bf16* x,
                                           const dradd_bf16* weight, float eps, int64_t n_rows,
                                           int64_t hidden, cudaStream_t stream, const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return run(dradd::kOutInt8, false, nullptr, out_q, scale, nullptr, x, nullptr, weight, eps, n_rows, hidden, stream,
               cfg);
}

dradd_status residual_add_fwd(dradd_bf16* residual_out, const dradd_bf16* x, const dradd_bf16* residual,
                              int64_t n_rows, int64_t hidden, cudaStream_t stream)
{
    if (n_rows < 0 || hidden <= 0)
        return DRADD_ERR_BAD_SHAPE;
    if (hidden % 8 != 0 || hidden > DRADD_MAX_HIDDEN)
        return DRADD_ERR_UNSUPPORTED_HIDDEN;
    if (n_rows > (INT64_MAX / 4) / hidden)
        return DRADD_ERR_BAD_SHAPE;
    if (n_rows == 0)
        return DRADD_OK;
    if (!residual_out || !x || !residual)
        return DRADD_ERR_NULL_PTR;
    if (!aligned(residual_out, 16) || !aligned(x, 16) || !aligned(residual, 16))
        return DRADD_ERR_MISALIGNED;
    const int64_t elems = n_rows * hidden;
    // inputs in the order check_overlaps expects: x, (weight slot, empty), residual
    const Range inputs[3] = {range_of(x, elems * 2), Range{}, range_of(residual, elems * 2)};
    const Range outs[1] = {range_of(residual_out, elems * 2)};
    const bool bf16_out[1] = {true};
    dradd_status st = check_overlaps(inputs, 3, outs, bf16_out, 1);
    if (st != DRADD_OK)
        return st;
    DeviceLimits L;
    st = query_limits(&L);
    if (st != DRADD_OK)
        return st;
    const bool dev = all_device_memory({residual_out, x, residual});
    return dradd::launch_residual_add(residual_out, x, residual, elems / 8, L.sm_count, dev, false, stream) ==
                   cudaSuccess
               ? DRADD_OK
               : DRADD_ERR_CUDA;
}

dradd_status fused_qk_rmsnorm_group_quant_fwd(void* q_out, float* q_scale, dradd_bf16* q_residual_out,
                                              dradd_bf16* k_out, const dradd_bf16* q,
                                              const dradd_bf16* q_residual, const dradd_bf16* q_weight,
                                              const dradd_bf16* k, const dradd_bf16* k_weight, float q_eps,
                                              float k_eps, int64_t n_q_rows, int64_t q_hidden, int64_t n_k_rows,
                                              int64_t k_hidden, int64_t group_size, cudaStream_t stream)
{
    return qk_run(q_out, q_scale, q_residual_out, k_out, q, q_residual, q_weight, k, k_weight, q_eps, k_eps,
                  n_q_rows, q_hidden, n_k_rows, k_hidden, group_size, stream, nullptr);
}

dradd_status fused_qk_rmsnorm_group_quant_fwd_with_config(
    void* q_out, float* q_scale, dradd_bf16* q_residual_out, dradd_bf16* k_out, const dradd_bf16* q,
    const dradd_bf16* q_residual, const dradd_bf16* q_weight, const dradd_bf16* k, const dradd_bf16* k_weight,
    float q_eps, float k_eps, int64_t n_q_rows, int64_t q_hidden, int64_t n_k_rows, int64_t k_hidden,
    int64_t group_size, cudaStream_t stream, const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return qk_run(q_out, q_scale, q_residual_out, k_out, q, q_residual, q_weight, k, k_weight, q_eps, k_eps,
                  n_q_rows, q_hidden, n_k_rows, k_hidden, group_size, stream, cfg);
}

dradd_status dradd_qk_resolve_config(int64_t n_q_rows, int64_t q_hidden, int64_t n_k_rows, int64_t k_hidden,
                                     int64_t group_size, int q_residual, int sm_count, const dradd_launch_cfg* cfg,
                                     dradd_qk_plan* plan)
{
    if (!plan)
        return DRADD_ERR_NULL_PTR;
    DeviceLimits L;
    if (sm_count > 0) {
        L.sm_count = sm_count;
    } else {
        const dradd_status st = query_limits(&L);
        if (st != DRADD_OK)
            return st;
    }
    QkLaunch r;
    const dradd_status st =
        sm_count > 0 ? qk_plan(n_q_rows, q_hidden, n_k_rows, k_hidden, group_size, q_residual != 0, L.sm_count, 0,
                               L.smem_per_block_optin, cfg, &r)
                     : qk_plan_on_device(n_q_rows, q_hidden, n_k_rows, k_hidden, group_size, q_residual != 0, L,
                                         cfg, &r);
    if (st != DRADD_OK)
        return st;
    plan->variant = r.threads == 0 ? 0
                    : (r.chunk  ? DRADD_VARIANT_CHUNK
                       : r.warp ? DRADD_VARIANT_WARP
                       : r.staged ? DRADD_VARIANT_STAGED
                                  : DRADD_VARIANT_ROWS);
    plan->threads_per_cta = r.threads;
    plan->dyn_smem_bytes = static_cast<int>(r.dyn_smem);
    plan->q_threads_per_row = r.q.T;
    plan->q_rows_per_cta = r.q.R;
    plan->q_stages = r.q.stages;
    plan->q_ctas = static_cast<int>(r.q.ctas);
    plan->k_threads_per_row = r.k.T;
    plan->k_rows_per_cta = r.k.R;
    plan->k_stages = r.k.stages;
    plan->k_ctas = static_cast<int>(r.k.ctas);
    return DRADD_OK;
}

dradd_status lse_merge_fwd(float* out, const float* lse_a, const float* lse_b, int64_t n, cudaStream_t stream)
{
    return lse_run(out, n, lse_a, n, lse_b, n, n > 0 ? 1 : 0, n, stream, nullptr);
}

dradd_status lse_merge_2d_fwd(float* out, int64_t out_stride, const float* lse_a, int64_t a_stride,
                              const float* lse_b, int64_t b_stride, int64_t n_rows, int64_t n_cols,
                              cudaStream_t stream)
{
    return lse_run(out, out_stride, lse_a, a_stride, lse_b, b_stride, n_rows, n_cols, stream, nullptr);
}

dradd_status lse_merge_2d_fwd_with_config(float* out, int64_t out_stride, const float* lse_a, int64_t a_stride,
                                          const float* lse_b, int64_t b_stride, int64_t n_rows, int64_t n_cols,
                                          cudaStream_t stream, const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return lse_run(out, out_stride, lse_a, a_stride, lse_b, b_stride, n_rows, n_cols, stream, cfg);
}

dradd_status invariant_unary_fwd(float* out, const float* x, int64_t n, int op, cudaStream_t stream)
{
    return unary_run(out, x, n, op, stream, nullptr);
}

dradd_status invariant_unary_fwd_with_config(float* out, const float* x, int64_t n, int op, cudaStream_t stream,
                                             const dradd_launch_cfg* cfg)
{
    if (!cfg)
        return DRADD_ERR_NULL_PTR;
    return unary_run(out, x, n, op, stream, cfg);
}

dradd_status dradd_device_status(cudaStream_t stream, int clear)
{
    unsigned word = 0;
    if (dradd::read_device_status(&word, clear != 0, stream) != cudaSuccess)
        return DRADD_ERR_CUDA;
    if (word & dradd::kDeviceStatusUndrained)
        return DRADD_ERR_UNDRAINED;
    return word ? DRADD_ERR_TIMEOUT : DRADD_OK;
}

dradd_status dradd_last_device_status(cudaStream_t stream)
{
    return dradd_device_status(stream, 1);
}

dradd_status dradd_bf16_convert_range(dradd_bf16* out, uint64_t first, int64_t count, int method,
                                      cudaStream_t stream)
{
    if (count < 0)
        return DRADD_ERR_BAD_SHAPE;
    if (count == 0)
        return DRADD_OK;
    if (!out)
        return DRADD_ERR_NULL_PTR;
    if (!aligned(out, 2))
        return DRADD_ERR_MISALIGNED;
    if (method < 0 || method > 5)
        return DRADD_ERR_BAD_CONFIG;
    return dradd::launch_convert(out, first, count, method, stream) == cudaSuccess ? DRADD_OK
                                                                                  : DRADD_ERR_CUDA;
}

const char* dradd_status_string(dradd_status status)
{
    switch (status) {
    case DRADD_OK: return "DRADD_OK";
    case DRADD_ERR_NULL_PTR: return "DRADD_ERR_NULL_PTR: a required pointer is NULL";
    case DRADD_ERR_BAD_SHAPE: return "DRADD_ERR_BAD_SHAPE: n_rows < 0 or hidden <= 0 (or too large)";
    case DRADD_ERR_UNSUPPORTED_HIDDEN:
        return "DRADD_ERR_UNSUPPORTED_HIDDEN: hidden must be a multiple of 8 and <= 32768";
    case DRADD_ERR_MISALIGNED: return "DRADD_ERR_MISALIGNED: pointers must be 16-byte aligned";
    case DRADD_ERR_BAD_EPS: return "DRADD_ERR_BAD_EPS: eps must be finite and >= 0";
    case DRADD_ERR_ALIAS: return "DRADD_ERR_ALIAS: buffers overlap other than as allowed";
    case DRADD_ERR_CUDA: return "DRADD_ERR_CUDA: a CUDA runtime call failed";
    case DRADD_ERR_TIMEOUT: return "DRADD_ERR_TIMEOUT: a kernel's bounded wait expired";
    case DRADD_ERR_BAD_CONFIG: return "DRADD_ERR_BAD_CONFIG: invalid launch configuration";
    case DRADD_ERR_UNDRAINED:
        return "DRADD_ERR_UNDRAINED: a bounded wait expired and an issued copy had not landed";
    default: return "DRADD_ERR_UNKNOWN";
    }
}

int dradd_abi_version(void) { return DRADD_ABI_VERSION; }

}  // extern "C"
