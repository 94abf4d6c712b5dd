/*
 * dradd.h -- C ABI of libdradd: deterministic fused residual-add + RMSNorm
 * forward for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one named rmsnorm2d_fwd_with_add on the ROCm/aiter
 * issue #5151 page ("rmsnorm2d_fwd_with_add truncates fp32->bf16 on gfx942,
 * biasing residual_out and compounding across layers"), section "Steps to
 * Reproduce", function reference():
 *
 *     acc          = fp32(x) + fp32(residual)                  (per element)
 *     residual_out = bf16(acc)
 *     out          = bf16((acc * rsqrt(mean(acc^2) + eps)) * fp32(weight))
 *
 * with both bf16 stores rounded to nearest, ties to even (the page's fix,
 * sections "Problem Description" and "Notes"), never truncated.
 *
 * Every result is a fixed function of the inputs; it does not depend on the
 * launch configuration, the variant chosen, the GPU's SM count or the run:
 *   - acc, acc^2, the mean, the sum of eps, the square root, the reciprocal
 *     and both products are single IEEE fp32 operations rounded to nearest
 *     (no fused multiply-add, no flush to zero);
 *   - mean(acc^2) = S / hidden, where S is the pairwise sum of the squares:
 *     the row is padded with +0 to P = the next power of two >= hidden, and
 *     the sum of a block is the rounded sum of its lower and upper halves;
 *   - rsqrt(v) = 1 / sqrt(v), both correctly rounded;
 *   - the products run left to right: (acc * inv) * weight.
 *
 * Conventions shared by every entry point:
 *   - bf16 values are passed as their 16-bit patterns (dradd_bf16).
 *   - x, residual, out, residual_out: row-major, n_rows x hidden, contiguous
 *     (row stride = hidden elements).  weight: hidden elements, shared by
 *     all rows.
 *   - All pointers are addressable by the current device: device memory
 *     (cudaMalloc'd), or host memory the device can reach (pinned or
 *     registered host memory, memory behind the Grace-Blackwell host link,
 *     managed memory).  With any non-device buffer the kernels read and
 *     write it directly over the host link (zero copy) and the register-load
 *     variant is used; an explicit DRADD_VARIANT_STAGED configuration (or a
 *     stage count or fault hook for the fused q/k call) with such a buffer
 *     is rejected with DRADD_ERR_BAD_CONFIG.  The caller allocates and owns
 *     every buffer; the library allocates no device memory and keeps no
 *     per-call state.
 *   - Every array pointer must be 16-byte aligned (scale: 4-byte aligned).
 *   - 1 <= hidden <= DRADD_MAX_HIDDEN and hidden % 8 == 0.  n_rows >= 0;
 *     n_rows == 0 is a successful no-op (pointers are not inspected).
 *   - eps must be finite and >= 0; it is used as the given fp32 value.
 *   - Aliasing: an output may be exactly the same buffer as x or as residual
 *     (e.g. residual_out == residual for an in-place residual update).  Any
 *     other overlap between buffers is rejected with DRADD_ERR_ALIAS.
 *   - The call enqueues work on `stream` (0 = the legacy default stream of
 *     the current device) and returns without synchronising.  Results are
 *     valid once the stream has reached that point.  Launch failures are
 *     returned as DRADD_ERR_CUDA at enqueue time.
 *   - Argument errors are detected on the host before any GPU work and leave
 *     every buffer untouched.
 *   - Calls that run at the same time on different streams share nothing
 *     except the device status word read by dradd_device_status().
 */
#ifndef DRADD_H
#define DRADD_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DRADD_ABI_VERSION 1
#define DRADD_MAX_HIDDEN 32768
#define DRADD_QK_MAX_HIDDEN 16384  /* q_hidden, k_hidden of the fused q/k call */

typedef uint16_t dradd_bf16;  /* raw bf16 bit pattern */
typedef int dradd_status;

enum {
    DRADD_OK = 0,
    DRADD_ERR_NULL_PTR = 1,           /* a required pointer is NULL                  */
    DRADD_ERR_BAD_SHAPE = 2,          /* n_rows < 0 or hidden <= 0                    */
    DRADD_ERR_UNSUPPORTED_HIDDEN = 3, /* hidden % 8 != 0 or hidden > DRADD_MAX_HIDDEN */
    DRADD_ERR_MISALIGNED = 4,         /* a pointer is not 16-byte (scale: 4) aligned  */
    DRADD_ERR_BAD_EPS = 5,            /* eps is NaN, infinite or negative             */
    DRADD_ERR_ALIAS = 6,              /* buffers overlap other than as allowed         */
    DRADD_ERR_CUDA = 7,               /* a CUDA runtime call failed                    */
    DRADD_ERR_TIMEOUT = 8,            /* a kernel's bounded wait expired (device)      */
    DRADD_ERR_BAD_CONFIG = 9,         /* an explicit launch configuration is invalid   */
    DRADD_ERR_UNDRAINED = 10          /* after a timeout, an issued bulk copy had not
                                         landed when the kernel stopped waiting (device) */
};

/*
 * add_rmsnorm_fwd -- residual-add + RMSNorm forward with bf16 out.
 * Page: ROCm/aiter issue #5151, "Steps to Reproduce", reference(); the
 * argument set mirrors the page's call rmsnorm2d_fwd_with_add(out, x,
 * residual, residual_out, weight, eps).
 *
 *   out           [n_rows x hidden] bf16, written: bf16_rne((acc*inv)*weight)
 *   residual_out  [n_rows x hidden] bf16, written: bf16_rne(acc)
 *   x, residual   [n_rows x hidden] bf16, read
 *   weight        [hidden] bf16, read
 *   eps           added to mean(acc^2) before the square root
 *   stream        CUDA stream to enqueue on
 * Returns DRADD_OK or one of the errors above.
 */
dradd_status add_rmsnorm_fwd(dradd_bf16* out, dradd_bf16* residual_out,
                             const dradd_bf16* x, const dradd_bf16* residual,
                             const dradd_bf16* weight, float eps,
                             int64_t n_rows, int64_t hidden, cudaStream_t stream);

/*
 * add_rmsnorm_quant_fwd -- the same forward with the normalised row emitted
 * as per-row symmetric int8 instead of bf16.  Page: ROCm/aiter issue #5151,
 * section "Cost of fixing": the quantised configurations take `out` through
 * a scaled cast (int8 here) rather than the bf16 store; residual_out is the
 * same bf16 store as in add_rmsnorm_fwd (bit-identical).
 *
 * With y = (acc * inv) * weight in fp32 (the value add_rmsnorm_fwd rounds):
 *   amax       = max over the row of |y|              (exact)
 *   scale[r]   = amax / 127                           (fp32, rounded once)
 *   out_q[r,i] = clamp(rint(y_i / scale[r]), -127, 127), rint ties to even,
 *                the quotient a correctly rounded fp32 division;
 *                scale[r] == 0 gives out_q[r,:] = 0.
 *
 *   out_q         [n_rows x hidden] int8, written (16-byte aligned)
 *   scale         [n_rows] fp32, written (4-byte aligned); q * scale ~ y
 *   residual_out  [n_rows x hidden] bf16, written
 *   other arguments as in add_rmsnorm_fwd.
 */
dradd_status add_rmsnorm_quant_fwd(int8_t* out_q, float* scale, dradd_bf16* residual_out,
                                   const dradd_bf16* x, const dradd_bf16* residual,
                                   const dradd_bf16* weight, float eps,
                                   int64_t n_rows, int64_t hidden, cudaStream_t stream);

/*
 * Explicit launch configuration.  It selects how the work is laid out on the
 * GPU and never changes a single output bit (that is what the invariance
 * tests check).  Zero in a field means "choose automatically".
 *
 *   variant          DRADD_VARIANT_ROWS: each group of threads_per_row
 *                    threads loads its row with 16-byte vector loads into
 *                    registers; DRADD_VARIANT_STAGED: rows are staged into
 *                    shared memory by bulk asynchronous copies (TMA engine)
 *                    several rows ahead of the compute.
 *   threads_per_row  power of two T with T * K * 8 == P (P = next power of
 *                    two >= hidden) for some K in {1, 2, 4, 8}: thread t of
 *                    a row owns the 8-element blocks t, t + T, ..., t + (K-1)T.
 *   rows_per_cta     ROWS: rows processed side by side by one CTA;
 *                    threads_per_row * rows_per_cta <= 1024 and a multiple
 *                    of 32.  STAGED: 1, or 2 for the plain RMSNorm with
 *                    int8, e4m3 or e2m1 out with K <= 4: every thread of a
 *                    CTA of threads_per_row threads carries two adjacent
 *                    rows through each step (one bulk copy and one barrier
 *                    per step serve both; a stage holds both rows).
 *   grid_ctas        number of CTAs; each loops over rows with a stride of
 *                    grid_ctas * rows_per_cta.
 *   stages           STAGED only: rows in flight per CTA (1..8), limited by
 *                    shared memory (2 * hidden * 2 bytes per stage).
 *   fault_inject     test hook, STAGED only: 1 withholds every CTA's first
 *                    copy so that its bounded wait expires; the kernel then
 *                    records DRADD_ERR_TIMEOUT in the device status word,
 *                    waits for its other copies and returns.  Outputs are
 *                    then unspecified.
 *   wait_limit_us    STAGED only: bound on each wait for a staged row, in
 *                    microseconds (0 = 1,000,000).
 *   serialize        0: launch with programmatic stream serialization, so the
 *                    kernel's CTAs may be scheduled while the previous kernel
 *                    in the stream drains; they wait for it to complete (and
 *                    its writes to be visible) before any global load or
 *                    store.  Before that wait, with every buffer in device
 *                    memory, a CTA may only prefetch its first input rows
 *                    into L2 (a hint that moves no data to the SM, so the
 *                    loads after the wait read what memory then holds).
 *                    1: plain launch.
 *   blocks_per_thread K (1, 2, 4 or 8): 8-element blocks per thread.  With
 *                    threads_per_row given it must agree (K = P / 8 / T);
 *                    alone it sets T = P / 8 / K (the automatic stage count
 *                    is then 2).
 *   cluster_ctas     DRADD_VARIANT_SPLIT only (2 or 4, 0 = 2): each row is
 *                    shared by a thread-block cluster of this many CTAs,
 *                    CTA r of the cluster staging and reducing the r-th of
 *                    that many equal slices of the padded row (P / C
 *                    elements, threads_per_row T and K blocks per thread
 *                    within the slice, T * K * 8 * C == P, T >= 32); the
 *                    slice sums meet through distributed shared memory and
 *                    are added in the same tree order.  bf16 output only
 *                    (the quantised entry points reject it); grid_ctas a
 *                    multiple of C.
 *
 * DRADD_VARIANT_WARP: one warp per row (threads_per_row 32, or 0), lane l
 * owning blocks l, l + 32, ... (K = P / 256, so 256 <= P <= 4096, and with
 * a residual P <= 2048); rows loaded straight into registers, the row's
 * reductions within the warp, the weights widened once per CTA into shared
 * memory.  rows_per_cta: warps per CTA (0 = 8, or 4 at P = 4096; at most
 * that); grid_ctas: 0 = as many CTAs as fit on the device at once (at most
 * one per rows_per_cta rows).  stages and fault_inject must be 0.
 *
 * DRADD_VARIANT_CHUNK: the fused q/k call only (see there); the other entry
 * points reject it.
 */
enum {
    DRADD_VARIANT_AUTO = 0,
    DRADD_VARIANT_ROWS = 1,
    DRADD_VARIANT_STAGED = 2,
    DRADD_VARIANT_SPLIT = 3,
    DRADD_VARIANT_WARP = 4,
    DRADD_VARIANT_CHUNK = 5
};

typedef struct dradd_launch_cfg {
    int variant;
    int threads_per_row;
    int rows_per_cta;
    int grid_ctas;
    int stages;
    int fault_inject;
    int wait_limit_us;
    int serialize;
    int blocks_per_thread;
    int cluster_ctas;
} dradd_launch_cfg;

dradd_status add_rmsnorm_fwd_with_config(dradd_bf16* out, dradd_bf16* residual_out,
                                         const dradd_bf16* x, const dradd_bf16* residual,
                                         const dradd_bf16* weight, float eps,
                                         int64_t n_rows, int64_t hidden, cudaStream_t stream,
                                         const dradd_launch_cfg* cfg);

dradd_status add_rmsnorm_quant_fwd_with_config(int8_t* out_q, float* scale,
                                               dradd_bf16* residual_out,
                                               const dradd_bf16* x, const dradd_bf16* residual,
                                               const dradd_bf16* weight, float eps,
                                               int64_t n_rows, int64_t hidden,
                                               cudaStream_t stream,
                                               const dradd_launch_cfg* cfg);

/*
 * dradd_resolve_config -- fill the automatic choices of *cfg for a call of
 * the given shape and operation, as the entry points would, and validate
 * the explicit ones.  `op` is one of DRADD_OP_* (0 and 1 are the bf16 and
 * int8 residual-add forms, 2 and 3 plain RMSNorm, 4 and 5 the fp8 forms,
 * 6 and 7 the fp4 forms).  grid_ctas is filled from
 * `sm_count` (pass 0 to query the current device); for the staged variant
 * the entry points size the grid with the CUDA occupancy calculator instead.
 * Does no GPU work when sm_count > 0.
 */
enum {
    DRADD_OP_ADD_RMSNORM = 0,
    DRADD_OP_ADD_RMSNORM_QUANT = 1,
    DRADD_OP_RMSNORM = 2,
    DRADD_OP_RMSNORM_QUANT = 3,
    DRADD_OP_ADD_RMSNORM_FP8 = 4,
    DRADD_OP_RMSNORM_FP8 = 5,
    DRADD_OP_ADD_RMSNORM_FP4 = 6,
    DRADD_OP_RMSNORM_FP4 = 7
};

dradd_status dradd_resolve_config(int64_t n_rows, int64_t hidden, int op, int sm_count,
                                  dradd_launch_cfg* cfg);

/*
 * rmsnorm_fwd -- plain RMSNorm forward, the residual-free half of the page's
 * reference() (ROCm/aiter issue #5151, "Steps to Reproduce"): acc = fp32(x)
 * (exact), then exactly the normalisation of add_rmsnorm_fwd:
 *   out = bf16_rne((acc * (1 / sqrt(S / hidden + eps))) * fp32(weight))
 * with the same pairwise tree, the same rounding steps and the same launch
 * invariance.  There is no residual and no residual_out.
 *
 *   out     [n_rows x hidden] bf16, written (may be exactly x)
 *   x       [n_rows x hidden] bf16, read
 *   weight  [hidden] bf16, read
 * Conventions, errors and aliasing as for add_rmsnorm_fwd.
 */
dradd_status rmsnorm_fwd(dradd_bf16* out, const dradd_bf16* x, const dradd_bf16* weight, float eps,
                         int64_t n_rows, int64_t hidden, cudaStream_t stream);

/*
 * rmsnorm_quant_fwd -- plain RMSNorm with the per-row symmetric int8 output
 * of add_rmsnorm_quant_fwd (same amax, scale and rounding rules).
 *   out_q [n_rows x hidden] int8, scale [n_rows] fp32, written.
 */
dradd_status rmsnorm_quant_fwd(int8_t* out_q, float* scale, const dradd_bf16* x,
                               const dradd_bf16* weight, float eps, int64_t n_rows, int64_t hidden,
                               cudaStream_t stream);

dradd_status rmsnorm_fwd_with_config(dradd_bf16* out, const dradd_bf16* x, const dradd_bf16* weight,
                                     float eps, int64_t n_rows, int64_t hidden, cudaStream_t stream,
                                     const dradd_launch_cfg* cfg);

dradd_status rmsnorm_quant_fwd_with_config(int8_t* out_q, float* scale, const dradd_bf16* x,
                                           const dradd_bf16* weight, float eps, int64_t n_rows,
                                           int64_t hidden, cudaStream_t stream,
                                           const dradd_launch_cfg* cfg);

/*
 * add_rmsnorm_fp8_fwd -- the residual-add + RMSNorm forward with the
 * normalised row emitted as per-row scaled fp8 e4m3 codes (OCP "e4m3fn":
 * 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * largest finite 448).  Page: ROCm/aiter issue #5151, "Cost of fixing": the
 * quantised configurations take out through a scaled cast to int8, fp8 or
 * fp4 instead of the bf16 store.  With y as in add_rmsnorm_quant_fwd:
 *   amax       = max over the row of |y|                 (exact)
 *   scale[r]   = amax / 448                              (fp32, rounded once)
 *   out_q[r,i] = e4m3(y_i / scale[r]): the quotient a correctly rounded fp32
 *                division, then rounded to the nearest e4m3 value, ties to
 *                the even code, magnitudes past 448 saturating to 448;
 *                scale[r] == 0 gives code 0.
 *   out_q         [n_rows x hidden] e4m3 codes (uint8), written (16-byte
 *                 aligned); code * scale ~ y
 *   scale, residual_out and the other arguments as in add_rmsnorm_quant_fwd.
 */
dradd_status add_rmsnorm_fp8_fwd(uint8_t* out_q, float* scale, dradd_bf16* residual_out,
                                 const dradd_bf16* x, const dradd_bf16* residual,
                                 const dradd_bf16* weight, float eps, int64_t n_rows,
                                 int64_t hidden, cudaStream_t stream);

dradd_status add_rmsnorm_fp8_fwd_with_config(uint8_t* out_q, float* scale, dradd_bf16* residual_out,
                                             const dradd_bf16* x, const dradd_bf16* residual,
                                             const dradd_bf16* weight, float eps, int64_t n_rows,
                                             int64_t hidden, cudaStream_t stream,
                                             const dradd_launch_cfg* cfg);

/* rmsnorm_fp8_fwd -- plain RMSNorm (no residual) with the same e4m3 output. */
dradd_status rmsnorm_fp8_fwd(uint8_t* out_q, float* scale, const dradd_bf16* x,
                             const dradd_bf16* weight, float eps, int64_t n_rows, int64_t hidden,
                             cudaStream_t stream);

dradd_status rmsnorm_fp8_fwd_with_config(uint8_t* out_q, float* scale, const dradd_bf16* x,
                                         const dradd_bf16* weight, float eps, int64_t n_rows,
                                         int64_t hidden, cudaStream_t stream,
                                         const dradd_launch_cfg* cfg);

/*
 * add_rmsnorm_fp4_fwd -- the residual-add + RMSNorm forward with the
 * normalised row emitted as per-row scaled fp4 e2m1 codes (1 sign, 2
 * exponent bits with bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2,
 * 3, 4, 6), the fp4 scaled cast of the page's "Cost of fixing":
 *   scale[r]   = amax / 6                                (fp32, rounded once)
 *   code       = e2m1(y_i / scale[r]): the correctly rounded fp32 quotient
 *                rounded to the nearest e2m1 value, ties to the even code,
 *                magnitudes past 6 saturating to 6; scale[r] == 0 gives 0.
 *   out_q         [n_rows x hidden / 2] bytes, written (16-byte aligned):
 *                 byte j of a row holds element 2j in its low nibble and
 *                 element 2j + 1 in its high nibble; bit 3 of a code is the
 *                 sign.
 *   scale, residual_out and the other arguments as in add_rmsnorm_quant_fwd.
 */
dradd_status add_rmsnorm_fp4_fwd(uint8_t* out_q, float* scale, dradd_bf16* residual_out,
                                 const dradd_bf16* x, const dradd_bf16* residual,
                                 const dradd_bf16* weight, float eps, int64_t n_rows,
                                 int64_t hidden, cudaStream_t stream);

dradd_status add_rmsnorm_fp4_fwd_with_config(uint8_t* out_q, float* scale, dradd_bf16* residual_out,
                                             const dradd_bf16* x, const dradd_bf16* residual,
                                             const dradd_bf16* weight, float eps, int64_t n_rows,
                                             int64_t hidden, cudaStream_t stream,
                                             const dradd_launch_cfg* cfg);

/* rmsnorm_fp4_fwd -- plain RMSNorm (no residual) with the same e2m1 output. */
dradd_status rmsnorm_fp4_fwd(uint8_t* out_q, float* scale, const dradd_bf16* x,
                             const dradd_bf16* weight, float eps, int64_t n_rows, int64_t hidden,
                             cudaStream_t stream);

dradd_status rmsnorm_fp4_fwd_with_config(uint8_t* out_q, float* scale, const dradd_bf16* x,
                                         const dradd_bf16* weight, float eps, int64_t n_rows,
                                         int64_t hidden, cudaStream_t stream,
                                         const dradd_launch_cfg* cfg);

/*
 * residual_add_fwd -- the residual update alone, the other half of the
 * page's reference(): residual_out = bf16_rne(fp32(x) + fp32(residual)),
 * element by element, bit-identical to add_rmsnorm_fwd's residual_out (the
 * store the page is about: "Problem Description", "Cost of fixing").
 *
 *   residual_out  [n_rows x hidden] bf16, written (may be exactly x or
 *                 residual)
 *   x, residual   [n_rows x hidden] bf16, read
 * Shape, alignment and aliasing rules as for add_rmsnorm_fwd (no weight,
 * no eps).
 */
dradd_status residual_add_fwd(dradd_bf16* residual_out, const dradd_bf16* x,
                              const dradd_bf16* residual, int64_t n_rows, int64_t hidden,
                              cudaStream_t stream);

/*
 * fused_qk_rmsnorm_group_quant_fwd -- two independent RMSNorms in one launch
 * ("q" and "k" rows), q optionally with a residual add and a per-group e4m3
 * output.  Page: ROCm/aiter issue #5151, section "Notes", which names the
 * fused q/k RMSNorm + group quant kernel among those whose bf16 residual
 * stores were not audited; the page prints no formula for it, and this is
 * the plainest reading of the name on top of the row function above:
 *   q rows (n_q_rows x q_hidden): with q_residual != NULL, acc = fp32(q) +
 *     fp32(q_residual) and q_residual_out = bf16_rne(acc) (the residual
 *     store, round to nearest even); else acc = fp32(q).  y = the row
 *     function of add_rmsnorm_fwd with q_weight and q_eps.
 *       group_size == 0: q_out = bf16_rne(y), [n_q_rows x q_hidden] bf16.
 *       group_size  > 0: y is cut into consecutive groups of group_size
 *         elements; each group gets scale = amax / 448 and codes
 *         e4m3(y / scale) exactly as a row of add_rmsnorm_fp8_fwd.
 *         q_out: [n_q_rows x q_hidden] e4m3 codes (uint8);
 *         q_scale: [n_q_rows x (q_hidden / group_size)] fp32, row-major.
 *         group_size: a power of two, 8 <= group_size <= 256, dividing
 *         q_hidden (else DRADD_ERR_BAD_SHAPE).
 *   k rows (n_k_rows x k_hidden): plain RMSNorm with k_weight and k_eps,
 *     k_out = bf16_rne(y).
 * q_hidden and k_hidden: multiples of 8, at most DRADD_QK_MAX_HIDDEN
 * (else DRADD_ERR_UNSUPPORTED_HIDDEN).  A per-head q/k norm is the same
 * call with rows = tokens x heads and hidden = the head size.  Either row count may be 0: that side is then
 * ignored (its pointers, hidden and eps are not inspected); both 0 is a
 * no-op.  q_residual_out is written only when q_residual is non-NULL.
 * Every result is bit-identical to two separate calls of the single-set
 * entry points and independent of the launch configuration.
 * Aliasing: q_out may be exactly q (bf16 out only), q_residual_out exactly
 * q_residual, k_out exactly k; no other overlap.  Alignment: every array
 * 16 bytes, q_scale 4 bytes.  Other conventions as for add_rmsnorm_fwd.
 */
dradd_status fused_qk_rmsnorm_group_quant_fwd(void* q_out, float* q_scale, dradd_bf16* q_residual_out,
                                              dradd_bf16* k_out, const dradd_bf16* q,
                                              const dradd_bf16* q_residual, const dradd_bf16* q_weight,
                                              const dradd_bf16* k, const dradd_bf16* k_weight, float q_eps,
                                              float k_eps, int64_t n_q_rows, int64_t q_hidden, int64_t n_k_rows,
                                              int64_t k_hidden, int64_t group_size, cudaStream_t stream);

/*
 * Test hook: the fused q/k call with an explicit configuration.  variant:
 * STAGED (rows staged through shared memory by bulk copies) or ROWS (rows
 * loaded straight into registers); AUTO picks by the longer side's padded
 * width P: staged for P <= 256 and P > 2048, rows in between, and staged
 * whenever stages or fault_inject is set.
 * threads_per_row is read here as the threads of a CTA: a power of two
 * 32..512, at most 256 when a side needs 8 blocks of 8 per thread.
 * blocks_per_thread: the least K both sides use (each side raises it to
 * what the CTA size needs; at most P / 8 and 8).  grid_ctas: total CTAs,
 * shared by the two sides.  stages (staged only): stages per side, 1..8.
 * fault_inject, wait_limit_us and serialize as for
 * add_rmsnorm_fwd_with_config (staged only for the first two);
 * rows_per_cta must be 0.  WARP: one warp per row on both sides, each lane
 * owning blocks l, l + 32, ... of its row (both sides 256 <= P <= 2048),
 * threads_per_row read as the threads of a CTA (a multiple of 32 up to 256,
 * 0 = 256), stages per warp ring (0 = 2), fault_inject and wait_limit_us
 * as for the staged variant, blocks_per_thread 0.  CHUNK: the q
 * rows in 512-element chunks, one warp a chunk and one CTA a row (the CTA
 * has hidden / 512 warps rounded up, 2..8: 512 < q P <= 4096), each warp
 * computing its chunk's subtree of the row's sum, the chunk sums folded in
 * the same tree order after one barrier; the k rows one warp each as in
 * WARP, in CTAs of the same size (256 <= k P <= 2048); stages per warp
 * ring (0 = 2), fault_inject and wait_limit_us as for the staged variant,
 * threads_per_row, blocks_per_thread and rows_per_cta 0.  Results never
 * depend on it.
 */
dradd_status fused_qk_rmsnorm_group_quant_fwd_with_config(
    void* q_out, float* q_scale, dradd_bf16* q_residual_out, dradd_bf16* k_out, const dradd_bf16* q,
    const dradd_bf16* q_residual, const dradd_bf16* q_weight, const dradd_bf16* k, const dradd_bf16* k_weight,
    float q_eps, float k_eps, int64_t n_q_rows, int64_t q_hidden, int64_t n_k_rows, int64_t k_hidden,
    int64_t group_size, cudaStream_t stream, const dradd_launch_cfg* cfg);

/* The launch plan of a fused q/k call (for tests and reports). */
typedef struct dradd_qk_plan {
    int variant;          /* DRADD_VARIANT_ROWS, _STAGED or _WARP (0 for an empty call) */
    int threads_per_cta;
    int dyn_smem_bytes;   /* staged: shared memory for the stages; warp: for the fp32 weights */
    int q_threads_per_row, q_rows_per_cta, q_stages, q_ctas;  /* 0 when n_q_rows == 0 */
    int k_threads_per_row, k_rows_per_cta, k_stages, k_ctas;  /* 0 when n_k_rows == 0 */
} dradd_qk_plan;

/*
 * dradd_qk_resolve_config -- the plan the fused q/k call would use, without
 * launching.  q_residual != 0: the call has a q residual (its stages hold
 * both tensors).  sm_count > 0 stands in for the device's SM count (no GPU
 * needed; the automatic grid then assumes 2048 / threads CTAs per SM, where
 * the real call asks the occupancy calculator); sm_count <= 0 asks the
 * current device, and for the staged and warp-per-row variants with an
 * automatic grid its occupancy calculator, as the call does, so the plan is
 * the call's.  cfg may be NULL (automatic).  Returns the shape and
 * configuration errors of the call.
 */
dradd_status dradd_qk_resolve_config(int64_t n_q_rows, int64_t q_hidden, int64_t n_k_rows, int64_t k_hidden,
                                     int64_t group_size, int q_residual, int sm_count,
                                     const dradd_launch_cfg* cfg, dradd_qk_plan* plan);

/*
 * Log-sum-exp merge and launch-invariant elementwise functions.
 * Page: ROCm/TransformerEngine issue #693, "CP LSE merge switches compiled
 * variants on ROCm, breaking forward reproducibility".  Context-parallel
 * attention merges the softmax log-sum-exp of blocks computed on different
 * ranks ("Summary"; one merge function is for the second half of the
 * sequence), and the page traces a forward mismatch to log1p (and cosh)
 * giving different bits under different launch configurations of the same
 * compiled function ("Root cause", "Minimal reproducer").  Here every
 * element is computed by one fixed sequence of fp32 operations whatever
 * the launch configuration: the results below depend on the inputs only.
 *
 * lse_merge_fwd -- out[i] = log(e^a[i] + e^b[i]), evaluated as
 *   hi + log1p(exp(lo - hi)) with hi = max(a, b), lo = min(a, b), in fp32:
 *   the CUDA math library's expf, then log1p of an argument in [0, 1] by
 *   the atanh series (IEEE operations only; within 2.95 x 2^-24 relative
 *   for every fp32 argument).  Both -inf (two empty blocks) gives -inf; a
 *   +inf operand gives +inf; NaN gives NaN.  Within 1 ulp(result) + 2^-22
 *   of the exact value (the bound the tests use).
 *   out, lse_a, lse_b: n fp32 values, 4-byte aligned; out may be exactly
 *   lse_a or lse_b (an in-place running merge); no other overlap.
 */
dradd_status lse_merge_fwd(float* out, const float* lse_a, const float* lse_b, int64_t n, cudaStream_t stream);

/*
 * lse_merge_2d_fwd -- the same merge over n_rows rows of n_cols elements
 * with a row stride (in elements, >= n_cols) per operand:
 *   out[r * out_stride + c] = merge(lse_a[r * a_stride + c],
 *                                   lse_b[r * b_stride + c]).
 * The second-half merge of a [rows x S] running lse with a [rows x S/2]
 * per-step lse is lse_merge_2d_fwd(lse + S/2, S, lse + S/2, S, step, S/2,
 * rows, S/2).  out may be exactly lse_a or lse_b (same address and stride);
 * no other overlap of the spans the three operands cover.
 */
dradd_status lse_merge_2d_fwd(float* out, int64_t out_stride, const float* lse_a, int64_t a_stride,
                              const float* lse_b, int64_t b_stride, int64_t n_rows, int64_t n_cols,
                              cudaStream_t stream);

/*
 * Test hook: the merge with an explicit configuration.  threads_per_row is
 * read as the threads of a CTA (a power of two, 32..1024), blocks_per_thread
 * as the elements a thread handles per pass (1, 2, 4, 8), grid_ctas as the
 * CTAs; serialize as above; every other field must be 0.  Results never
 * depend on it.
 */
dradd_status lse_merge_2d_fwd_with_config(float* out, int64_t out_stride, const float* lse_a, int64_t a_stride,
                                          const float* lse_b, int64_t b_stride, int64_t n_rows, int64_t n_cols,
                                          cudaStream_t stream, const dradd_launch_cfg* cfg);

enum { DRADD_UNARY_LOG1P = 0, DRADD_UNARY_COSH = 1, DRADD_UNARY_EXP = 2 };

/*
 * invariant_unary_fwd -- out[i] = f(x[i]) for f = log1pf, coshf or expf
 * (DRADD_UNARY_*; CUDA math library: within 1, 3 and 2 ulp in the tests),
 * the same bits under every launch configuration.  n fp32 values, 4-byte
 * aligned; out may be exactly x; an unknown op is DRADD_ERR_BAD_CONFIG.
 */
dradd_status invariant_unary_fwd(float* out, const float* x, int64_t n, int op, cudaStream_t stream);

/* Test hook: invariant_unary_fwd with an explicit configuration (fields as
 * for lse_merge_2d_fwd_with_config). */
dradd_status invariant_unary_fwd_with_config(float* out, const float* x, int64_t n, int op, cudaStream_t stream,
                                             const dradd_launch_cfg* cfg);

/*
 * dradd_device_status -- synchronise `stream`, then return DRADD_OK or the
 * error a kernel recorded on the current device since the last clear:
 * DRADD_ERR_TIMEOUT (a bounded wait expired) or DRADD_ERR_UNDRAINED (it
 * expired and, after several more wait limits, a bulk copy the kernel had
 * issued still had not landed in shared memory: the device's state is
 * suspect and the context should be rebuilt).  The word is read, and with
 * clear != 0 reset, by one atomic exchange on `stream`: a kernel on another
 * stream that records an error at the same time is either seen by this read
 * or left for the next one.
 */
dradd_status dradd_device_status(cudaStream_t stream, int clear);

/*
 * dradd_last_device_status -- the optional check after a call: synchronise
 * `stream`, return DRADD_OK or the error a kernel recorded on the current
 * device since the last read (DRADD_ERR_TIMEOUT: a bounded wait for a
 * staged row expired, and that call's outputs are unspecified), and reset
 * the word.  Equal to dradd_device_status(stream, 1).
 */
dradd_status dradd_last_device_status(cudaStream_t stream);

/*
 * dradd_bf16_convert_range -- test hook: convert the `count` fp32 bit
 * patterns first, first+1, ... (mod 2^32) on the device, with method
 * 0 = the bf16 conversion the kernels use, 1 = integer round-half-even bit
 * arithmetic to bf16, 2 = the hardware cvt.rn.bf16x2.f32 instruction,
 * 3 = the e4m3 conversion the fp8 kernels use (code in the low byte),
 * 4 = the e2m1 conversion the fp4 kernels use (code in the low nibble),
 * 5 = CUDA's own __float2bfloat16_rn (a library reference for method 0).
 * `out` is a device array of `count` 16-bit words (2-byte aligned).
 */
dradd_status dradd_bf16_convert_range(dradd_bf16* out, uint64_t first, int64_t count,
                                      int method, cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* dradd_status_string(dradd_status status);

/* DRADD_ABI_VERSION of the loaded library. */
int dradd_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DRADD_H */
