// Fused q/k RMSNorm kernels with bf16 q out, one warp per row: every
// (KQ, KK) pair up to 8, q with and without a residual.
#include "dradd_qk.cuh"

namespace dradd {

QkKernelFn qk_fn_bf16_warp(int kq, int kk, bool add)
{
    return add ? qk_warp_table<false, true>(kq, kk) : qk_warp_table<false, false>(kq, kk);
}

QkKernelFn qk_fn_bf16_chunk(int kk, bool add)
{
    return add ? qk_chunk_table<false, true>(kk) : qk_chunk_table<false, false>(kk);
}

}  // namespace dradd
