// Fused q/k RMSNorm kernels with per-group e4m3 q out, one warp per row:
// every (KQ, KK) pair up to 8, q with and without a residual; and the
// chunked-q kernels (q rows in 512-element chunks, one warp each).
#include "dradd_qk.cuh"

namespace dradd {

QkKernelFn qk_fn_e4m3_warp(int kq, int kk, bool add)
{
    return add ? qk_warp_table<true, true>(kq, kk) : qk_warp_table<true, false>(kq, kk);
}

QkKernelFn qk_fn_e4m3_chunk(int kk, bool add)
{
    return add ? qk_chunk_table<true, true>(kk) : qk_chunk_table<true, false>(kk);
}

}  // namespace dradd
