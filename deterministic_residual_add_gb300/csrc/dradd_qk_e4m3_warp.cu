// Fused q/k RMSNorm kernels with per-group e4m3 q out, one warp per row:
// every (KQ, KK) pair up to 8, q with and without a residual.
#include "dradd_qk.cuh"

namespace dradd {

QkKernelFn qk_fn_e4m3_warp(int kq, int kk, bool add)
{
    return add ? qk_warp_table<true, true>(kq, kk) : qk_warp_table<true, false>(kq, kk);
}

}  // namespace dradd
