// Fused q/k RMSNorm kernels with per-group e4m3 q out, rows staged through
// shared memory: every (KQ, KK) pair, q with and without a residual.
#include "dradd_qk.cuh"

namespace dradd {

QkKernelFn qk_fn_e4m3_staged(int kq, int kk, bool add)
{
    return add ? qk_table<true, true, true>(kq, kk) : qk_table<true, false, true>(kq, kk);
}

}  // namespace dradd
