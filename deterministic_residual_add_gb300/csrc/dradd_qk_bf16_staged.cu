// Fused q/k RMSNorm kernels with bf16 q out, rows staged through shared
// memory: every (KQ, KK) pair, q with and without a residual.
#include "dradd_qk.cuh"

namespace dradd {

QkKernelFn qk_fn_bf16_staged(int kq, int kk, bool add)
{
    return add ? qk_table<false, true, true>(kq, kk) : qk_table<false, false, true>(kq, kk);
}

}  // namespace dradd
