// Fused q/k RMSNorm kernels with bf16 q out: every (KQ, KK) pair, q with
// and without a residual.
#include "dradd_kernels.cuh"

namespace dradd {

QkKernelFn qk_fn_bf16(int kq, int kk, bool add)
{
    return add ? qk_table<false, true>(kq, kk) : qk_table<false, false>(kq, kk);
}

}  // namespace dradd
