// Fused q/k RMSNorm kernels with bf16 q out, rows loaded into registers: every
// (KQ, KK) pair, q with and without a residual.
#include "dradd_qk.cuh"

namespace dradd {

QkKernelFn qk_fn_bf16_rows(int kq, int kk, bool add)
{
    return add ? qk_table<false, true, false>(kq, kk) : qk_table<false, false, false>(kq, kk);
}

}  // namespace dradd
