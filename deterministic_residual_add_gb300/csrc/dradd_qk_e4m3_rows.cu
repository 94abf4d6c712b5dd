// Fused q/k RMSNorm kernels with per-group e4m3 q out, rows loaded into
// registers: every (KQ, KK) pair, q with and without a residual.
#include "dradd_qk.cuh"

namespace dradd {

QkKernelFn qk_fn_e4m3_rows(int kq, int kk, bool add)
{
    return add ? qk_table<true, true, false>(kq, kk) : qk_table<true, false, false>(kq, kk);
}

}  // namespace dradd
