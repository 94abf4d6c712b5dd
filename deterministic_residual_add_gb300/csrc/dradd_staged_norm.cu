// dradd_staged_norm.cu -- staged kernels of plain RMSNorm (no residual),
// bf16 and int8 out.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_norm(int T, int K, bool quant) { return staged_table<false>(T, K, quant); }

}  // namespace dradd
