// dradd_staged_add.cu -- staged kernels of the residual-add + RMSNorm
// forward (bf16 and int8 out), one translation unit so that the build can
// compile the modes in parallel.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_add(int T, int K, bool quant) { return staged_table<true>(T, K, quant); }

}  // namespace dradd
