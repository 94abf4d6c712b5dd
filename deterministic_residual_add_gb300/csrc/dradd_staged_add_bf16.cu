// dradd_staged_add_bf16.cu -- staged kernels of the residual-add + RMSNorm
// forward with bf16 out; one translation unit per (mode, output) so
// that the build compiles them in parallel.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_add_bf16(int T, int K) { return staged_table<kOutBf16, true>(T, K); }

}  // namespace dradd
