// dradd_staged_add_e2m1.cu -- staged kernels of the residual-add + RMSNorm
// forward with per-row fp4 e2m1 out; one translation unit per (mode,
// output) so that the build compiles them in parallel.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_add_e2m1(int T, int K) { return staged_table<kOutE2m1, true>(T, K); }

}  // namespace dradd
