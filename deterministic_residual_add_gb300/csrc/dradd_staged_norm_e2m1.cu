// dradd_staged_norm_e2m1.cu -- staged kernels of the plain RMSNorm (no residual)
// forward with per-row fp4 e2m1 out; one translation unit per (mode,
// output) so that the build compiles them in parallel.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_norm_e2m1(int T, int K) { return staged_table<kOutE2m1, false>(T, K); }
KernelFn staged_pair_fn_norm_e2m1(int T, int K) { return staged_pair_table<kOutE2m1>(T, K); }

}  // namespace dradd
