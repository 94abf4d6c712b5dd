// dradd_staged_norm_e4m3.cu -- staged kernels of the plain RMSNorm (no residual)
// forward with per-row e4m3 out; one translation unit per (mode, output) so
// that the build compiles them in parallel.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_norm_e4m3(int T, int K) { return staged_table<kOutE4m3, false>(T, K); }
KernelFn staged_pair_fn_norm_e4m3(int T, int K) { return staged_pair_table<kOutE4m3>(T, K); }

}  // namespace dradd
