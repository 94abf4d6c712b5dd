// dradd_staged_norm_int8.cu -- staged kernels of the plain RMSNorm (no residual)
// forward with per-row int8 out; one translation unit per (mode, output) so
// that the build compiles them in parallel.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_norm_int8(int T, int K) { return staged_table<kOutInt8, false>(T, K); }
KernelFn staged_pair_fn_norm_int8(int T, int K) { return staged_pair_table<kOutInt8>(T, K); }

}  // namespace dradd
