// dradd_staged_add_e4m3.cu -- staged kernels of the residual-add + RMSNorm
// forward with per-row e4m3 out; one translation unit per (mode, output) so
// that the build compiles them in parallel.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_add_e4m3(int T, int K) { return staged_table<kOutE4m3, true>(T, K); }

}  // namespace dradd
