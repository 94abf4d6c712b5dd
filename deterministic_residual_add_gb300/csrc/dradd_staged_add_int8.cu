// dradd_staged_add_int8.cu -- staged kernels of the residual-add + RMSNorm
// forward with per-row int8 out; one translation unit per (mode, output) so
// that the build compiles them in parallel.
#include "dradd_kernels.cuh"

namespace dradd {

KernelFn staged_fn_add_int8(int T, int K) { return staged_table<kOutInt8, true>(T, K); }

}  // namespace dradd
