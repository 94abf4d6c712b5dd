// dradd_warp_add.cu -- warp-per-row kernels of the residual-add + RMSNorm
// forward (every output kind); one translation unit per mode so that the
// build compiles them in parallel.
#include "dradd_warp.cuh"

namespace dradd {

KernelFn warp_fn_add(int out, int K)
{
    switch (out) {
    case kOutBf16: return warp_table<kOutBf16, true>(K);
    case kOutInt8: return warp_table<kOutInt8, true>(K);
    case kOutE4m3: return warp_table<kOutE4m3, true>(K);
    case kOutE2m1: return warp_table<kOutE2m1, true>(K);
    default: return nullptr;
    }
}

}  // namespace dradd
