// dradd_warp_norm.cu -- warp-per-row kernels of the plain RMSNorm forward
// (no residual; every output kind).
#include "dradd_warp.cuh"

namespace dradd {

KernelFn warp_fn_norm(int out, int K)
{
    switch (out) {
    case kOutBf16: return warp_table<kOutBf16, false>(K);
    case kOutInt8: return warp_table<kOutInt8, false>(K);
    case kOutE4m3: return warp_table<kOutE4m3, false>(K);
    case kOutE2m1: return warp_table<kOutE2m1, false>(K);
    default: return nullptr;
    }
}

}  // namespace dradd
