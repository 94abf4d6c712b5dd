// Split-row kernels (a cluster of 2 or 4 CTAs per row), bf16 out, residual-add form.
#include "dradd_split.cuh"

namespace dradd {

KernelFn split_fn_add(int T, int K, int C)
{
    return C == 2 ? split_table<2, true>(T, K) : C == 4 ? split_table<4, true>(T, K) : nullptr;
}

}  // namespace dradd
