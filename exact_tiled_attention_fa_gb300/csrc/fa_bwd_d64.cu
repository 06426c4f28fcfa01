// Backward tensor-core kernel instances for head size 64.
#include "fa_bwd_kernel.cuh"

namespace fa {
cudaError_t launch_bwd_64(const BwdParams& p, bool causal, fa_dtype grad_dtype, cudaStream_t st)
{
    return launch_bwd_d<64>(p, causal, grad_dtype, st);
}
}  // namespace fa
