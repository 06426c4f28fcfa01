// Forward kernel instances for head size 128 (causal / non-causal, bf16 / fp32 output).
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_128(const FwdParams& p, bool causal, fa_dtype o_dtype, cudaStream_t st)
{
    return launch_fwd_d<128>(p, causal, o_dtype, st);
}
}  // namespace fa
