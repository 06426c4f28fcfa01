// Forward kernel instances for head size 128 (causal / non-causal, bf16 / fp32 output, and fp32
// split-mode partials).
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_128(const FwdParams& p, bool causal, fa_dtype o_dtype, cudaStream_t st)
{
    return launch_fwd_d<128>(p, causal, o_dtype, st);
}
cudaError_t launch_fwd_split_128(const FwdParams& p, bool causal, cudaStream_t st)
{
    return launch_fwd_split_d<128>(p, causal, st);
}
}  // namespace fa
