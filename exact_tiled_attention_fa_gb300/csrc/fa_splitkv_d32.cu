// Split-KV tensor-core kernel instances for head size 32.
#include "fa_splitkv_kernel.cuh"

namespace fa {
cudaError_t launch_splitkv_32(const SplitParams& p, bool causal, bool varlen, cudaStream_t st)
{
    return launch_splitkv_d<32>(p, causal, varlen, st);
}
}  // namespace fa
