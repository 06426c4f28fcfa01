// Grouped-query decode on the tensor core, transposed form (head size 128, 5-32 heads per group).
#include "fa_gqa_kernel.cuh"

namespace fa {
cudaError_t launch_gqa_tc(const SplitParams& p, cudaStream_t st) { return launch_gqa(p, st); }
}  // namespace fa
