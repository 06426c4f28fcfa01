// fa_kernel_common.cuh -- small device helpers shared by the forward and backward
// kernels: failure recording and row stores in the output element type.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace fa {

constexpr unsigned long long kDrainLimitNs = 1000000000ull;  // 1 s for draining after a failure

__device__ __forceinline__ void record_failure(int* status, volatile int* abort_flag, int code)
{
    *abort_flag = 1;
    atomicCAS(status, 0, code);
}

template <typename OutT>
__device__ __forceinline__ void store_row32(OutT* dst, const float (&v)[32]);

template <>
__device__ __forceinline__ void store_row32<float>(float* dst, const float (&v)[32])
{
#pragma unroll
    for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}

template <>
__device__ __forceinline__ void store_row32<__nv_bfloat16>(__nv_bfloat16* dst, const float (&v)[32])
{
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        uint4 u;
        u.x = pack_bf16x2(v[i + 0], v[i + 1]);
        u.y = pack_bf16x2(v[i + 2], v[i + 3]);
        u.z = pack_bf16x2(v[i + 4], v[i + 5]);
        u.w = pack_bf16x2(v[i + 6], v[i + 7]);
        *reinterpret_cast<uint4*>(dst + i) = u;
    }
}

// 32 fp32 values of a row to a 32-byte aligned destination, in 32-byte stores (a warp writing one
// row per thread then fills whole sectors instead of halves).
__device__ __forceinline__ void store_row32_aligned32(float* dst, const float (&v)[32])
{
#pragma unroll
    for (int i = 0; i < 32; i += 8) st_global_v8_f32(dst + i, v + i);
}

template <typename OutT>
__device__ __forceinline__ void store_row16(OutT* dst, const float (&v)[16]);

template <>
__device__ __forceinline__ void store_row16<float>(float* dst, const float (&v)[16])
{
#pragma unroll
    for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}

template <>
__device__ __forceinline__ void store_row16<__nv_bfloat16>(__nv_bfloat16* dst, const float (&v)[16])
{
#pragma unroll
    for (int i = 0; i < 16; i += 8) {
        uint4 u;
        u.x = pack_bf16x2(v[i + 0], v[i + 1]);
        u.y = pack_bf16x2(v[i + 2], v[i + 3]);
        u.z = pack_bf16x2(v[i + 4], v[i + 5]);
        u.w = pack_bf16x2(v[i + 6], v[i + 7]);
        *reinterpret_cast<uint4*>(dst + i) = u;
    }
}

// Launch with programmatic stream serialization: the kernel may start (and run its setup) while
// the previous kernel on the stream finishes, if that kernel has called grid_launch_dependents.
// Every kernel launched this way calls grid_dependency_wait() before its first global read or write
// that the previous kernel could affect, and calls grid_launch_dependents() only after that wait:
// the wait returns once the previous kernel has completed and its writes are visible, so when any
// of these kernels starts, every kernel before its immediate predecessor has completed.
template <typename... Expected, typename... Actual>
inline cudaError_t launch_pdl(void (*kern)(Expected...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, const Actual&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace fa
