// fa_bwd.cu -- the two memory-bound kernels around the backward's tensor-core kernel.
//
// Preparation ("flash_lab.py", section 3 `flash_bwd`, first step): for every query row
// D_i = sum_c dO_ic O_ic, stored pre-multiplied by the scale (the tensor-core kernel
// folds the scale into dS); the forward's log-sum-exp is stored in base 2, with +inf
// for rows past N and rows that see no key (their P is then exactly 0); and the fp32
// dQ accumulator is zeroed.  Rows are padded to whole 128-row query tiles.
//
// dQ conversion: the accumulator, laid out per (head, query tile) as [d/4][128 rows][4] (d = 128:
// the tensor-core kernel's atomics from one warp cover 512 contiguous bytes) or [4][d/4][32][4]
// (d <= 64: each warp's bulk reductions cover 2 KB blocks), is written out as dQ [head][N][d] in
// the gradient dtype.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"

namespace fa {

constexpr int kPrepThreads = 256;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8])
{
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ void load8(const float* p, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// One thread per 8 elements of a padded row; the G = d / 8 threads of a row are
// consecutive lanes of one warp and reduce with shuffles.
template <typename OT>
__global__ void __launch_bounds__(kPrepThreads) fa_bwd_prep_kernel(const BwdPrepParams p)
{
    grid_dependency_wait();    // O, dO and LSE are written by earlier kernels on the stream
    grid_launch_dependents();  // the tensor-core kernel may begin its setup (it waits for this grid)
    const int G = p.d / 8;
    const long long rows = static_cast<long long>(p.BH) * p.Tr * kBlockM;
    const long long t = static_cast<long long>(blockIdx.x) * kPrepThreads + threadIdx.x;
    const long long row = t / G;
    const int c = static_cast<int>(t - row * G);
    const bool in_range = row < rows;
    float acc = 0.f;
    int bh = 0, q = 0;
    if (in_range) {
        bh = static_cast<int>(row / (static_cast<long long>(p.Tr) * kBlockM));
        q = static_cast<int>(row - static_cast<long long>(bh) * p.Tr * kBlockM);
        if (q < p.N) {
            const size_t e = (static_cast<size_t>(bh) * p.N + q) * p.d + 8 * c;
            float g[8], o[8];
            load8(reinterpret_cast<const __nv_bfloat16*>(p.d_o) + e, g);
            load8(reinterpret_cast<const OT*>(p.o) + e, o);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc = fmaf(g[i], o[i], acc);
        }
        // zero 8 floats of the dQ accumulator (it holds rows * d = 8 * (rows * G) floats)
        float4* z = reinterpret_cast<float4*>(p.dq_acc + 8 * t);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int w = G / 2; w >= 1; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (in_range && c == 0) {
        float l2 = INFINITY, ds = 0.f;
        if (q < p.N) {
            const float lse = p.lse[static_cast<size_t>(bh) * p.N + q];
            if (lse != -INFINITY) l2 = lse * 1.4426950408889634f;
            ds = p.scale * acc;
        }
        p.lse2[row] = l2;
        p.dsc[row] = ds;
    }
}

// One thread per query row: reads its row from the d / 4 planes (a warp reads 512
// contiguous bytes per plane), all of them before the first store, and writes it contiguously.
template <typename GradT, int D>
__global__ void __launch_bounds__(128) fa_bwd_dq_kernel(const BwdDqParams p)
{
    grid_dependency_wait();  // the accumulator is complete once the tensor-core kernel has finished
    grid_launch_dependents();
    const long long row = static_cast<long long>(blockIdx.x) * 128 + threadIdx.x;
    if (row >= static_cast<long long>(p.BH) * p.N) return;
    const int bh = static_cast<int>(row / p.N);
    const int q = static_cast<int>(row - static_cast<long long>(bh) * p.N);
    const int qt = q % kBlockM;  // row within the query tile
    constexpr bool kBulk = dq_bulk(D);
    // plane stride: 128 rows of a tile ([d/4][128][4]) or the 32 rows of a row quarter ([4][d/4][32][4])
    constexpr int kPlane = kBulk ? 32 * 4 : kBlockM * 4;
    const float* __restrict__ src = p.dq_acc + (static_cast<size_t>(bh) * p.Tr + q / kBlockM) * (D * kBlockM) +
                                    (kBulk ? (qt / 32) * (D * 32) + (qt % 32) * 4 : qt * 4);
    GradT* __restrict__ dst = reinterpret_cast<GradT*>(p.dq) + static_cast<size_t>(row) * D;
    float v[D];
#pragma unroll
    for (int e = 0; e < D / 4; ++e) {
        const float4 f = __ldcs(reinterpret_cast<const float4*>(src + static_cast<size_t>(e) * kPlane));
        v[4 * e] = f.x; v[4 * e + 1] = f.y; v[4 * e + 2] = f.z; v[4 * e + 3] = f.w;
    }
#pragma unroll
    for (int c = 0; c < D; c += 16) store_row16<GradT>(dst + c, *reinterpret_cast<const float(*)[16]>(&v[c]));
}

cudaError_t launch_bwd_prep(const BwdPrepParams& p, fa_dtype o_dtype, cudaStream_t st)
{
    const long long threads = static_cast<long long>(p.BH) * p.Tr * kBlockM * (p.d / 8);
    const long long blocks = (threads + kPrepThreads - 1) / kPrepThreads;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (o_dtype == FA_F32) return launch_pdl(fa_bwd_prep_kernel<float>, static_cast<unsigned>(blocks), kPrepThreads, 0, st, p);
    return launch_pdl(fa_bwd_prep_kernel<__nv_bfloat16>, static_cast<unsigned>(blocks), kPrepThreads, 0, st, p);
}

cudaError_t launch_bwd_dq(const BwdDqParams& p, fa_dtype grad_dtype, cudaStream_t st)
{
    const long long rows = static_cast<long long>(p.BH) * p.N;
    const long long blocks = (rows + 127) / 128;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned g = static_cast<unsigned>(blocks);
    const bool f32 = grad_dtype == FA_F32;
    switch (p.d) {
    case 32: return f32 ? launch_pdl(fa_bwd_dq_kernel<float, 32>, g, 128, 0, st, p)
                        : launch_pdl(fa_bwd_dq_kernel<__nv_bfloat16, 32>, g, 128, 0, st, p);
    case 64: return f32 ? launch_pdl(fa_bwd_dq_kernel<float, 64>, g, 128, 0, st, p)
                        : launch_pdl(fa_bwd_dq_kernel<__nv_bfloat16, 64>, g, 128, 0, st, p);
    case 128: return f32 ? launch_pdl(fa_bwd_dq_kernel<float, 128>, g, 128, 0, st, p)
                         : launch_pdl(fa_bwd_dq_kernel<__nv_bfloat16, 128>, g, 128, 0, st, p);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
