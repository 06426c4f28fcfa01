// fa_decode.cu -- split-KV single-query decode and the log-sum-exp combine.
//
// Algorithm: "flash_lab.py -- FlashAttention, flash-decoding and megakernel in
// numpy", section 4 `split_kv_decode`.  With one query per (b, h) a query-tiled
// forward would leave most of the GPU idle, so the keys are cut into splits;
// each split computes its own normalised output o_s and log-sum-exp lse_s, and
// a second kernel merges them (lse = log sum_s exp(lse_s),
// o = sum_s exp(lse_s - lse) o_s -- the lse form of section 1 `merge_states`).
//
// The split kernel is bound by HBM bandwidth (R FMAs per key element for R query
// heads sharing a key/value head), so it uses no tensor core: every lane streams 16-byte slices of key rows with
// read-only, L1-bypassing loads, D/8 lanes cooperate on one key, eight loads of
// K and eight of V are in flight per lane before any arithmetic, and the
// softmax is online per warp in the base-2 domain.  Partial states go to
// per-split slots (no atomics), so the result is deterministic.
#include <cuda_bf16.h>

#include <cstdint>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kDecWarps = 4;
constexpr int kDecSteps = 8;  // 16-byte loads of K (and of V) in flight per lane

__device__ __forceinline__ int clamp_len(int n, int hi, int* status)
{
    if (n < 0 || n > hi) {
        atomicCAS(status, 0, FA_ERR_INVALID_ARG);
        n = n < 0 ? 0 : hi;
    }
    return n;
}

__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <int D, int R>
struct DecCfg {
    static constexpr int kLanesPerKey = D / 8;                    // 8 bf16 (16 B) per lane
    static constexpr int kKeysPerStep = 32 / kLanesPerKey;        // keys one warp-wide load covers
    // 16-byte loads of K (and of V) in flight per lane: fewer as the packed query rows take registers
    static constexpr int kSteps = R <= 2 ? kDecSteps : (R == 4 ? 4 : 2);
    static constexpr int kKeysPerIter = kSteps * kKeysPerStep;    // keys per warp per iteration
};

template <typename OutT>
__device__ __forceinline__ void store_out(OutT* o, size_t i, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* o, size_t i, float v)
{
    o[i] = v;
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* o, size_t i, float v)
{
    o[i] = __float2bfloat16_rn(v);
}

// Eight 16-byte global loads in one statement: all 32 results are defined together, so the
// eight requests are issued back to back and are in flight at once.
#define FA_LD_V4X8(OP)                                                                                            \
    asm volatile(OP " {%0, %1, %2, %3}, [%32];\n\t" OP " {%4, %5, %6, %7}, [%33];\n\t" OP                     \
                    " {%8, %9, %10, %11}, [%34];\n\t" OP " {%12, %13, %14, %15}, [%35];\n\t" OP                 \
                    " {%16, %17, %18, %19}, [%36];\n\t" OP " {%20, %21, %22, %23}, [%37];\n\t" OP               \
                    " {%24, %25, %26, %27}, [%38];\n\t" OP " {%28, %29, %30, %31}, [%39];"                      \
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),         \
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),      \
                   "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),   \
                   "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),   \
                   "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])                                           \
                 : "l"(p[0]), "l"(p[1]), "l"(p[2]), "l"(p[3]), "l"(p[4]), "l"(p[5]), "l"(p[6]), "l"(p[7]))

// kL2: read at L2 (`ld.global.cg`: partial states that other CTAs of the running kernel wrote);
// otherwise through the non-coherent path without L1 allocation (written before the kernel).
template <bool kL2>
__device__ __forceinline__ void ld_v4x8(const void* const (&p)[8], uint32_t (&r)[32])
{
    if constexpr (kL2)
        FA_LD_V4X8("ld.global.cg.v4.u32");
    else
        FA_LD_V4X8("ld.global.nc.L1::no_allocate.v4.u32");
}
#undef FA_LD_V4X8

template <bool kL2>
__device__ __forceinline__ float ld_part(const float* p)
{
    if constexpr (kL2)
        return __ldcg(p);
    else
        return __ldg(p);
}

// Log-sum-exp combine of one row's first n_valid partial states by one warp ("flash_lab.py"
// section 1 `merge_states`: lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s).
// store_o(c, value) receives columns c < dv (lane l: VEC * (l + 32 i) + e, i < IT, with
// IT * 32 * VEC >= dv) and store_lse(L) the row's lse from lane 0; with every part empty
// (lse = -inf) the row is 0 and its lse -inf.  Empty parts are never read.  The parts are
// added in increasing order, one FMA per part and column, but the loads of U parts are issued
// together (VEC = 4: eight float4 loads by one statement), so a row pays about one memory
// latency per U parts rather than one per part.  (The empty row leaves through its own stores:
// with the two exits joined, the compiler interleaved the loads with the FMAs, 40 -> 32
// registers, and a 256-part merge took 41 us instead of 27.)
template <int VEC, int IT, bool kL2, typename StoreO, typename StoreL>
__device__ __forceinline__ void merge_row(const float* lse_row, long long lse_stride, const float* o_row,
                                          long long o_stride, int n_valid, int dv, int lane, StoreO store_o,
                                          StoreL store_lse)
{
    constexpr int U = IT >= 8 ? 1 : 8 / IT;
    float M = -INFINITY;
    for (int s = lane; s < n_valid; s += 32) M = fmaxf(M, ld_part<kL2>(lse_row + s * lse_stride));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M == -INFINITY) {  // every part empty: O = 0, LSE = -inf
        for (int c = lane; c < dv; c += 32) store_o(c, 0.f);
        if (lane == 0) store_lse(-INFINITY);
        return;
    }
    float sum = 0.f;
    for (int s = lane; s < n_valid; s += 32) {
        const float x = ld_part<kL2>(lse_row + s * lse_stride);
        if (x != -INFINITY) sum += ex2((x - M) * kLog2e);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float L = M + log2f(sum) * kLn2;

    float acc[IT][VEC];
#pragma unroll
    for (int i = 0; i < IT; ++i)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[i][e] = 0.f;
    for (int base = 0; base < n_valid; base += 32) {
        // lane l weighs part base + l; the warp walks the non-empty ones in order
        const int s = base + lane;
        const float x = s < n_valid ? ld_part<kL2>(lse_row + s * lse_stride) : -INFINITY;
        const float w_lane = x == -INFINITY ? 0.f : ex2((x - L) * kLog2e);
        unsigned live = __ballot_sync(0xffffffffu, x != -INFINITY);
        while (live != 0u) {
            // U parts per batch; slots past the last live part re-read the batch's first part
            // (finite: it was written) with weight 0, so every load is unconditional and in flight
            // together, and fmaf(0, v, acc) leaves acc as it was
            const int j0 = __ffs(live) - 1;
            float w[U];
            const float* op[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = live != 0u ? __ffs(live) - 1 : j0;
                const float wj = __shfl_sync(0xffffffffu, w_lane, j);
                w[u] = live != 0u ? wj : 0.f;
                op[u] = o_row + static_cast<long long>(base + j) * o_stride;
                live &= live - 1u;
            }
            if constexpr (VEC == 4) {
                static_assert(U * IT == 8, "eight loads per batch");
                const void* a[8];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int i = 0; i < IT; ++i) {
                        const int c = 4 * (lane + 32 * i);
                        a[u * IT + i] = op[u] + (c < dv ? c : 0);  // columns past dv: read, never stored
                    }
                uint32_t v[32];
                ld_v4x8<kL2>(a, v);
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int i = 0; i < IT; ++i)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int k = (u * IT + i) * 4 + e;
                            acc[i][e] = fmaf(w[u], __uint_as_float(v[k]), acc[i][e]);
                        }
            } else {
                static_assert(VEC == 1, "float or float4 columns");
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int i = 0; i < IT; ++i) {
                        const int c = lane + 32 * i;
                        acc[i][0] = fmaf(w[u], ld_part<kL2>(op[u] + (c < dv ? c : 0)), acc[i][0]);
                    }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int c = VEC * (lane + 32 * i);
        if (c < dv) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) store_o(c + e, acc[i][e]);
        }
    }
    if (lane == 0) store_lse(L);
}

// One CTA per (split, KV head g, sequence b).  The R query heads g*R .. g*R+R-1 share the
// KV head ("flash_lab.py" section 4: the query heads of a GQA group are packed as the rows
// of q), so each K/V element is read once and used R times.  R = 1 is plain multi-head
// attention.  Writes o_part / lse_part of a non-empty split for each of the R heads.
// o[i] = v in the output dtype.
__device__ __forceinline__ void store_row_value(const DecodeParams& p, size_t i, float v)
{
    if (p.o_dtype == FA_F32)
        reinterpret_cast<float*>(p.o)[i] = v;
    else
        reinterpret_cast<__nv_bfloat16*>(p.o)[i] = __float2bfloat16_rn(v);
}

template <int D, int R, bool FUSED>
__global__ void __launch_bounds__(kDecWarps * 32) fa_decode_split_kernel(const DecodeParams p)
{
    grid_dependency_wait();    // launched as a programmatic dependent of the previous kernel
    grid_launch_dependents();  // the merge that follows may begin launching (it waits for this grid)
    using C = DecCfg<D, R>;
    constexpr int S = C::kSteps;
    const int s = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int n = clamp_len(p.seqlens[b], p.Nk_max, p.status);
    const int k0 = s * p.chunk;
    const size_t bkv = static_cast<size_t>(b) * p.Hkv + g;
    const size_t bq0 = static_cast<size_t>(b) * p.H + static_cast<size_t>(g) * R;  // first query head
    if (k0 >= n) {  // empty split: nothing to write, the combine skips it
        if (FUSED && n == 0 && s == 0) {
            // no split has a key: with the combine fused, split 0 writes O = 0, LSE = -inf
            for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
                const int r = idx / D;
                store_row_value(p, (bq0 + r) * D + (idx - r * D), 0.f);
                if (idx - r * D == 0 && p.lse != nullptr) p.lse[bq0 + r] = -INFINITY;
            }
        }
        return;
    }
    const int k1 = min(n, k0 + p.chunk);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int grp = lane / C::kLanesPerKey;  // which key of a step this lane serves
    const int sub = lane % C::kLanesPerKey;  // which 8-element slice of the row

    float q[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        unpack8(*reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + (bq0 + r) * D + sub * 8),
                q[r]);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[r][i] *= p.scale_log2;  // scores come out in the base-2 domain
    }

    const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(p.k) + bkv * p.Nk_max * D + sub * 8;
    const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(p.v) + bkv * p.Nk_max * D + sub * 8;

    float m[R], l[R], acc[R][8];  // per packed row: running max (warp-uniform), this lane group's sum and output
#pragma unroll
    for (int r = 0; r < R; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[r][i] = 0.f;
    }

    for (int base = k0 + warp * C::kKeysPerIter; base < k1; base += kDecWarps * C::kKeysPerIter) {
        uint4 kr[S], vr[S];
#pragma unroll
        for (int t = 0; t < S; ++t) {
            const int key = base + t * C::kKeysPerStep + grp;
            if (key < k1) {
                kr[t] = ld_stream_v4(kb + static_cast<size_t>(key) * D);
                vr[t] = ld_stream_v4(vb + static_cast<size_t>(key) * D);
            } else {
                kr[t] = make_uint4(0, 0, 0, 0);
                vr[t] = make_uint4(0, 0, 0, 0);
            }
        }
        float sc[S][R];
#pragma unroll
        for (int t = 0; t < S; ++t) {
            float kf[8];
            unpack8(kr[t], kf);
            const int key = base + t * C::kKeysPerStep + grp;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float x = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) x = fmaf(q[r][i], kf[i], x);
#pragma unroll
                for (int o = C::kLanesPerKey / 2; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                sc[t][r] = key < k1 ? x : -INFINITY;
            }
        }
        float m_new[R], alpha[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float bm = sc[0][r];
#pragma unroll
            for (int t = 1; t < S; ++t) bm = fmaxf(bm, sc[t][r]);
#pragma unroll
            for (int o = C::kLanesPerKey; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
            // key `base` (group 0, step 0) is always visible, so bm is finite
            m_new[r] = fmaxf(m[r], bm);
            alpha[r] = ex2(m[r] - m_new[r]);  // 0 on the first block (m = -inf)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[r][i] *= alpha[r];
            l[r] *= alpha[r];
        }
#pragma unroll
        for (int t = 0; t < S; ++t) {
            float vf[8];
            unpack8(vr[t], vf);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float pt = ex2(sc[t][r] - m_new[r]);  // 0 for keys past the split
                l[r] += pt;
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[r][i] = fmaf(pt, vf[i], acc[r][i]);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) m[r] = m_new[r];
    }
    // Sum the lane groups of the warp (they share m).
#pragma unroll
    for (int o = C::kLanesPerKey; o < 32; o <<= 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            l[r] += __shfl_xor_sync(0xffffffffu, l[r], o);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[r][i] += __shfl_xor_sync(0xffffffffu, acc[r][i], o);
        }
    }
    // Merge the warps (each with its own max) through shared memory.
    __shared__ float sm_m[kDecWarps][R], sm_l[kDecWarps][R];
    __shared__ float sm_acc[kDecWarps][R][D];
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            sm_m[warp][r] = m[r];
            sm_l[warp][r] = l[r];
        }
    }
    if (grp == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) sm_acc[warp][r][sub * 8 + i] = acc[r][i];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < R * D; idx += kDecWarps * 32) {
        const int r = idx / D;
        const int c = idx - r * D;
        float M = sm_m[0][r];
#pragma unroll
        for (int w = 1; w < kDecWarps; ++w) M = fmaxf(M, sm_m[w][r]);
        float L = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            const float f = sm_m[w][r] == -INFINITY ? 0.f : ex2(sm_m[w][r] - M);
            L += sm_l[w][r] * f;
            o = fmaf(sm_acc[w][r][c], f, o);
        }
        const size_t slot = (bq0 + r) * p.n_splits + s;
        p.o_part[slot * D + c] = o / L;
        if (c == 0) p.lse_part[slot] = (M + log2f(L)) * kLn2;
    }
    if constexpr (!FUSED) return;
    // ---- fused combine: the last split CTA of this (b, key/value head) to finish merges the
    // R rows ("flash_lab.py" section 4: lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s).
    __threadfence();  // this CTA's partials are visible device-wide before it is counted
    __syncthreads();
    __shared__ int is_last;
    const int n_valid = min(p.n_splits, (n + p.chunk - 1) / p.chunk);
    if (threadIdx.x == 0) {
        const unsigned int prev = atomicAdd(&p.counters[bkv], 1u);
        is_last = prev == static_cast<unsigned int>(n_valid - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    if (warp < R) {  // warp r merges query row r (merge_row, partials read at L2)
        const size_t row = bq0 + warp;
        merge_row<4, 1, true>(
            p.lse_part + row * p.n_splits, 1, p.o_part + row * p.n_splits * D, D, n_valid, D, lane,
            [o = p.o, f32 = p.o_dtype == FA_F32, row](int c, float v) {
                if (f32)
                    reinterpret_cast<float*>(o)[row * D + c] = v;
                else
                    reinterpret_cast<__nv_bfloat16*>(o)[row * D + c] = __float2bfloat16_rn(v);
            },
            [lse = p.lse, row](float L) {
                if (lse != nullptr) lse[row] = L;
            });
    }
    if (threadIdx.x == 0) p.counters[bkv] = 0u;  // ready for the next call
}

// One warp per row: combine the row's valid parts (merge_row).
template <typename OutT, int VEC, int IT>
__global__ void __launch_bounds__(128) fa_merge_kernel(const MergeParams p)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    if (row >= p.rows) return;
    int n_valid = p.n_parts;
    if (p.seqlens != nullptr) {
        const int n = clamp_len(p.seqlens[row / p.H], p.Nk_max, p.status);
        n_valid = min(p.n_parts, (n + p.chunk - 1) / p.chunk);
    }
    OutT* out = reinterpret_cast<OutT*>(p.o) + static_cast<size_t>(row) * p.dv;
    float* lse = p.lse;
    grid_dependency_wait();  // the parts are written by the split kernel launched before this one
    grid_launch_dependents();
    merge_row<VEC, IT, false>(
        p.lse_parts + static_cast<size_t>(row) * p.lse_row_stride, p.lse_part_stride,
        p.o_parts + static_cast<size_t>(row) * p.o_row_stride, p.o_part_stride, n_valid, p.dv, lane,
        [out](int c, float v) { store_out<OutT>(out, c, v); },
        [lse, row](float L) {
            if (lse != nullptr) lse[row] = L;
        });
}

template <typename OutT>
cudaError_t launch_merge_t(const MergeParams& p, cudaStream_t st)
{
    // Launched with programmatic stream serialization: the merge's CTAs may be scheduled while
    // the split kernel's last CTAs still run, and wait in-kernel for its completion, so the
    // launch latency between the two kernels is hidden.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((p.rows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // float4 loads when every part row starts on 16 bytes (dv <= 512)
    const bool vec4 = p.dv % 4 == 0 && p.o_part_stride % 4 == 0 && p.o_row_stride % 4 == 0 &&
                      (reinterpret_cast<uintptr_t>(p.o_parts) & 15u) == 0;
    if (!vec4) return cudaLaunchKernelEx(&cfg, fa_merge_kernel<OutT, 1, 16>, p);
    if (p.dv <= 128) return cudaLaunchKernelEx(&cfg, fa_merge_kernel<OutT, 4, 1>, p);
    if (p.dv <= 256) return cudaLaunchKernelEx(&cfg, fa_merge_kernel<OutT, 4, 2>, p);
    return cudaLaunchKernelEx(&cfg, fa_merge_kernel<OutT, 4, 4>, p);
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams& p, fa_dtype o_dtype, cudaStream_t st)
{
    dim3 grid(p.n_splits, p.Hkv, p.B);
    const int R = p.H / p.Hkv;
    cudaError_t e;
    switch (R) {
    case 1:
        e = p.counters != nullptr ? launch_pdl(fa_decode_split_kernel<D, 1, true>, grid, kDecWarps * 32, 0, st, p)
                                  : launch_pdl(fa_decode_split_kernel<D, 1, false>, grid, kDecWarps * 32, 0, st, p);
        break;
    case 2: e = launch_pdl(fa_decode_split_kernel<D, 2, false>, grid, kDecWarps * 32, 0, st, p); break;
    case 4: e = launch_pdl(fa_decode_split_kernel<D, 4, false>, grid, kDecWarps * 32, 0, st, p); break;
    default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || p.counters != nullptr) return e;  // fused: no second launch
    MergeParams m{};
    m.o_parts = p.o_part;
    m.lse_parts = p.lse_part;
    m.o_part_stride = D;
    m.o_row_stride = static_cast<long long>(p.n_splits) * D;
    m.lse_part_stride = 1;
    m.lse_row_stride = p.n_splits;
    m.n_parts = p.n_splits;
    m.rows = p.B * p.H;
    m.dv = D;
    m.seqlens = p.seqlens;
    m.H = p.H;
    m.chunk = p.chunk;
    m.Nk_max = p.Nk_max;
    m.o = p.o;
    m.lse = p.lse;
    m.status = p.status;
    return launch_merge(m, o_dtype, st);
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, fa_dtype o_dtype, cudaStream_t st)
{
    if (p.dv <= 0 || p.dv > 512) return cudaErrorInvalidValue;
    return o_dtype == FA_F32 ? launch_merge_t<float>(p, st) : launch_merge_t<__nv_bfloat16>(p, st);
}

cudaError_t launch_decode(const DecodeParams& p, int d, fa_dtype o_dtype, cudaStream_t st)
{
    switch (d) {
    case 32: return launch_decode_d<32>(p, o_dtype, st);
    case 64: return launch_decode_d<64>(p, o_dtype, st);
    case 128: return launch_decode_d<128>(p, o_dtype, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
