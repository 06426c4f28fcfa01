// fa_fwd_kernel.cuh -- exact attention forward for sm_103a.
//
// Algorithm: "flash_lab.py -- FlashAttention, flash-decoding and megakernel in
// numpy", section 3 `flash_fwd`, FlashAttention-2 loop order: each CTA owns one
// tile of 128 query rows and walks the key/value tiles of its head, keeping the
// running row max m and row sum l (section 1, `softmax_online`: the old sum is
// rescaled by exp(m_old - m_new)) and an unnormalised O accumulator on chip.
// O is divided by l once at the end and LSE = m + log l.  With a causal mask
// the walk stops at the first tile lying wholly after the tile's last query
// position (query i sits at position Nk - N + i; "02_flash_forward.py", demo 1).
//
// GB300 mapping (one CTA of 6 warps per 128-row query tile):
//   warp 4      TMA producer: Q once, then K_j / V_j into a 2-stage ring.
//   warp 5      tcgen05 issuer: S_j = Q K_j^T into one of two TMEM score buffers,
//               and O += P_j V_j into a TMEM accumulator; commits signal barriers.
//               S_{j+1} is issued before P_j is ready, so the tensor core
//               computes the next scores while the softmax of this tile runs.
//   warps 0..3  softmax: thread t owns query row t (= TMEM lane t); reads its
//               score row from TMEM, masks, updates m and l in the base-2 domain
//               with a log2(e)-prescaled scale, writes P (bf16) to shared memory
//               in the 128-byte-swizzled K-major layout the MMA reads, and
//               rescales its O row in TMEM when its max grew.  Then the
//               epilogue: O / l and LSE to global memory.
// The running max moves whenever a tile raises it, so the largest P of the
// row is exactly 1 in bf16.  (Keeping a stale max to skip rescales, with P up
// to 2^k, would leave that dominant weight rounded: with values of magnitude
// ~8 the O error then reaches 2e-2, above the 1e-2 the results must meet.)
// A warp rescales its O rows in TMEM only when the max of one of its rows grew.
//
// Every barrier wait is bounded (FwdParams::wait_limit_ns).  A role whose wait
// runs out records FA_ERR_TIMEOUT, raises the CTA's abort flag so the other
// roles stop too, and every role then drains what it has in flight (TMA copies,
// tensor-core operations) before the CTA frees its tensor memory and exits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

constexpr unsigned long long kDrainLimitNs = 1000000000ull;  // 1 s for draining after a failure

template <int D>
struct FwdCfg {
    static_assert(D == 32 || D == 64 || D == 128, "head size");
    static constexpr int kCB = D < 64 ? D : 64;        // elements per column block (swizzle span)
    static constexpr int kNumCB = D / kCB;             // column blocks per row
    static constexpr int kRowBytes = kCB * 2;          // 64 or 128 bytes
    static constexpr uint32_t kLayout = kRowBytes == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int kAtomBytes = 8 * kRowBytes;   // 8-row swizzle atom
    static constexpr int kBlkBytes = kBlockM * kRowBytes;  // one 128-row column block
    static constexpr int kTileBytes = kNumCB * kBlkBytes;  // 128 x D bf16
    static constexpr int kPBlkBytes = kBlockM * 128;       // 128 rows x 64 keys bf16
    static constexpr int kPBytes = 2 * kPBlkBytes;         // P tile: two 64-key column blocks
    static constexpr int kStages = 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffP = kOffV + kStages * kTileBytes;
    static constexpr int kOffBar = kOffP + kPBytes;
    static constexpr int kNumBars = 12;
    static constexpr int kUsedBytes = kOffBar + kNumBars * 8 + 16;
    // At least 120 KB so that only one CTA (holding all 512 TMEM columns) fits per SM.
    static constexpr int kSmemBytes = (kUsedBytes + 1024 > 120 * 1024 ? kUsedBytes + 1024 : 120 * 1024);
    static constexpr int kTmemCols = 512;
    static constexpr int kColS0 = 0;
    static constexpr int kColO = 256;
    static constexpr uint32_t kIdescS = idesc_bf16(kBlockM, kBlockN, false);
    static constexpr uint32_t kIdescO = idesc_bf16(kBlockM, D, true);
};

// barrier slots
enum : int {
    kBarQFull = 0,
    kBarKFull = 1,   // +stage
    kBarVFull = 3,   // +stage
    kBarKVEmpty = 5, // +stage
    kBarSFull = 7,   // +score buffer
    kBarPFull = 9,
    kBarPVDone = 10,
    kBarDrain = 11
};

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

template <int D, bool CAUSAL, typename OutT>
__global__ void __launch_bounds__(192, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p)
{
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kOffBar;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Work item: heaviest query tiles first (under a causal mask the last tile
    // of every head has the most visible keys).
    const int tile_rev = blockIdx.x / p.BH;
    const int bh = blockIdx.x - tile_rev * p.BH;
    const int qt = p.n_qtiles - 1 - tile_rev;
    const int i0 = qt * kBlockM;
    const int br = min(kBlockM, p.N - i0);
    const int off = p.Nk - p.N;  // query i sits at key position off + i
    const int n_kv_all = (p.Nk + kBlockN - 1) / kBlockN;
    int n_kv = n_kv_all;
    if (CAUSAL) {
        const int last_pos = off + i0 + br - 1;  // position of the tile's last query row
        n_kv = last_pos < 0 ? 0 : min(n_kv_all, last_pos / kBlockN + 1);
    }
    const unsigned long long limit = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQFull), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(kBarKFull + s), 1);
            mbar_init(bar(kBarVFull + s), 1);
            mbar_init(bar(kBarKVEmpty + s), 1);
            mbar_init(bar(kBarSFull + s), 1);
        }
        mbar_init(bar(kBarPFull), kBlockM);
        mbar_init(bar(kBarPVDone), 1);
        mbar_init(bar(kBarDrain), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_kv > 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            int last_issued[2] = {-1, -1};
            mbar_arrive_expect_tx(bar(kBarQFull), C::kTileBytes);
#pragma unroll
            for (int cb = 0; cb < C::kNumCB; ++cb)
                tma_load_3d(sbase + C::kOffQ + cb * C::kBlkBytes, &p.tm_q, bar(kBarQFull), cb * C::kCB,
                            i0, bh, pol_q);
            bool ok = true;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j & 1;
                if (j >= 2 && !mbar_wait(bar(kBarKVEmpty + s), ((j >> 1) + 1) & 1, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(kBarKFull + s), C::kTileBytes);
#pragma unroll
                for (int cb = 0; cb < C::kNumCB; ++cb)
                    tma_load_3d(sbase + C::kOffK + s * C::kTileBytes + cb * C::kBlkBytes, &p.tm_k,
                                bar(kBarKFull + s), cb * C::kCB, j * kBlockN, bh, pol_kv);
                mbar_arrive_expect_tx(bar(kBarVFull + s), C::kTileBytes);
#pragma unroll
                for (int cb = 0; cb < C::kNumCB; ++cb)
                    tma_load_3d(sbase + C::kOffV + s * C::kTileBytes + cb * C::kBlkBytes, &p.tm_v,
                                bar(kBarVFull + s), cb * C::kCB, j * kBlockN, bh, pol_kv);
                last_issued[s] = j;
            }
            if (!ok) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            // Every issued copy must have landed before the CTA may exit.
            mbar_wait(bar(kBarQFull), 0, kDrainLimitNs, nullptr);
            for (int s = 0; s < 2; ++s) {
                if (last_issued[s] < 0) continue;
                const uint32_t par = (last_issued[s] >> 1) & 1;
                mbar_wait(bar(kBarKFull + s), par, kDrainLimitNs, nullptr);
                mbar_wait(bar(kBarVFull + s), par, kDrainLimitNs, nullptr);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            auto issue_s = [&](int j) {
                const int s = j & 1;
                const uint32_t d_tmem = tmem + C::kColS0 + 128u * static_cast<uint32_t>(s);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int cb = (kk * 16) / C::kCB;
                    const int within = ((kk * 16) % C::kCB) * 2;
                    const uint64_t a = smem_desc(sbase + C::kOffQ + cb * C::kBlkBytes + within, 16,
                                                 C::kAtomBytes, C::kLayout);
                    const uint64_t b = smem_desc(
                        sbase + C::kOffK + s * C::kTileBytes + cb * C::kBlkBytes + within, 16,
                        C::kAtomBytes, C::kLayout);
                    umma_ss(d_tmem, a, b, C::kIdescS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int j) {
                const int s = j & 1;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    const uint64_t a = smem_desc(sbase + C::kOffP + (kk >> 2) * C::kPBlkBytes + (kk & 3) * 32,
                                                 16, 1024, kSwizzle128B);
                    const uint64_t b = smem_desc(
                        sbase + C::kOffV + s * C::kTileBytes + kk * 16 * C::kRowBytes, C::kBlkBytes,
                        C::kAtomBytes, C::kLayout);
                    umma_ss(tmem + C::kColO, a, b, C::kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = true;
            if (n_kv > 0) {
                ok = mbar_wait(bar(kBarQFull), 0, limit, abort_flag) &&
                     mbar_wait(bar(kBarKFull + 0), 0, limit, abort_flag);
                if (ok) {
                    tc_fence_after_sync();
                    issue_s(0);
                    umma_commit(bar(kBarSFull + 0));
                }
                for (int j = 0; ok && j < n_kv; ++j) {
                    if (j + 1 < n_kv) {
                        // buffer (j+1)&1 last held S_{j-1}, read before P_{j-1} was signalled
                        if (!mbar_wait(bar(kBarKFull + ((j + 1) & 1)), ((j + 1) >> 1) & 1, limit,
                                       abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        issue_s(j + 1);
                        umma_commit(bar(kBarSFull + ((j + 1) & 1)));
                    }
                    if (!mbar_wait(bar(kBarPFull), j & 1, limit, abort_flag) ||
                        !mbar_wait(bar(kBarVFull + (j & 1)), (j >> 1) & 1, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    issue_pv(j);
                    umma_commit(bar(kBarPVDone));
                    umma_commit(bar(kBarKVEmpty + (j & 1)));
                }
            }
            if (!ok) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            // Wait for every tensor-core operation this thread issued.
            umma_commit(bar(kBarDrain));
            mbar_wait(bar(kBarDrain), 0, kDrainLimitNs, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int r = threadIdx.x;  // query row within the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const int qpos = off + i0 + r;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY;  // running max of scale*log2(e)*S over the visible keys
        float l = 0.f;
        bool ok = true;
        const uint32_t p_row = sbase + C::kOffP + static_cast<uint32_t>(r) * 128u;
        const uint32_t swz = static_cast<uint32_t>(r & 7);

        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + sb), (j >> 1) & 1, limit, abort_flag));
            if (!ok) break;
            tc_fence_after_sync();
            float s[kBlockN];
            {
                uint32_t u[32];
#pragma unroll
                for (int c = 0; c < kBlockN / 32; ++c) {
                    tmem_ld32(tmem + lane_base + C::kColS0 + 128u * sb + 32u * c, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(u[i]);
                }
            }
            const int k0 = j * kBlockN;
            const bool need_mask = (k0 + kBlockN > p.Nk) || (CAUSAL && k0 + kBlockN - 1 > off + i0);
            if (need_mask) {
                const int last = CAUSAL ? min(qpos, p.Nk - 1) : p.Nk - 1;  // last visible key
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (k0 + c > last) s[c] = -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int c = 1; c < kBlockN; ++c) mx = fmaxf(mx, s[c]);
            const float mt = mx * sl2;
            const bool grow = mt > m_ref;
            float alpha = 1.f;
            if (grow) {
                alpha = ex2(m_ref - mt);  // 0 when m_ref = -inf
                m_ref = mt;
            }
            const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
            float rs = 0.f;
            uint32_t pk[kBlockN / 2];
#pragma unroll
            for (int c = 0; c < kBlockN; c += 2) {
                const float p0 = ex2(fmaf(s[c], sl2, -m_use));
                const float p1 = ex2(fmaf(s[c + 1], sl2, -m_use));
                rs += p0 + p1;
                pk[c / 2] = pack_bf16x2(p0, p1);
            }
            // P_{j-1} V_{j-1} must have finished before P is overwritten or O rescaled.
            if (j > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarPVDone), (j - 1) & 1, limit, abort_flag));
                if (!ok) break;
                tc_fence_after_sync();
            }
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                const uint32_t addr = p_row + static_cast<uint32_t>(ch >> 3) * C::kPBlkBytes +
                                      ((static_cast<uint32_t>(ch & 7) ^ swz) << 4);
                st_shared_v4(addr, pk[ch * 4 + 0], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
            }
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t u[32];
                    const uint32_t ta = tmem + lane_base + C::kColO + 32u * c;
                    tmem_ld32(ta, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                    tmem_st32(ta, u);
                }
                tmem_st_wait();
            }
            l = l * alpha + rs;
            fence_proxy_async_shared();
            tc_fence_before_sync();
            mbar_arrive(bar(kBarPFull));
        }
        if (ok && n_kv > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarPVDone), (n_kv - 1) & 1, limit, abort_flag));
        }
        if (!ok) {
            record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
        } else {
            tc_fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const size_t row = static_cast<size_t>(bh) * p.N + static_cast<size_t>(i0 + r);
            OutT* orow = reinterpret_cast<OutT*>(p.o) + row * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                if (n_kv > 0) {
                    uint32_t u[32];
                    tmem_ld32(tmem + lane_base + C::kColO + 32u * c, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]) * inv;
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                }
                if (r < br) store_row32<OutT>(orow + 32 * c, v);
            }
            if (p.lse != nullptr && r < br)
                p.lse[row] = l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool CAUSAL, typename OutT>
cudaError_t launch_fwd_t(const FwdParams& p, cudaStream_t st)
{
    using C = FwdCfg<D>;
    auto kern = fa_fwd_kernel<D, CAUSAL, OutT>;
    static bool configured[64] = {};  // the shared-memory attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.n_qtiles);
    kern<<<grid, 192, C::kSmemBytes, st>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const FwdParams& p, bool causal, fa_dtype o_dtype, cudaStream_t st)
{
    if (o_dtype == FA_F32)
        return causal ? launch_fwd_t<D, true, float>(p, st) : launch_fwd_t<D, false, float>(p, st);
    return causal ? launch_fwd_t<D, true, __nv_bfloat16>(p, st) : launch_fwd_t<D, false, __nv_bfloat16>(p, st);
}

}  // namespace fa
