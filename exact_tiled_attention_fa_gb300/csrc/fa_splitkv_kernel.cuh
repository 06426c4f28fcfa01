// fa_splitkv_kernel.cuh -- exact attention over one key split of one query tile, for sm_103a.
//
// Algorithm: "flash_lab.py -- FlashAttention, flash-decoding and megakernel in numpy",
// section 4 `split_kv_decode`: the keys are cut into splits; each split computes its own
// normalised output o_s = softmax(q K_s^T) V_s and log-sum-exp lse_s, and the splits are
// merged afterwards (lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s; the merge
// kernel in fa_decode.cu).  Within a split the walk over key tiles is the FlashAttention-2
// loop of section 3 `flash_fwd` (running max m and sum l, O rescaled by exp(m_old - m_new)).
//
// Used for grouped-query decode: the rows of the query tile are the R query heads that share one
// key/value head ("flash_lab.py" section 4 packs a group's query heads as the rows of q;
// `decode_attention_time` method "fd" pads them to a tensor-core tile), each sequence with its
// own cached length (VARLEN).  The kernel also carries a causal form for a tile of 128 queries
// of one head (query i at position Nk - N + i), which the prefill with few query tiles used
// before it moved to the forward kernel's split mode; only the decode form is instantiated.
//
// GB300 mapping: one CTA per (split, query tile, group); six warps.
//   warps 0-3  softmax: thread t owns row t of the tile (TMEM lane t).
//   warp 4     TMA producer: the query tile once, K_j and V_j into a ring.
//   warp 5     tcgen05 issuer: S = Q K_j^T (SS) into TMEM; O += P V_j (P from TMEM).
// Tensor memory: S (128 fp32 columns), O (d columns), P (64 columns of packed bf16).
// S(j+1) is issued as soon as the softmax has read S(j).
// Cache rows past a sequence's length may hold anything (the tests fill them with NaN):
// their scores are masked, and before P V_j of the last tile the softmax zeroes those V rows
// in shared memory, so 0 * NaN never reaches the accumulator.
// Every barrier wait is bounded; a wait that runs out records FA_ERR_TIMEOUT, the roles
// drain what they have in flight and the CTA returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"
#include "ptx.cuh"

namespace fa {

constexpr int kSkThreads = 192;
constexpr int kSkWarpProducer = 4;
constexpr int kSkWarpMma = 5;

enum : int {
    kSbQFull = 0,
    kSbSFull = 1,
    kSbSFree = 2,
    kSbPFull = 3,
    kSbPVDone = 4,
    kSbOReady = 5,
    kSbDrain = 6,
    kSbKVFull = 8,   // + stage
    kSbKVEmpty = 12, // + stage
    kSbCount = 16
};

template <int D>
struct SkCfg {
    static_assert(D == 32 || D == 64 || D == 128, "head size");
    static constexpr int kCB = D < 64 ? D : 64;
    static constexpr int kNumCB = D / kCB;
    static constexpr int kRowBytes = kCB * 2;
    static constexpr uint32_t kLayout = kRowBytes == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int kAtomBytes = 8 * kRowBytes;
    static constexpr int kBlkBytes = kBlockM * kRowBytes;
    static constexpr int kTileBytes = kNumCB * kBlkBytes;  // 128 x D bf16
    static constexpr int kStages = D == 128 ? 2 : (D == 64 ? 3 : 4);
    static_assert(kStages <= 4, "barrier slots");
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kTileBytes;                         // + stage * kTileBytes
    static constexpr int kOffV = kOffK + kStages * kTileBytes;       // + stage * kTileBytes
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    static constexpr int kUsedBytes = kOffBar + kSbCount * 8 + 16;
    static constexpr int kSmemBytes = kUsedBytes + 1024;             // + alignment slack
    static constexpr int kTmemCols = D == 128 ? 512 : 256;
    static constexpr uint32_t kColS = 0, kColO = 128, kColP = 128 + D;
    static constexpr uint32_t kIdescS = idesc_bf16(kBlockM, kBlockN, false);
    static constexpr uint32_t kIdescO = idesc_bf16(kBlockM, D, true);
};

template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kSkThreads, 1) fa_splitkv_kernel(const __grid_constant__ SplitParams p)
{
    grid_dependency_wait();    // launched as a programmatic dependent of the previous kernel
    grid_launch_dependents();  // the merge that follows may begin launching (it waits for this grid)
    using C = SkCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t sk_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sk_smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + kSbCount * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long limit = p.wait_limit_ns;

    // ---- work item: split s, query tile qt, group g
    const int s = blockIdx.x;
    const int qt = blockIdx.y;
    const int g = blockIdx.z;
    const int row0 = qt * kBlockM;                         // first row of the tile within the group
    const int rows = min(kBlockM, p.rows_per_group - row0);
    int len = p.Nk;                                        // keys that exist for this group
    if (VARLEN) {
        const int b = g / p.groups_per_batch;
        len = p.seqlens[b];
        if (len < 0 || len > p.Nk) {
            if (threadIdx.x == 0) atomicCAS(p.status, 0, FA_ERR_INVALID_ARG);
            len = len < 0 ? 0 : p.Nk;
        }
    }
    const int kl = s * p.chunk;                            // the split's keys: [kl, kh)
    int kh = min(len, kl + p.chunk);
    if (CAUSAL) kh = min(kh, p.causal_off + row0 + rows);  // the tile's last row sees keys < this
    const int j_begin = kl / kBlockN;
    const int nt = kh > kl ? (kh - kl + kBlockN - 1) / kBlockN : 0;

    if (threadIdx.x == 0) {
        mbar_init(bar(kSbQFull), 1);
        mbar_init(bar(kSbSFull), 1);
        mbar_init(bar(kSbSFree), kBlockM);
        mbar_init(bar(kSbPFull), kBlockM);
        mbar_init(bar(kSbPVDone), 1);
        mbar_init(bar(kSbOReady), 1);
        mbar_init(bar(kSbDrain), 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(bar(kSbKVFull + i), 1);
            mbar_init(bar(kSbKVEmpty + i), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kSkWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == kSkWarpProducer) {
        // ============================================================ producer
        if (lane == 0 && nt > 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
            const uint64_t pol = policy_evict_last();  // K/V of a group are read by each of its query tiles
            mbar_arrive_expect_tx(bar(kSbQFull), C::kTileBytes);
#pragma unroll
            for (int cb = 0; cb < C::kNumCB; ++cb)
                tma_load_3d(sbase + C::kOffQ + cb * C::kBlkBytes, &p.tm_q, bar(kSbQFull), cb * C::kCB, row0, g, pol);
            int issued = 0;
            bool ok = true;
            for (int t = 0; t < nt; ++t) {
                const int st = t % S;
                if (t >= S && !mbar_wait(bar(kSbKVEmpty + st), static_cast<uint32_t>(t / S - 1) & 1, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                const int k0 = (j_begin + t) * kBlockN;
                mbar_arrive_expect_tx(bar(kSbKVFull + st), 2 * C::kTileBytes);
#pragma unroll
                for (int cb = 0; cb < C::kNumCB; ++cb) {
                    tma_load_3d(sbase + C::kOffK + st * C::kTileBytes + cb * C::kBlkBytes, &p.tm_k, bar(kSbKVFull + st),
                                cb * C::kCB, k0, g, pol);
                    tma_load_3d(sbase + C::kOffV + st * C::kTileBytes + cb * C::kBlkBytes, &p.tm_v, bar(kSbKVFull + st),
                                cb * C::kCB, k0, g, pol);
                }
                ++issued;
            }
            if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            mbar_wait(bar(kSbQFull), 0, kDrainLimitNs, nullptr);
            for (int t = issued - S < 0 ? 0 : issued - S; t < issued; ++t)
                mbar_wait(bar(kSbKVFull + t % S), static_cast<uint32_t>(t / S) & 1, kDrainLimitNs, nullptr);
        }
    } else if (warp == kSkWarpMma) {
        // ============================================================ MMA issuer
        if (lane == 0 && nt > 0) {
            bool ok = true;
            auto wait = [&](int b, int parity) -> bool {
                ok = ok && mbar_wait(bar(b), static_cast<uint32_t>(parity) & 1, limit, abort_flag);
                return ok;
            };
            auto issue_s = [&](int st) {
                const uint64_t a0 = smem_desc(sbase + C::kOffQ, 16, C::kAtomBytes, C::kLayout);
                const uint64_t b0 = smem_desc(sbase + C::kOffK + st * C::kTileBytes, 16, C::kAtomBytes, C::kLayout);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = ((kk * 16) / C::kCB * C::kBlkBytes + ((kk * 16) % C::kCB) * 2) >> 4;
                    umma_ss(tmem + C::kColS, a0 + o, b0 + o, C::kIdescS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int st, bool accumulate) {
                const uint64_t b0 = smem_desc(sbase + C::kOffV + st * C::kTileBytes, C::kBlkBytes, C::kAtomBytes, C::kLayout);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    umma_ts(tmem + C::kColO, tmem + C::kColP + 8u * kk, b0 + ((kk * 16 * C::kRowBytes) >> 4), C::kIdescO,
                            (accumulate || kk > 0) ? 1u : 0u);
            };
            if (wait(kSbQFull, 0) && wait(kSbKVFull, 0)) {
                tc_fence_after_sync();
                issue_s(0);
                umma_commit(bar(kSbSFull));
            }
            for (int t = 0; ok && t < nt; ++t) {
                const int st = t % S;
                if (t + 1 < nt) {  // S(t+1) as soon as the softmax has read S(t)
                    const int sn = (t + 1) % S;
                    if (!wait(kSbKVFull + sn, (t + 1) / S) || !wait(kSbSFree, t)) break;
                    tc_fence_after_sync();
                    issue_s(sn);
                    umma_commit(bar(kSbSFull));
                }
                if (!wait(kSbPFull, t)) break;
                tc_fence_after_sync();
                issue_pv(st, t > 0);
                umma_commit(bar(kSbPVDone));
                umma_commit(bar(kSbKVEmpty + st));
            }
            umma_commit(bar(kSbOReady));
            if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            umma_commit(bar(kSbDrain));
            mbar_wait(bar(kSbDrain), 0, kDrainLimitNs, nullptr);
        }
    } else {
        // ============================================================ softmax + epilogue
        const int r = threadIdx.x;  // row of the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t t_s = tmem + lane_base + C::kColS;
        const uint32_t t_o = tmem + lane_base + C::kColO;
        const uint32_t t_p = tmem + lane_base + C::kColP;
        const float sl2 = p.scale_log2;
        const int qpos = p.causal_off + row0 + r;  // position of this row's query (causal)
        const int last = CAUSAL ? min(qpos, kh - 1) : kh - 1;  // last key this row sees in the split
        float m_run = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t < nt; ++t) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kSbSFull), t & 1, limit, abort_flag));
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t u[kBlockN];
            float mq[4];
            tmem_ld32_max(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&u[0]), mq[0]);
            tmem_ld32_max(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]), mq[1]);
            tmem_ld32_max(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&u[64]), mq[2]);
            tmem_ld32_max(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&u[96]), mq[3]);
            tmem_ld_wait();
            tc_fence_before_sync();
            mbar_arrive(bar(kSbSFree));
            float sv[kBlockN];
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) sv[c] = __uint_as_float(u[c]);
            const int k0 = (j_begin + t) * kBlockN;
            if (k0 + kBlockN - 1 > (CAUSAL ? min(p.causal_off + row0, kh - 1) : kh - 1)) {
                // keys past the split, past the sequence or after the row's position: -inf (this
                // also drops the scores of rows that were never loaded or hold padding)
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (k0 + c > last) sv[c] = -INFINITY;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float a = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 32; ++c) a = fmaxf(a, sv[32 * q4 + c]);
                    mq[q4] = a;
                }
            }
            const float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * sl2;
            const bool grow = mt > m_run;
            float alpha = 1.f;
            if (grow) {
                alpha = ex2(m_run - mt);  // 0 when m_run = -inf
                m_run = mt;
            }
            const float m_use = m_run == -INFINITY ? 0.f : m_run;
            // packed two-wide scale-and-subtract and four running pairs for the row sum
            const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-m_use, -m_use);
            float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            uint32_t pk[kBlockN / 2];
#pragma unroll
            for (int c = 0; c < kBlockN; c += 8) {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float2 x = __ffma2_rn(make_float2(sv[c + 2 * h], sv[c + 2 * h + 1]), sl2x2, negm);
                    const float2 e = make_float2(ex2(x.x), ex2(x.y));
                    rs2[h] = __fadd2_rn(rs2[h], e);
                    pk[c / 2 + h] = pack_bf16x2(e.x, e.y);
                }
            }
            const float rs = ((rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y)) + ((rs2[2].x + rs2[2].y) + (rs2[3].x + rs2[3].y));
            // O and the P columns are free once P(t-1) V_{t-1} has completed
            if (t > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kSbPVDone), (t - 1) & 1, limit, abort_flag));
                if (!ok) break;
                tc_fence_after_sync();
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t oc[32];
                        tmem_ld32(t_o + 32u * c, oc);
                        tmem_ld_wait();
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 v = __fmul2_rn(make_float2(__uint_as_float(oc[e]), __uint_as_float(oc[e + 1])), a2);
                            oc[e] = __float_as_uint(v.x);
                            oc[e + 1] = __float_as_uint(v.y);
                        }
                        tmem_st32(t_o + 32u * c, oc);
                    }
                }
            }
            if (VARLEN && k0 + kBlockN > len) {
                // V rows past the sequence may hold anything: zero them before P V_t reads them
                // (their P is 0, but 0 * NaN would poison O).  Row r of each 128-row column
                // block is one 128-byte (or 64-byte) line whatever the swizzle.
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kSbKVFull + t % S), static_cast<uint32_t>(t / S) & 1, limit,
                                                       abort_flag));
                if (!ok) break;
                if (k0 + r >= len) {
                    const uint32_t vrow = sbase + C::kOffV + (t % S) * C::kTileBytes + r * C::kRowBytes;
#pragma unroll
                    for (int cb = 0; cb < C::kNumCB; ++cb)
#pragma unroll
                        for (int c16 = 0; c16 < C::kRowBytes; c16 += 16)
                            st_shared_v4(vrow + cb * C::kBlkBytes + c16, 0u, 0u, 0u, 0u);
                }
                fence_proxy_async_shared();
            }
            tmem_st32(t_p + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st32(t_p + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(bar(kSbPFull));
            l = l * alpha + rs;
        }
        if (ok && nt > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kSbOReady), 0, limit, abort_flag));
            if (ok) tc_fence_after_sync();
        }
        if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
        // epilogue: the split's normalised output and log-sum-exp for this row (o = 0, lse = -inf
        // when the row sees no key of the split).  The TMEM loads are warp-collective
        // (.sync.aligned): every lane of the warp issues them, only rows of the tile store.
        if (ok) {  // uniform across the warp (from __all_sync)
            const bool valid = r < rows;
            const size_t slot =
                (static_cast<size_t>(g) * p.rows_per_group + row0 + (valid ? r : 0)) * p.n_splits + s;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float* orow = p.o_part + slot * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                if (nt > 0) {
                    uint32_t o[32];
                    tmem_ld32(t_o + 32u * c, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv;
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0.f;
                }
                if (valid) store_row32<float>(orow + 32 * c, v);
            }
            if (valid) p.lse_part[slot] = l > 0.f ? (m_run + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kSkWarpMma) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool CAUSAL, bool VARLEN>
cudaError_t launch_splitkv_t(const SplitParams& p, cudaStream_t st)
{
    using C = SkCfg<D>;
    auto kern = fa_splitkv_kernel<D, CAUSAL, VARLEN>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    dim3 grid(p.n_splits, p.n_qtiles, p.n_groups);
    return launch_pdl(kern, grid, kSkThreads, C::kSmemBytes, st, p);
}

template <int D>
cudaError_t launch_splitkv_d(const SplitParams& p, bool causal, bool varlen, cudaStream_t st)
{
    if (!varlen || causal) return cudaErrorInvalidValue;  // grouped-query decode only
    return launch_splitkv_t<D, false, true>(p, st);
}

}  // namespace fa
