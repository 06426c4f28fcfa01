// fa_gqa_kernel.cuh -- grouped-query split-KV decode on the tensor core with the product
// transposed, for sm_103a (head size 128, 5 to 32 query heads per key/value head).
//
// Algorithm: "flash_lab.py -- FlashAttention, flash-decoding and megakernel in numpy",
// section 4 `split_kv_decode` with the R query heads of a key/value head packed together (q of
// shape [R, d]; `decode_attention_time` method "fd"): each split of a sequence's cached keys
// gives, for every query head h of the group, the split's normalised output o_s[h] and
// log-sum-exp lse_s[h]; the merge kernel combines the splits.  Within a split the key tiles are
// walked with the online softmax of section 1 (running max m and sum l per query head, the
// accumulator rescaled by exp(m_old - m_new)).
//
// Why transposed.  With R query heads as the rows of a 128-row tile, R of 128 rows are live, and
// the per-tile cost of a row-per-thread softmax (128 exponentials per thread) is paid for R rows
// of work.  Here the tile is turned around: S^T = K_j Q^T puts the 128 keys of the tile on the
// TMEM lanes and the query heads on NQ columns (R padded to a multiple of 16), so thread t (the
// key of lane t) handles R scores per tile; the per-head maximum over the tile's keys is a
// reduction across threads (warp shuffles, then the four warps through shared memory).  The
// thread writes its key's weights P^T into shared memory as the rows of a K-major B operand,
// and the output accumulates transposed, O^T += V_j^T P^T (A = the V tile read MN-major, M = the
// 128 value columns), so TMEM lane t of O^T is value column t and the rescale by exp(m_old -
// m_new) multiplies column h by that head's factor.
//
// One CTA per (split, group = (sequence, key/value head)); six warps:
//   warps 0-3  compute: thread t owns key t of S^T and value column t of O^T.
//   warp 4     TMA producer: the group's NQ query rows once, K_j and V_j into rings of their own.
//   warp 5     tcgen05 issuer: S^T(j+1) as soon as S^T(j) has been read, O^T += V_j^T P^T(j).
// Tensor memory: S^T in columns [0, NQ), O^T in [NQ, 2 NQ).
// Cache rows past a sequence's length may hold anything (the tests fill them with NaN): their
// scores are masked, and before the last tile's product the compute threads zero those V rows
// in shared memory (a weight of 0 times NaN would still be NaN).
// Every barrier wait is bounded; a wait that runs out records FA_ERR_TIMEOUT, the roles drain
// what they have in flight and the CTA returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"
#include "ptx.cuh"

namespace fa {

constexpr int kGqD = 128;  // head size of this kernel

// Warp layout for RH heads per group: one set of four compute warps (thread t = key t / value
// column t) per 8 heads, so a thread handles 8 heads; then the producer and the issuer.  Each set
// reads the same TMEM lanes, its own columns.
template <int RH>
struct GqShape {
    static constexpr int kSets = RH / 8;
    static constexpr int kRHS = RH / kSets;  // heads per set
    static constexpr int kCompute = 4 * kSets;
    static constexpr int kThreads = 32 * (kCompute + 2);
    static constexpr int kWarpProducer = kCompute;
    static constexpr int kWarpMma = kCompute + 1;
};

enum : int {
    kGbQFull = 0,
    kGbSFull = 1,
    kGbSFree = 2,   // the compute threads have read S^T (count 128)
    kGbPFull = 3,   // P^T written and O^T rescaled (count 128)
    kGbPVDone = 4,
    kGbOReady = 5,
    kGbDrain = 6,
    kGbKFull = 8,    // + K stage (up to 3)
    kGbKEmpty = 11,  // + K stage: S^T of the tile has completed
    kGbVFull = 14,   // + V stage (up to 2)
    kGbVEmpty = 16,  // + V stage: the tile's product has completed
    kGbRed = 18,     // + 2 * set + tile parity: a set's four warps' partial maxima (or sums) are in (count 4)
    kGbCount = 26
};

template <int RH>
struct GqCfg {
    static constexpr int NQ = RH < 16 ? 16 : RH;  // MMA columns: the heads padded to 16 or 32
    static_assert(RH == 8 || RH == 16 || RH == 32, "heads per group handled by the compute threads");
    static constexpr int kNQ = NQ;
    // K and V go through separate rings: K_j is free once S^T(j) has completed, early in the tile,
    // V_j only after the product.  With 8 heads two K stages and one V stage keep a CTA at ~109 KB
    // and 96 registers a thread, so two CTAs share an SM and each one's wait for V is covered by
    // the other's work.  16 and 32 heads (two warp sets of compute threads) run once per SM with
    // deeper rings.
    static constexpr int kKStages = RH == 8 ? 2 : 3;
    static constexpr int kVStages = RH == 8 ? 1 : 2;
    static constexpr int kCtasPerSm = RH == 8 ? 2 : 1;
    static constexpr int kRowBytes = 128;                       // one 64-element column block row
    static constexpr int kBlkBytes = kBlockN * kRowBytes;       // 128 rows of one column block
    static constexpr int kTileBytes = 2 * kBlkBytes;            // 128 x 128 bf16 (K or V tile)
    static constexpr int kQBlkBytes = NQ * kRowBytes;           // NQ query rows of one column block
    static constexpr int kQBytes = 2 * kQBlkBytes;
    static constexpr int kPBlkBytes = NQ * kRowBytes;           // P^T: NQ rows x 64 keys
    static constexpr int kPBytes = 2 * kPBlkBytes;              // NQ rows x 128 keys
    static constexpr int kOffK = 0;                              // + stage * kTileBytes
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;  // + stage * kTileBytes
    static constexpr int kOffQ = kOffV + kVStages * kTileBytes;
    static constexpr int kOffP = kOffQ + kQBytes;               // two P^T buffers
    static constexpr int kOffRed = kOffP + 2 * kPBytes;         // [2][sets][4 warps][heads per set] floats
    static constexpr int kOffBar = kOffRed + 2 * 4 * NQ * 4;
    static constexpr int kUsedBytes = kOffBar + kGbCount * 8 + 16;
    static constexpr int kSmemBytes = kUsedBytes + 1024;        // + alignment slack
    static_assert(kSmemBytes * kCtasPerSm <= 228 * 1024 - kCtasPerSm * 1024, "shared memory per SM");
    static constexpr int kTmemCols = 2 * NQ < 32 ? 32 : 2 * NQ;
    static constexpr uint32_t kColS = 0, kColO = NQ;
    // S^T = K Q^T: M = 128 keys, N = NQ heads, both operands K-major
    static constexpr uint32_t kIdescS = idesc_bf16(kBlockN, NQ, false);
    // O^T += V^T P^T: M = 128 value columns (A = V read MN-major), N = NQ heads (B = P^T, K-major)
    static constexpr uint32_t kIdescO = idesc_bf16_a_mn(kGqD, NQ);
};

__device__ __forceinline__ void st_shared_u16(uint32_t addr, unsigned short v)
{
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Grid: (n_splits, key/value heads, sequences).  RH: query heads per group rounded up to a
// multiple of 8 (the heads the compute threads handle); the MMAs use NQ = max(RH, 16) columns.
// The query map is [groups][R][128] with a box of NQ rows (rows past R are zero-filled), the K/V
// maps [groups][Nk][128] with 128-row boxes.
template <int RH>
__global__ void __launch_bounds__(GqShape<RH>::kThreads, GqCfg<RH>::kCtasPerSm)
    fa_gqa_kernel(const __grid_constant__ SplitParams p)
{
    grid_dependency_wait();    // launched as a programmatic dependent of the previous kernel
    grid_launch_dependents();  // the merge that follows may begin launching (it waits for this grid)
    using C = GqCfg<RH>;
    using G = GqShape<RH>;
    constexpr int kGqWarpProducer = G::kWarpProducer;
    constexpr int kGqWarpMma = G::kWarpMma;
    constexpr int SK = C::kKStages;
    constexpr int SV = C::kVStages;
    extern __shared__ uint8_t gq_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gq_smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + kGbCount * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long limit = p.wait_limit_ns;

    // ---- work item: split s of group g = (sequence b, key/value head)
    const int s = blockIdx.x;
    const int b = blockIdx.z;
    const int g = b * p.groups_per_batch + blockIdx.y;
    const int R = p.rows_per_group;
    int len = p.seqlens[b];
    if (len < 0 || len > p.Nk) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, FA_ERR_INVALID_ARG);
        len = len < 0 ? 0 : p.Nk;
    }
    const int kl = s * p.chunk;  // the split's keys: [kl, kh)
    const int kh = min(len, kl + p.chunk);
    const int j_begin = kl / kBlockN;
    const int nt = kh > kl ? (kh - kl + kBlockN - 1) / kBlockN : 0;

    if (threadIdx.x == 0) {
        mbar_init(bar(kGbQFull), 1);
        mbar_init(bar(kGbSFull), 1);
        mbar_init(bar(kGbSFree), 32 * G::kCompute);
        mbar_init(bar(kGbPFull), 32 * G::kCompute);
        mbar_init(bar(kGbPVDone), 1);
        mbar_init(bar(kGbOReady), 1);
        mbar_init(bar(kGbDrain), 1);
        for (int i = 0; i < SK; ++i) {
            mbar_init(bar(kGbKFull + i), 1);
            mbar_init(bar(kGbKEmpty + i), 1);
        }
        for (int i = 0; i < SV; ++i) {
            mbar_init(bar(kGbVFull + i), 1);
            mbar_init(bar(kGbVEmpty + i), 1);
        }
        for (int i = 0; i < 2 * G::kSets; ++i) mbar_init(bar(kGbRed + i), 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kGqWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == kGqWarpProducer) {
        // ============================================================ producer
        if (lane == 0 && nt > 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
            const uint64_t pol = policy_evict_first();  // each K/V tile is read by one CTA only
            mbar_arrive_expect_tx(bar(kGbQFull), C::kQBytes);
            for (int cb = 0; cb < 2; ++cb)
                tma_load_3d(sbase + C::kOffQ + cb * C::kQBlkBytes, &p.tm_q, bar(kGbQFull), cb * 64, 0, g, pol);
            // K runs one tile ahead of V: K_j is released early in tile j (once S^T(j) is done),
            // V_j only after the product of tile j
            int k_issued = 0, v_issued = 0;
            bool ok = true;
            auto load_k = [&](int t) -> bool {
                const int st = t % SK;
                if (t >= SK && !mbar_wait(bar(kGbKEmpty + st), static_cast<uint32_t>(t / SK - 1) & 1, limit, abort_flag))
                    return false;
                mbar_arrive_expect_tx(bar(kGbKFull + st), C::kTileBytes);
                for (int cb = 0; cb < 2; ++cb)
                    tma_load_3d(sbase + C::kOffK + st * C::kTileBytes + cb * C::kBlkBytes, &p.tm_k, bar(kGbKFull + st),
                                cb * 64, (j_begin + t) * kBlockN, g, pol);
                ++k_issued;
                return true;
            };
            auto load_v = [&](int t) -> bool {
                const int st = t % SV;
                if (t >= SV && !mbar_wait(bar(kGbVEmpty + st), static_cast<uint32_t>(t / SV - 1) & 1, limit, abort_flag))
                    return false;
                mbar_arrive_expect_tx(bar(kGbVFull + st), C::kTileBytes);
                for (int cb = 0; cb < 2; ++cb)
                    tma_load_3d(sbase + C::kOffV + st * C::kTileBytes + cb * C::kBlkBytes, &p.tm_v, bar(kGbVFull + st),
                                cb * 64, (j_begin + t) * kBlockN, g, pol);
                ++v_issued;
                return true;
            };
            ok = load_k(0);
            for (int t = 0; ok && t < nt; ++t) {
                if (t + 1 < nt && !load_k(t + 1)) {
                    ok = false;
                    break;
                }
                if (!load_v(t)) {
                    ok = false;
                    break;
                }
            }
            if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            mbar_wait(bar(kGbQFull), 0, kDrainLimitNs, nullptr);
            for (int t = k_issued - SK < 0 ? 0 : k_issued - SK; t < k_issued; ++t)
                mbar_wait(bar(kGbKFull + t % SK), static_cast<uint32_t>(t / SK) & 1, kDrainLimitNs, nullptr);
            for (int t = v_issued - SV < 0 ? 0 : v_issued - SV; t < v_issued; ++t)
                mbar_wait(bar(kGbVFull + t % SV), static_cast<uint32_t>(t / SV) & 1, kDrainLimitNs, nullptr);
        }
    } else if (warp == kGqWarpMma) {
        // ============================================================ MMA issuer
        if (lane == 0 && nt > 0) {
            bool ok = true;
            auto wait = [&](int bb, int parity) -> bool {
                ok = ok && mbar_wait(bar(bb), static_cast<uint32_t>(parity) & 1, limit, abort_flag);
                return ok;
            };
            // S^T = K_j Q^T: A = the K tile (128 keys, K-major), B = the NQ query rows (K-major).
            auto issue_s = [&](int st) {
                const uint64_t a0 = smem_desc(sbase + C::kOffK + st * C::kTileBytes, 16, 1024, kSwizzle128B);
                const uint64_t b0 = smem_desc(sbase + C::kOffQ, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < kGqD / 16; ++kk) {
                    const uint32_t oa = ((kk / 4) * C::kBlkBytes + (kk % 4) * 32) >> 4;
                    const uint32_t ob = ((kk / 4) * C::kQBlkBytes + (kk % 4) * 32) >> 4;
                    umma_ss(tmem + C::kColS, a0 + oa, b0 + ob, C::kIdescS, kk > 0 ? 1u : 0u);
                }
            };
            // O^T += V_j^T P^T: A = the V tile read MN-major (its 128 value columns contiguous per
            // key row; the two 64-column blocks kBlkBytes apart), B = P^T (NQ rows of keys, K-major).
            auto issue_pv = [&](int st, int pbuf, bool accumulate) {
                const uint64_t a0 = smem_desc(sbase + C::kOffV + st * C::kTileBytes, C::kBlkBytes, 1024, kSwizzle128B);
                const uint64_t b0 = smem_desc(sbase + C::kOffP + pbuf * C::kPBytes, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    const uint32_t oa = (kk * 16 * C::kRowBytes) >> 4;
                    const uint32_t ob = ((kk / 4) * C::kPBlkBytes + (kk % 4) * 32) >> 4;
                    umma_ss(tmem + C::kColO, a0 + oa, b0 + ob, C::kIdescO, (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            if (wait(kGbQFull, 0) && wait(kGbKFull, 0)) {
                tc_fence_after_sync();
                issue_s(0);
                umma_commit(bar(kGbSFull));
                umma_commit(bar(kGbKEmpty));  // K_0 is free once S^T(0) has completed
            }
            for (int t = 0; ok && t < nt; ++t) {
                const int sv = t % SV;
                if (t + 1 < nt) {  // S^T(t+1) as soon as the compute threads have read S^T(t)
                    const int sn = (t + 1) % SK;
                    if (!wait(kGbKFull + sn, (t + 1) / SK) || !wait(kGbSFree, t)) break;
                    tc_fence_after_sync();
                    issue_s(sn);
                    umma_commit(bar(kGbSFull));
                    umma_commit(bar(kGbKEmpty + sn));
                }
                if (!wait(kGbVFull + sv, t / SV) || !wait(kGbPFull, t)) break;
                tc_fence_after_sync();
                issue_pv(sv, t & 1, t > 0);
                umma_commit(bar(kGbPVDone));
                umma_commit(bar(kGbVEmpty + sv));
            }
            umma_commit(bar(kGbOReady));
            if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            umma_commit(bar(kGbDrain));
            mbar_wait(bar(kGbDrain), 0, kDrainLimitNs, nullptr);
        }
    } else {
        // ============================================================ compute
        constexpr int RS = G::kRHS;  // heads of this thread's set
        const int set = warp >> 2;
        const int h0 = set * RS;     // first head of the set
        const int wq = warp & 3;     // warp within the set: TMEM lanes 32 wq .. 32 wq + 31
        const int k = threadIdx.x & 127;  // key k of S^T and value column k of O^T (TMEM lane k)
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t t_s = tmem + lane_base + C::kColS + static_cast<uint32_t>(h0);
        const uint32_t t_o = tmem + lane_base + C::kColO + static_cast<uint32_t>(h0);
        float* red = reinterpret_cast<float*>(smem + C::kOffRed);
        const float sl2 = p.scale_log2;
        float m_run[RS], l[RS];  // per head: running max (base 2, scale folded in), this key's share of l
#pragma unroll
        for (int i = 0; i < RS; ++i) {
            m_run[i] = -INFINITY;
            l[i] = 0.f;
        }
        auto ld_cols = [&](uint32_t taddr, uint32_t (&r)[RS]) {
            if constexpr (RS == 8) tmem_ld8(taddr, r);
            else tmem_ld16(taddr, r);
        };
        auto st_cols = [&](uint32_t taddr, const uint32_t (&r)[RS]) {
            if constexpr (RS == 8) tmem_st8(taddr, r);
            else tmem_st16(taddr, r);
        };
        // The set's four warps' values of each head combined through shared memory (use: exchange
        // number, alternating between two buffers and barriers per set).  False if the wait ran out.
        auto exchange = [&](float (&v)[RS], int use, bool is_max) -> bool {
            float* rb = red + ((use & 1) * G::kSets + set) * 4 * RS;
            const int rbar = kGbRed + 2 * set + (use & 1);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < RS; ++i) rb[wq * RS + i] = v[i];
                mbar_arrive(bar(rbar));
            }
            if (!__all_sync(0xffffffffu, mbar_wait(bar(rbar), static_cast<uint32_t>(use >> 1) & 1, limit, abort_flag)))
                return false;
#pragma unroll
            for (int i = 0; i < RS; ++i)
                v[i] = is_max ? fmaxf(fmaxf(rb[i], rb[RS + i]), fmaxf(rb[2 * RS + i], rb[3 * RS + i]))
                              : (rb[i] + rb[RS + i]) + (rb[2 * RS + i] + rb[3 * RS + i]);
            return true;
        };
        bool ok = true;
        for (int t = 0; t < nt; ++t) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kGbSFull), t & 1, limit, abort_flag));
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t u[RS];
            ld_cols(t_s, u);
            tmem_ld_wait();
            tc_fence_before_sync();
            mbar_arrive(bar(kGbSFree));
            const int k0 = (j_begin + t) * kBlockN;
            const bool live = k0 + k < kh;  // keys past the split or the sequence weigh 0
            float sv[RS], mx[RS];
#pragma unroll
            for (int i = 0; i < RS; ++i) {
                sv[i] = live ? __uint_as_float(u[i]) : -INFINITY;
                mx[i] = sv[i];
            }
            // each head's maximum over the tile's 128 keys
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int i = 0; i < RS; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], off));
            ok = exchange(mx, t, true);
            if (!ok) break;
            // new running maxima and rescale factors: the same in every thread of the set
            float alpha[RS];
            bool grew = false;
#pragma unroll
            for (int i = 0; i < RS; ++i) {
                const float mt = mx[i] * sl2;
                alpha[i] = 1.f;
                if (mt > m_run[i]) {
                    alpha[i] = ex2(m_run[i] - mt);  // 0 when m_run = -inf
                    m_run[i] = mt;
                    grew = true;
                }
            }
            // this key's weights: P^T row h, column k of the K-major 128-byte-swizzled B operand
            const uint32_t pb = sbase + C::kOffP + (t & 1) * C::kPBytes + (k >> 6) * C::kPBlkBytes;
            const int e = k & 63;
#pragma unroll
            for (int i = 0; i < RS; ++i) {
                const int h = h0 + i;
                const float mu = m_run[i] == -INFINITY ? 0.f : m_run[i];
                const float pv = ex2(fmaf(sv[i], sl2, -mu));
                l[i] = fmaf(l[i], alpha[i], pv);
                st_shared_u16(pb + h * C::kRowBytes + ((static_cast<uint32_t>((e >> 3) ^ (h & 7))) << 4) + (e & 7) * 2,
                              __bfloat16_as_ushort(__float2bfloat16_rn(pv)));
            }
            if (set == 0 && k0 + kBlockN > len) {
                // V rows past the sequence may hold anything: zero them before the product reads
                // them (their weight is 0, but 0 * NaN would poison O).  Row k of each 128-row column
                // block is one 128-byte line whatever the swizzle.  V_t is waited for only after the
                // previous product has completed: with one V stage, the stage's barrier could
                // otherwise still be on V_{t-1}'s phase, whose parity reads as V_t's being done.
                bool w = t == 0 || mbar_wait(bar(kGbPVDone), (t - 1) & 1, limit, abort_flag);
                w = w && mbar_wait(bar(kGbVFull + t % SV), static_cast<uint32_t>(t / SV) & 1, limit, abort_flag);
                ok = __all_sync(0xffffffffu, w);
                if (!ok) break;
                if (k0 + k >= len) {
                    const uint32_t vrow = sbase + C::kOffV + (t % SV) * C::kTileBytes + k * C::kRowBytes;
#pragma unroll
                    for (int cb = 0; cb < 2; ++cb)
#pragma unroll
                        for (int c16 = 0; c16 < C::kRowBytes; c16 += 16)
                            st_shared_v4(vrow + cb * C::kBlkBytes + c16, 0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_shared();
            // O^T columns of heads whose maximum grew, once the previous product has completed
            if (t > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kGbPVDone), (t - 1) & 1, limit, abort_flag));
                if (!ok) break;
                tc_fence_after_sync();
                if (grew) {  // the same in every thread of the set
                    uint32_t o[RS];
                    ld_cols(t_o, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < RS; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha[i]);
                    st_cols(t_o, o);
                    tmem_st_wait();
                }
            }
            tc_fence_before_sync();
            mbar_arrive(bar(kGbPFull));
        }
        if (ok && nt > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kGbOReady), 0, limit, abort_flag));
            if (ok) tc_fence_after_sync();
        }
        // epilogue: each head's sum over all keys of the split, then the split's normalised
        // output (thread k writes value column k of the set's heads: coalesced rows) and
        // log-sum-exp (o = 0, lse = -inf for a split with no key).
        if (ok && nt > 0) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int i = 0; i < RS; ++i) l[i] += __shfl_xor_sync(0xffffffffu, l[i], off);
            ok = exchange(l, nt, false);
        }
        if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
        if (ok) {  // uniform across the warp (from __all_sync)
            uint32_t o[RS];
            if (nt > 0) {
                ld_cols(t_o, o);
                tmem_ld_wait();
            }
            const size_t row0 = static_cast<size_t>(g) * R;
#pragma unroll
            for (int i = 0; i < RS; ++i) {
                const int h = h0 + i;
                if (h < R) {
                    const size_t slot = (row0 + h) * p.n_splits + s;
                    const float val = (nt > 0 && l[i] > 0.f) ? __uint_as_float(o[i]) / l[i] : 0.f;
                    p.o_part[slot * kGqD + k] = val;
                    if (k == i)
                        p.lse_part[slot] = (nt > 0 && l[i] > 0.f) ? (m_run[i] + lg2_approx(l[i])) * 0.69314718055994531f
                                                                  : -INFINITY;
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kGqWarpMma) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int RH>
cudaError_t launch_gqa_t(const SplitParams& p, cudaStream_t st)
{
    using C = GqCfg<RH>;
    auto kern = fa_gqa_kernel<RH>;
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
    dim3 grid(p.n_splits, p.groups_per_batch, p.n_groups / p.groups_per_batch);
    return launch_pdl(kern, grid, GqShape<RH>::kThreads, C::kSmemBytes, st, p);
}

// Query heads per group R in [5, 32], head size 128.
inline cudaError_t launch_gqa(const SplitParams& p, cudaStream_t st)
{
    const int R = p.rows_per_group;
    if (R <= 8) return launch_gqa_t<8>(p, st);
    if (R <= 16) return launch_gqa_t<16>(p, st);
    if (R <= 32) return launch_gqa_t<32>(p, st);
    return cudaErrorInvalidValue;
}

}  // namespace fa
