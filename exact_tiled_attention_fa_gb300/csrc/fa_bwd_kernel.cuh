// fa_bwd_kernel.cuh -- exact attention backward for sm_103a.
//
// Algorithm: "flash_lab.py -- FlashAttention, flash-decoding and megakernel in
// numpy", section 3 `flash_bwd` (the FlashAttention-2 form of the backward): P is
// not stored by the forward but recomputed on chip from Q, K and the forward's
// log-sum-exp L, P = exp(S - L).  With D_i = sum dO_i o O_i (one number per row,
// computed by the preparation kernel), for a key tile j and every query tile i
// that sees one of its keys:
//   S = Q_i K_j^T scale (causal mask),  P = exp(S - L_i)
//   dV_j += P^T dO_i,  dP = dO_i V_j^T,  dS = P o (dP - D_i)
//   dQ_i += dS K_j scale,  dK_j += dS^T Q_i scale
// The skipped tiles are those whose last query position lies before the key tile's
// first key (query i sits at position Nk - N + i).
//
// GB300 mapping.  A persistent grid (one CTA per SM) walks work items (head, 128-key tile
// j); an item's K_j, V_j load while the previous item runs (double-buffered for d <= 64)
// and its dK_j, dV_j are written while the next item's first products run.  Per item, the CTA
// computes the transposed
// products S^T = K_j Q_i^T and dP^T = V_j dO_i^T, so that a TMEM lane is a key:
// the rows of P^T and dS^T that a thread produces are exactly the A operand rows
// the tensor core needs for dV_j += P^T dO_i (A read from tensor memory) and
// dK_j += dS^T Q_i.  dV_j and dK_j stay in tensor memory for the whole walk.  The
// threads write their dS^T rows to shared memory: read there as K-major rows they are
// the A operand of dK (d <= 64; d = 128 keeps dS^T in tensor memory too), and read as
// MN-major (M-contiguous) they are dS, the A operand of dQ_i = dS K_j.  dQ_i (fp32, TMEM) is added
// into a zeroed fp32 accumulator in global memory, for d <= 64 with bulk reductions from shared
// memory (2 KB blocks; fp32 atomics from the threads measured 13 % slower, the L2's atomic rate being
// the limit), for d = 128 with vector atomics; a final kernel converts it.  The scale is folded into
// dS (both dQ and dK carry it).
//
// Sixteen warps (four warpgroups):
//   warps 0-3 / 4-7  compute: thread t of the warpgroup owns key row t (TMEM lane t)
//                    and half of the query columns (warpgroup 0: queries 0-63,
//                    warpgroup 1: queries 64-127 of the tile).  Per query tile it
//                    reads S^T and writes P^T (bf16), then reads dP^T and writes dS^T
//                    (bf16) to shared memory (and for d = 128 to tensor memory).  At the
//                    end it writes dK_j and dV_j.
//   warp 8           TMA producer: K_j and V_j once; Q_i, dO_i, L_i and D_i into a
//                    ring of three stages (two for d = 128).
//   warps 9, 10      tcgen05 issuers.  Every barrier wait or commit stalls the issuing
//                    thread for a few hundred cycles while the tensor core queues only a
//                    few of these small MMAs, so the work is split: warp 9 issues
//                    S^T(t+1) and dP^T(t+1) as soon as the compute warps have loaded S^T(t)
//                    and dP^T(t) (d <= 64; for d = 128 once dV(t) has read P^T(t) and dQ(t)
//                    has been read out); warp 10 issues dV(t), dK(t), dQ(t) as P^T(t) and
//                    dS^T(t) become ready.  The tensor core works on tile t's products
//                    while the compute warps exponentiate t+1.
//   warps 12-15      dQ reduction: thread t owns query row t of the dQ tile.
// Tensor memory (512 columns): S^T [0,128), dP^T [128,256), dV [256,256+d),
// dK [256+d,256+2d), dQ [384,384+d) and P^T [448,512) for d <= 64: P^T(t) is stored
// once dV(t-1) has read P^T(t-1), dS(t) into shared memory once dK(t-1) and dQ(t-1) have
// read dS(t-1).  For d = 128 there is no room: P^T(t) overwrites the S^T columns it came from,
// dS^T(t) the dP^T columns, dQ(t) overwrites those again once dK(t) has read dS^T,
// and dP(t+1) waits until the dQ reduction warps have read dQ(t) out.
//
// Ordering: a commit tracks every earlier tensor-core operation of its issuing thread.
// For d = 128, S^T(t+1) is issued only after dV(t) has completed, so its arrival also
// tells the compute warps that P^T(t) has been read, and the arrival of dP^T(t+1)
// that dK(t) and dQ(t) have read dS(t).  For d <= 64 the compute warps wait for those
// completions themselves.
//
// Every barrier wait is bounded (BwdParams::wait_limit_ns); a role whose wait runs
// out records FA_ERR_TIMEOUT and raises the CTA's abort flag, each role drains what
// it has in flight, and the CTA frees its tensor memory and exits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"
#include "ptx.cuh"

namespace fa {

constexpr int kBwdThreads = 512;
constexpr int kBwdWarpProducer = 8;
constexpr int kBwdWarpMma = 9;   // warp 9 issues S and dP, warp 10 issues dV, dK and dQ
constexpr int kBwdWarpDq = 12;  // warps 12-15
// Register split after launch (setmaxnreg): the two compute warpgroups grow, the
// control and dQ warpgroups shrink.  The launcher checks kBwdThreads * (registers at
// launch) >= 256 * kBwdComputeRegs + 128 * (kBwdControlRegs + kBwdDqRegs).
constexpr int kBwdComputeRegs = 184;
constexpr int kBwdControlRegs = 80;
constexpr int kBwdDqRegs = 64;

constexpr int kBwdMaxQStages = 3;
constexpr int kBwdMaxKVBufs = 2;
enum : int {
    kBbKVFull = 0,    // +buffer: K_j and V_j landed
    kBbKVEmpty = kBbKVFull + kBwdMaxKVBufs,  // +buffer: both issuers are done with the item's K_j, V_j
    kBbQFull = kBbKVEmpty + kBwdMaxKVBufs,   // +stage: Q_i, dO_i, L_i, D_i landed
    kBbQEmpty = kBbQFull + kBwdMaxQStages,   // +stage: both issuers' tensor-core work on it is done
    kBbSFull = kBbQEmpty + kBwdMaxQStages,   // S^T(t) in TMEM
    kBbDPFull,        // dP^T(t) in TMEM
    kBbPReady,        // P^T(t) written (256 arrivals)
    kBbDSReady,       // dS^T(t) written to TMEM and shared memory (256 arrivals)
    kBbDQFull,        // dQ(t) in TMEM
    kBbDQFree,        // dQ(t) read out of TMEM (128 arrivals)
    kBbDone,          // dV and dK of an item are complete (committed by their issuer alone)
    kBbDrain,         // +issuer (2)
    kBbDPFree = kBbDrain + 2,  // dP^T(t) loaded into registers (256 arrivals)
    kBbDVDone,        // dV(t) has read P^T(t)
    kBbSFree,         // S^T(t) loaded into registers (256 arrivals; d <= 64)
    kBbStageFull,     // the item's dK, dV rows written to the staging tiles (256 arrivals)
    kBbStageFree,     // the bulk stores of the staging tiles have read them
    kBbCount
};

template <int D>
struct BwdCfg {
    static_assert(D == 32 || D == 64 || D == 128, "head size");
    static constexpr int kCB = D < 64 ? D : 64;            // elements per column block
    static constexpr int kNumCB = D / kCB;
    static constexpr int kRowBytes = kCB * 2;
    static constexpr uint32_t kLayout = kRowBytes == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int kAtomBytes = 8 * kRowBytes;
    static constexpr int kBlkBytes = kBlockM * kRowBytes;
    static constexpr int kTileBytes = kNumCB * kBlkBytes;  // 128 x D bf16
    static constexpr int kDSBlk = kBlockM * 128;           // dS: 128 keys x 64 queries (128 B rows)
    // Q_i / dO_i ring depth: a stage is reloaded only after dK of its tile has completed, so
    // two stages leave the S^T(t+2) issue waiting for the load; d = 128 has room for two only.
    static constexpr int kQStages = D == 128 ? 2 : 3;
    static_assert(kQStages <= kBwdMaxQStages, "barrier slots");
    // K_j / V_j buffers: two for d <= 64, so the next item's K and V load while this item runs
    static constexpr int kKVBufs = D == 128 ? 1 : 2;
    static_assert(kKVBufs <= kBwdMaxKVBufs, "barrier slots");
    static constexpr int kOffK = 0;                                       // + buffer * kTileBytes
    static constexpr int kOffV = kKVBufs * kTileBytes;                    // + buffer * kTileBytes
    static constexpr int kOffQ = 2 * kKVBufs * kTileBytes;                // + stage * kTileBytes
    static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;          // + stage * kTileBytes
    static constexpr int kOffDS = kOffDO + kQStages * kTileBytes;         // two query halves of kDSBlk
    static constexpr int kOffL = kOffDS + 2 * kDSBlk;                     // + stage * 512
    static constexpr int kOffDsc = kOffL + kQStages * 512;                // + stage * 512
    // dQ staging for the bulk reductions (dq_bulk): per dQ warp two 2 KB blocks of 32 rows x 16 columns
    static constexpr bool kDQBulk = dq_bulk(D);
    static constexpr int kOffDQS = kOffDsc + kQStages * 512;
    static constexpr int kOffBar = kOffDQS + (kDQBulk ? 4 * 2 * 2048 : 0);
    static constexpr int kNumBars = 26;
    static_assert(kBbCount <= kNumBars, "barrier slots");
    static constexpr int kUsedBytes = kOffBar + kNumBars * 8 + 16;
    static constexpr int kMaxSmem = 232448;                // 227 KB per CTA
    // Up to 1 KB of slack to align the base to the 1024-byte swizzle atom.
    static constexpr int kSmemBytes = kUsedBytes + 1024 <= kMaxSmem ? kUsedBytes + 1024 : kMaxSmem;
    static_assert(kUsedBytes <= kMaxSmem, "shared memory");
    static constexpr int kTmemCols = 512;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    static constexpr uint32_t kColDQ = D == 128 ? 128 : 384;
    static constexpr bool kDQAlias = D == 128;
    // d <= 64: P^T has the last 64 columns to itself and dS^T stays in shared memory, so
    // S^T(t+1) and dP^T(t+1) may start as soon as S^T(t), dP^T(t) are loaded.
    static constexpr bool kDSOwn = D <= 64;
    static constexpr uint32_t kColDS = kColDP;  // d = 128: dS^T over the dP^T columns
    static constexpr uint32_t kColP = kDSOwn ? 448 : kColS;
    static constexpr uint32_t kPHalf = kDSOwn ? 32 : 64;  // columns between the query halves of P^T (and dS^T)
    static constexpr uint32_t kIdescT = idesc_bf16(kBlockN, kBlockM, false);  // S^T, dP^T
    static constexpr uint32_t kIdescAcc = idesc_bf16(kBlockN, D, true);     // dV, dK
    static constexpr uint32_t kIdescDQ = idesc_bf16(kBlockM, D, true) | (1u << 15);  // A MN-major
};

template <int D, bool CAUSAL, typename GradT>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_kernel(const __grid_constant__ BwdParams p)
{
    using C = BwdCfg<D>;
    // No grid_launch_dependents here: letting the dQ conversion that follows launch early made
    // the backward 6 % slower (B=64 H=16 N=1024 d=64); it starts once this grid's CTAs have exited.
    extern __shared__ __align__(1024) uint8_t bwd_smem_raw[];
    const uint32_t raw = smem_u32(bwd_smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    if (pad + C::kUsedBytes > static_cast<uint32_t>(C::kSmemBytes)) {  // cannot align the swizzled tiles
        grid_dependency_wait();
        if (threadIdx.x == 0) atomicCAS(p.status, 0, FA_ERR_UNSUPPORTED);
        return;
    }
    uint8_t* smem = bwd_smem_raw + pad;
    const uint32_t sbase = raw + pad;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long limit = p.wait_limit_ns;

    // ---- work items: (head bh, key tile j), walked persistently.  CTA c takes items c, c + G,
    // c + 2G, ... of the head-major order (the CTAs running at one time share a few heads, so
    // those heads' Q and dO come from HBM once).  Under a causal mask the key tiles of a head
    // are rotated by the head index, so that a CTA's items mix heavy and light walks.
    const int n_items = p.BH * p.Tc;
    const int off = p.Nk - p.N;
    struct Item {
        int bh, j0, i_first, n;
    };
    // CTA c walks items c, c + G, c + 2G, ...; the cursor keeps each item's head, its key tile
    // before the rotation and the rotation (head mod Tc) up to date by additions, as the per-item
    // bookkeeping otherwise costs divisions on warps that share issue slots with busy ones.
    struct Cursor {
        int x, bh, jr, rot;
    };
    auto first_item = [&]() -> Cursor {
        Cursor c;
        c.x = blockIdx.x;
        c.bh = c.x / p.Tc;
        c.jr = c.x - c.bh * p.Tc;
        c.rot = c.bh % p.Tc;
        return c;
    };
    auto next_item = [&](Cursor& c) {
        c.x += gridDim.x;
        c.bh += p.step_heads;
        c.jr += p.step_jr;
        c.rot += p.step_rot;
        if (c.jr >= p.Tc) {
            c.jr -= p.Tc;
            c.bh += 1;
            c.rot += 1;
        }
        if (c.rot >= p.Tc) c.rot -= p.Tc;
    };
    auto item_at = [&](const Cursor& c) -> Item {
        Item it;
        it.bh = c.bh;
        int j = c.jr;
        if (CAUSAL) {
            j += c.rot;  // (jr + bh) mod Tc
            if (j >= p.Tc) j -= p.Tc;
        }
        it.j0 = j * kBlockN;
        it.i_first = 0;
        if (CAUSAL) {
            const int a = it.j0 - off - (kBlockM - 1);  // first tile whose last row position reaches j0
            it.i_first = a <= 0 ? 0 : (a + kBlockM - 1) / kBlockM;
        }
        it.n = p.Tr > it.i_first ? p.Tr - it.i_first : 0;
        return it;
    };
    constexpr int QS = C::kQStages;
    constexpr int KVB = C::kKVBufs;
    // dK_j and dV_j leave through shared memory and bulk tensor stores when both tiles fit in
    // the dS buffer, which no tensor-core operation reads once the item's last dQ is done
    // (bf16 gradients with d <= 64, fp32 with d = 32); otherwise each thread stores its row.
    constexpr int kGRow = D * static_cast<int>(sizeof(GradT));  // bytes of a gradient row
    constexpr bool kStageGrad = C::kDSOwn && kGRow <= 128;
    constexpr int kGTile = kBlockN * kGRow;                      // one staged 128-row tile
    static_assert(!kStageGrad || 2 * kGTile <= 2 * C::kDSBlk, "staging tiles exceed the dS buffer");

    if (threadIdx.x == 0) {
        for (int i = 0; i < KVB; ++i) {
            mbar_init(bar(kBbKVFull + i), 1);
            mbar_init(bar(kBbKVEmpty + i), 2);  // one commit from each issuer
        }
        for (int s = 0; s < QS; ++s) {
            mbar_init(bar(kBbQFull + s), 1);
            mbar_init(bar(kBbQEmpty + s), 2);
        }
        mbar_init(bar(kBbDrain), 1);
        mbar_init(bar(kBbDrain + 1), 1);
        mbar_init(bar(kBbSFull), 1);
        mbar_init(bar(kBbDPFull), 1);
        mbar_init(bar(kBbPReady), 256);
        mbar_init(bar(kBbDSReady), 256);
        mbar_init(bar(kBbDQFull), 1);
        mbar_init(bar(kBbDQFree), 128);
        mbar_init(bar(kBbDPFree), 256);
        // Only warp 10 (dV, dK) commits Done: with two K/V buffers warp 9 may finish the next
        // item before warp 10 finishes this one, and a second arrival of its own would complete
        // the phase early.
        mbar_init(bar(kBbDone), 1);
        mbar_init(bar(kBbDVDone), 1);
        mbar_init(bar(kBbSFree), 256);
        mbar_init(bar(kBbStageFull), 256);
        mbar_init(bar(kBbStageFree), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kBwdWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // Launched with programmatic stream serialization: the setup above may overlap the preparation
    // kernel; every global read and write comes after it has completed.
    grid_dependency_wait();

    if (warp >= 8 && warp < 12) {
        regs_decrease<kBwdControlRegs>();
        if (warp == kBwdWarpProducer && lane == 0) {
            // ============================================================ producer
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
            prefetch_tensormap(&p.tm_do);
            if (kStageGrad) {
                prefetch_tensormap(&p.tm_dk);
                prefetch_tensormap(&p.tm_dv);
            }
            const uint64_t pol_keep = policy_evict_last();  // Q_i, dO_i: read by every key tile of the head
            const uint64_t pol_once = policy_evict_first(); // K_j, V_j: read by one CTA only
            int g = 0;        // query tiles loaded (Q ring position)
            int kv = 0;       // items whose K/V were loaded
            bool ok = true;
            for (Cursor cur = first_item(); ok && cur.x < n_items; next_item(cur)) {
                const Item it = item_at(cur);
                if (it.n == 0) continue;  // no query tile sees this key tile (every role skips it)
                const int kb = kv % KVB;
                if (kv >= KVB && !mbar_wait(bar(kBbKVEmpty + kb), static_cast<uint32_t>(kv / KVB - 1) & 1, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(kBbKVFull + kb), 2 * C::kTileBytes);
#pragma unroll
                for (int cb = 0; cb < C::kNumCB; ++cb) {
                    tma_load_3d(sbase + C::kOffK + kb * C::kTileBytes + cb * C::kBlkBytes, &p.tm_k, bar(kBbKVFull + kb),
                                cb * C::kCB, it.j0, it.bh, pol_once);
                    tma_load_3d(sbase + C::kOffV + kb * C::kTileBytes + cb * C::kBlkBytes, &p.tm_v, bar(kBbKVFull + kb),
                                cb * C::kCB, it.j0, it.bh, pol_once);
                }
                ++kv;
                for (int t = 0; t < it.n; ++t, ++g) {
                    const int s = g % QS;
                    if (g >= QS && !mbar_wait(bar(kBbQEmpty + s), static_cast<uint32_t>(g / QS - 1) & 1, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int i0 = (it.i_first + t) * kBlockM;
                    mbar_arrive_expect_tx(bar(kBbQFull + s), 2 * C::kTileBytes + 2 * 512);
#pragma unroll
                    for (int cb = 0; cb < C::kNumCB; ++cb) {
                        tma_load_3d(sbase + C::kOffQ + s * C::kTileBytes + cb * C::kBlkBytes, &p.tm_q, bar(kBbQFull + s),
                                    cb * C::kCB, i0, it.bh, pol_keep);
                        tma_load_3d(sbase + C::kOffDO + s * C::kTileBytes + cb * C::kBlkBytes, &p.tm_do,
                                    bar(kBbQFull + s), cb * C::kCB, i0, it.bh, pol_keep);
                    }
                    const size_t row = static_cast<size_t>(it.bh) * p.Tr * kBlockM + i0;
                    bulk_load(sbase + C::kOffL + s * 512, p.lse2 + row, 512, bar(kBbQFull + s));
                    bulk_load(sbase + C::kOffDsc + s * 512, p.dsc + row, 512, bar(kBbQFull + s));
                }
            }
            if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            // every issued copy lands before the CTA may exit
            for (int t = kv - KVB < 0 ? 0 : kv - KVB; t < kv; ++t)
                mbar_wait(bar(kBbKVFull + t % KVB), static_cast<uint32_t>(t / KVB) & 1, kDrainLimitNs, nullptr);
            for (int t = g - QS < 0 ? 0 : g - QS; t < g; ++t)
                mbar_wait(bar(kBbQFull + t % QS), static_cast<uint32_t>(t / QS) & 1, kDrainLimitNs, nullptr);
        } else if ((warp == kBwdWarpMma || warp == kBwdWarpMma + 1) && lane == 0) {
            // ============================================================ MMA issuers
            // Barrier operations stall the issuing thread for a few hundred cycles, and the
            // tensor core holds only a short queue of these small MMAs: one issuer that also
            // waits and commits leaves the tensor core idle much of the time.  Warp 9 issues
            // the transposed products S^T, dP^T; warp 10 the accumulations dV, dK and dQ.
            const bool issuer_t = warp == kBwdWarpMma;
            bool ok = true;
            auto wait = [&](int b, int parity) -> bool {
                ok = ok && mbar_wait(bar(b), static_cast<uint32_t>(parity) & 1, limit, abort_flag);
                return ok;
            };
            // S^T = K_j Q_i^T or dP^T = V_j dO_i^T: both operands K-major in shared memory.
            auto issue_t = [&](uint32_t d_col, int a_off, int b_off) {
                const uint64_t a0 = smem_desc(sbase + a_off, 16, C::kAtomBytes, C::kLayout);
                const uint64_t b0 = smem_desc(sbase + b_off, 16, C::kAtomBytes, C::kLayout);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = ((kk * 16) / C::kCB * C::kBlkBytes + ((kk * 16) % C::kCB) * 2) >> 4;
                    umma_ss(tmem + d_col, a0 + o, b0 + o, C::kIdescT, kk > 0 ? 1u : 0u);
                }
            };
            // dV += P^T dO_i or dK += dS^T Q_i: A (bf16, packed two per column) from TMEM, the two
            // query halves half_stride columns apart (64 when each half sits over its own 64
            // source columns, 32 when packed back to back); B MN-major in shared memory.
            auto issue_acc = [&](uint32_t d_col, uint32_t a_col, uint32_t half_stride, int b_off, bool accumulate) {
                const uint64_t b0 = smem_desc(sbase + b_off, C::kBlkBytes, C::kAtomBytes, C::kLayout);
#pragma unroll
                for (int kk = 0; kk < kBlockM / 16; ++kk)
                    umma_ts(tmem + d_col, tmem + a_col + half_stride * (kk >> 2) + 8u * (kk & 3),
                            b0 + ((kk * 16 * C::kRowBytes) >> 4), C::kIdescAcc, (accumulate || kk > 0) ? 1u : 0u);
            };
            // d <= 64: dK += dS^T Q_i with A = dS^T read from the shared-memory dS buffer, whose key
            // rows hold their 128 queries as two swizzled 64-query blocks (K-major for this product).
            auto issue_dk_smem = [&](int q_off, bool accumulate) {
                const uint64_t a0 = smem_desc(sbase + C::kOffDS, 16, 1024, kSwizzle128B);
                const uint64_t b0 = smem_desc(sbase + q_off, C::kBlkBytes, C::kAtomBytes, C::kLayout);
#pragma unroll
                for (int kk = 0; kk < kBlockM / 16; ++kk) {
                    const uint32_t ao = ((kk * 16) / 64 * C::kDSBlk + ((kk * 16) % 64) * 2) >> 4;
                    umma_ss(tmem + C::kColDK, a0 + ao, b0 + ((kk * 16 * C::kRowBytes) >> 4), C::kIdescAcc,
                            (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            // dQ = dS K_j: A = dS (MN-major, two 64-query blocks), B = K_j (MN-major).
            auto issue_dq = [&](int k_off) {
                const uint64_t a0 = smem_desc(sbase + C::kOffDS, C::kDSBlk, 1024, kSwizzle128B);
                const uint64_t b0 = smem_desc(sbase + k_off, C::kBlkBytes, C::kAtomBytes, C::kLayout);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    umma_ss(tmem + C::kColDQ, a0 + ((kk * 16 * 128) >> 4), b0 + ((kk * 16 * C::kRowBytes) >> 4),
                            C::kIdescDQ, kk > 0 ? 1u : 0u);
            };
            int g = 0;  // query tiles processed (all items)
            int k = 0;  // items processed
            for (Cursor cur = first_item(); ok && cur.x < n_items; next_item(cur)) {
                const Item it = item_at(cur);
                if (it.n == 0) continue;
                const int kb = k % KVB;
                const int k_off = C::kOffK + kb * C::kTileBytes;
                const int v_off = C::kOffV + kb * C::kTileBytes;
                if (!wait(kBbKVFull + kb, k / KVB)) break;
                if (issuer_t) {
                    // S^T and dP^T of every query tile; a Q stage is released (one of two arrivals)
                    // once dP^T has been issued, this issuer's last read of it.
                    for (int t = 0; t < it.n; ++t, ++g) {
                        const int s = g % QS;
                        // S^T(g) overwrites S^T(g-1), loaded by the compute warps (d <= 64), or
                        // P^T(g-1) (d = 128), which dV(g-1) must have read
                        if ((g > 0 && !wait(C::kDSOwn ? kBbSFree : kBbDVDone, g - 1)) || !wait(kBbQFull + s, g / QS)) break;
                        tc_fence_after_sync();
                        issue_t(C::kColS, k_off, C::kOffQ + s * C::kTileBytes);
                        umma_commit(bar(kBbSFull));
                        // dP^T(g) overwrites dP^T(g-1): loaded by the compute warps (d <= 64), or, with
                        // dS^T and dQ in those columns (d = 128), dK and dQ done and dQ read out
                        if (g > 0 && !wait(C::kDSOwn ? kBbDPFree : kBbDQFree, g - 1)) break;
                        tc_fence_after_sync();
                        issue_t(C::kColDP, v_off, C::kOffDO + s * C::kTileBytes);
                        umma_commit(bar(kBbDPFull));
                        umma_commit(bar(kBbQEmpty + s));
                    }
                } else {
                    for (int t = 0; t < it.n; ++t, ++g) {
                        const int s = g % QS;
                        if (!wait(kBbPReady, g)) break;
                        tc_fence_after_sync();
                        issue_acc(C::kColDV, C::kColP, C::kPHalf, C::kOffDO + s * C::kTileBytes, t > 0);
                        umma_commit(bar(kBbDVDone));
                        if (!wait(kBbDSReady, g)) break;
                        tc_fence_after_sync();
                        if constexpr (C::kDSOwn)
                            issue_dk_smem(C::kOffQ + s * C::kTileBytes, t > 0);
                        else
                            issue_acc(C::kColDK, C::kColDS, C::kPHalf, C::kOffQ + s * C::kTileBytes, t > 0);
                        umma_commit(bar(kBbQEmpty + s));
                        if (!C::kDQAlias && g > 0 && !wait(kBbDQFree, g - 1)) break;
                        tc_fence_after_sync();
                        issue_dq(k_off);
                        umma_commit(bar(kBbDQFull));
                    }
                }
                if (!ok) break;
                umma_commit(bar(kBbKVEmpty + kb));  // this issuer's reads of K_j, V_j are done
                if (!issuer_t) umma_commit(bar(kBbDone));
                ++k;
            }
            if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            const int me = issuer_t ? 0 : 1;
            umma_commit(bar(kBbDrain + me));
            mbar_wait(bar(kBbDrain + me), 0, kDrainLimitNs, nullptr);
        }
    } else if (warp >= kBwdWarpDq) {
        regs_decrease<kBwdDqRegs>();
        // ============================================================ dQ reduction
        const int r = threadIdx.x & 127;  // query row of the tile == TMEM lane
        const uint32_t t_dq = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::kColDQ;
        bool ok = true;
        int g = 0;
        if constexpr (C::kDQBulk) {
            // Each warp stages its 32 rows 16 columns at a time (column groups of 4: lane l writes 16
            // bytes at (group * 32 + l) * 16, so a warp's stores hit distinct banks) and lane 0 adds the
            // 2 KB block into the accumulator with one bulk reduction; two blocks alternate, and before
            // refilling one, lane 0 waits until the reduction issued from it has read it.
            const int wq = warp & 3;
            const int lane = threadIdx.x & 31;
            const uint32_t stg = sbase + C::kOffDQS + static_cast<uint32_t>(wq) * 4096u;
            int chunks = 0;
            for (Cursor cur = first_item(); ok && cur.x < n_items; next_item(cur)) {
                const Item it = item_at(cur);
                for (int t = 0; t < it.n; ++t, ++g) {
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(kBbDQFull), g & 1, limit, abort_flag));
                    if (!ok) break;
                    tc_fence_after_sync();
                    // this warp's [d/4][32][4] block of the (head, query tile) accumulator
                    float* acc = p.dq_acc + (static_cast<size_t>(it.bh) * p.Tr + (it.i_first + t)) * (D * kBlockM) +
                                 static_cast<size_t>(wq) * (D * 32);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(t_dq + 32u * c, v);
                        tmem_ld_wait();
                        if (c == D / 32 - 1) {  // the whole dQ row is in registers: release the columns
                            tc_fence_before_sync();
                            mbar_arrive(bar(kBbDQFree));
                        }
#pragma unroll
                        for (int k2 = 0; k2 < 2; ++k2, ++chunks) {
                            const uint32_t blk = stg + static_cast<uint32_t>(chunks & 1) * 2048u;
                            if (lane == 0) bulk_wait_read<1>();  // the reduction from this block two chunks ago read it
                            __syncwarp();
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                st_shared_v4(blk + static_cast<uint32_t>(q4 * 32 + lane) * 16u, v[16 * k2 + 4 * q4],
                                             v[16 * k2 + 4 * q4 + 1], v[16 * k2 + 4 * q4 + 2], v[16 * k2 + 4 * q4 + 3]);
                            fence_proxy_async_shared();
                            __syncwarp();
                            if (lane == 0) {
                                bulk_reduce_add_f32(acc + (2 * c + k2) * (4 * 32 * 4), blk, 2048u);
                                bulk_commit_group();
                            }
                        }
                    }
                }
            }
            if (lane == 0 && chunks > 0) bulk_wait_all();  // reductions complete before the CTA exits
        }
        for (Cursor cur = first_item(); !C::kDQBulk && ok && cur.x < n_items; next_item(cur)) {
            const Item it = item_at(cur);
            for (int t = 0; t < it.n; ++t, ++g) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kBbDQFull), g & 1, limit, abort_flag));
                if (!ok) break;
                tc_fence_after_sync();
                float* acc = p.dq_acc + (static_cast<size_t>(it.bh) * p.Tr + (it.i_first + t)) * (D / 4) * (kBlockM * 4) +
                             r * 4;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(t_dq + 32u * c, v);
                    tmem_ld_wait();
                    if (c == D / 32 - 1) {  // the whole dQ row is in registers: release the columns
                        tc_fence_before_sync();
                        mbar_arrive(bar(kBbDQFree));
                    }
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        red_add_v4(acc + static_cast<size_t>(c * 8 + e / 4) * (kBlockM * 4), __uint_as_float(v[e]),
                                   __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                }
            }
        }
        if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
    } else {
        regs_increase<kBwdComputeRegs>();
        // ============================================================ compute
        const int h = warp >> 2;                 // query half of the tile
        const int kr = threadIdx.x & 127;        // key row of the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t t_s = tmem + lane_base + C::kColS + 64u * h;
        const uint32_t t_dp = tmem + lane_base + C::kColDP + 64u * h;
        const uint32_t t_ds = tmem + lane_base + C::kColDS + C::kPHalf * h;
        const uint32_t t_p = tmem + lane_base + C::kColP + C::kPHalf * h;
        const uint32_t ds_row = sbase + C::kOffDS + h * C::kDSBlk + kr * 128;  // this thread's dS^T row
        const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 sc2 = make_float2(p.scale, p.scale);
        bool ok = true;
        int g = 0;
        int k = 0;
        int staged = 0;            // items whose dK, dV went out through the staging tiles
        bool stage_busy = false;   // the last of those stores may still be reading the dS buffer
        for (Cursor cur = first_item(); ok && cur.x < n_items; next_item(cur)) {
            const Item it = item_at(cur);
            const int key = it.j0 + kr;
            const bool valid = key < p.Nk;
            const size_t row = (static_cast<size_t>(it.bh) * p.Nk + (valid ? key : 0)) * D + h * (D / 2);
            GradT* dk = reinterpret_cast<GradT*>(p.dk) + row;
            GradT* dv = reinterpret_cast<GradT*>(p.dv) + row;
            if (it.n == 0) {  // no query sees these keys: zero gradients, no tensor-core work
                float z[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) z[e] = 0.f;
                if (valid)
                    for (int c = 0; c < D / 2; c += 16) {
                        store_row16<GradT>(dv + c, z);
                        store_row16<GradT>(dk + c, z);
                    }
                continue;
            }
            for (int t = 0; t < it.n; ++t, ++g) {
                const int s = g % QS;
                const int i0 = (it.i_first + t) * kBlockM;
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kBbSFull), g & 1, limit, abort_flag));
                if (!ok) break;
                tc_fence_after_sync();
                uint32_t u[64];
                tmem_ld32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
                tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
                tmem_ld_wait();
                if constexpr (C::kDSOwn) {  // the S^T columns may now be overwritten by the next S^T
                    tc_fence_before_sync();
                    mbar_arrive(bar(kBbSFree));
                }
                // P = exp2(S scale log2(e) - L log2(e)); L = +inf gives 0 (row past N or with no key)
                const uint32_t l_addr = sbase + C::kOffL + s * 512 + h * 256;
                float pf[64];
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 l4 = ld_shared_f4(l_addr + c * 4);
                    const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), sl2,
                                                  make_float2(-l4.x, -l4.y));
                    const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])), sl2,
                                                  make_float2(-l4.z, -l4.w));
                    pf[c] = ex2(x01.x);
                    pf[c + 1] = ex2(x01.y);
                    pf[c + 2] = ex2(x23.x);
                    pf[c + 3] = ex2(x23.y);
                }
                if (CAUSAL && off + i0 < it.j0 + kBlockN - 1) {
                    // key j0 + kr is hidden from query i0 + q when j0 + kr > off + i0 + q
                    const int thr = it.j0 + kr - off - i0 - 64 * h;  // my columns c < thr are masked
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c < thr) pf[c] = 0.f;
                }
#pragma unroll
                for (int c = 0; c < 64; c += 2) pk[c / 2] = pack_bf16x2(pf[c], pf[c + 1]);
                if (C::kDSOwn && g > 0) {  // dV must have read the previous P^T from these columns
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(kBbDVDone), (g - 1) & 1, limit, abort_flag));
                    if (!ok) break;
                    tc_fence_after_sync();
                }
                tmem_st32(t_p, pk);
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(bar(kBbPReady));

                ok = __all_sync(0xffffffffu, mbar_wait(bar(kBbDPFull), g & 1, limit, abort_flag));
                if (!ok) break;
                tc_fence_after_sync();
                tmem_ld32(t_dp, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
                tmem_ld32(t_dp + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
                tmem_ld_wait();
                if constexpr (C::kDSOwn) {  // the dP^T columns may now be overwritten by the next dP^T
                    tc_fence_before_sync();
                    mbar_arrive(bar(kBbDPFree));
                }
                // dS' = scale dS = P o (dP scale - scale D)
                const uint32_t d_addr = sbase + C::kOffDsc + s * 512 + h * 256;
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 d4 = ld_shared_f4(d_addr + c * 4);
                    const float2 y01 = __ffma2_rn(make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), sc2,
                                                  make_float2(-d4.x, -d4.y));
                    const float2 y23 = __ffma2_rn(make_float2(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])), sc2,
                                                  make_float2(-d4.z, -d4.w));
                    const float2 g01 = __fmul2_rn(y01, make_float2(pf[c], pf[c + 1]));
                    const float2 g23 = __fmul2_rn(y23, make_float2(pf[c + 2], pf[c + 3]));
                    pk[c / 2] = pack_bf16x2(g01.x, g01.y);
                    pk[c / 2 + 1] = pack_bf16x2(g23.x, g23.y);
                }
                if constexpr (C::kDSOwn) {
                    // the previous dK and dQ must have read the previous dS from shared memory (dQ is
                    // issued after dK by the same thread, so its completion covers both)
                    ok = __all_sync(0xffffffffu, g == 0 || mbar_wait(bar(kBbDQFull), (g - 1) & 1, limit, abort_flag));
                    if (!ok) break;
                    tc_fence_after_sync();
                }
                if (kStageGrad && stage_busy) {  // the previous item's bulk stores read the dS buffer
                    if (threadIdx.x == 0) {
                        bulk_wait_read_all();
                        mbar_arrive(bar(kBbStageFree));
                    }
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(kBbStageFree), (staged - 1) & 1, limit, abort_flag));
                    if (!ok) break;
                    stage_busy = false;
                }
                if constexpr (!C::kDSOwn) tmem_st32(t_ds, pk);  // d = 128: dK reads dS^T from tensor memory
                // dS^T row kr into the MN-major dS operand: 16-byte chunk q8 of the 128-byte row goes
                // to chunk q8 ^ (kr mod 8) (128-byte swizzle).
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8)
                    st_shared_v4(ds_row + ((q8 ^ (kr & 7)) << 4), pk[4 * q8], pk[4 * q8 + 1], pk[4 * q8 + 2],
                                 pk[4 * q8 + 3]);
                fence_proxy_async_shared();
                if constexpr (!C::kDSOwn) tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(bar(kBbDSReady));
            }
            if (!ok) break;
            // dK_j and dV_j of this item: this thread writes key row j0 + kr, columns of its half.
            // The next item's first dV and dK (which overwrite these columns) are issued only after
            // this warpgroup's next P^T arrival, i.e. after these loads.
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kBbDone), k & 1, limit, abort_flag));
            if (!ok) break;
            ++k;
            tc_fence_after_sync();
            if constexpr (kStageGrad) {
                // Row kr of each tile, this thread's half of the columns, into the staging tiles
                // (dV at the start of the dS buffer, dK after it), 16-byte chunks swizzled like
                // the tensor maps (chunk index XOR kr mod 8 for 128-byte rows, XOR (kr / 2) mod 4
                // for 64-byte rows); one thread then stores both tiles, rows past Nk clipped.
                constexpr int kEpc = 16 / static_cast<int>(sizeof(GradT));  // elements per chunk
                constexpr int kHalfChunks = kGRow / 32;                     // chunks of a half row
                const uint32_t sw = kGRow == 128 ? static_cast<uint32_t>(kr & 7) : static_cast<uint32_t>((kr >> 1) & 3);
                const uint32_t stg = sbase + C::kOffDS + static_cast<uint32_t>(kr) * kGRow;
                uint32_t a[D / 2], b[D / 2];
#pragma unroll
                for (int c = 0; c < D / 2; c += 16) {
                    tmem_ld16(tmem + lane_base + C::kColDV + h * (D / 2) + c, *reinterpret_cast<uint32_t(*)[16]>(&a[c]));
                    tmem_ld16(tmem + lane_base + C::kColDK + h * (D / 2) + c, *reinterpret_cast<uint32_t(*)[16]>(&b[c]));
                }
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < kHalfChunks; ++q) {
                    const uint32_t off = ((static_cast<uint32_t>(h * kHalfChunks + q) ^ sw) << 4);
                    const int e = q * kEpc;
                    if constexpr (sizeof(GradT) == 2) {
                        st_shared_v4(stg + off, pack_bf16x2(__uint_as_float(a[e]), __uint_as_float(a[e + 1])),
                                     pack_bf16x2(__uint_as_float(a[e + 2]), __uint_as_float(a[e + 3])),
                                     pack_bf16x2(__uint_as_float(a[e + 4]), __uint_as_float(a[e + 5])),
                                     pack_bf16x2(__uint_as_float(a[e + 6]), __uint_as_float(a[e + 7])));
                        st_shared_v4(stg + kGTile + off, pack_bf16x2(__uint_as_float(b[e]), __uint_as_float(b[e + 1])),
                                     pack_bf16x2(__uint_as_float(b[e + 2]), __uint_as_float(b[e + 3])),
                                     pack_bf16x2(__uint_as_float(b[e + 4]), __uint_as_float(b[e + 5])),
                                     pack_bf16x2(__uint_as_float(b[e + 6]), __uint_as_float(b[e + 7])));
                    } else {
                        st_shared_v4(stg + off, a[e], a[e + 1], a[e + 2], a[e + 3]);
                        st_shared_v4(stg + kGTile + off, b[e], b[e + 1], b[e + 2], b[e + 3]);
                    }
                }
                fence_proxy_async_shared();
                mbar_arrive(bar(kBbStageFull));
                bool stored = true;
                if (threadIdx.x == 0) {
                    stored = mbar_wait(bar(kBbStageFull), staged & 1, limit, abort_flag);
                    if (stored) {
                        tma_store_3d(&p.tm_dv, sbase + C::kOffDS, 0, it.j0, it.bh);
                        tma_store_3d(&p.tm_dk, sbase + C::kOffDS + kGTile, 0, it.j0, it.bh);
                        bulk_commit_group();
                    }
                }
                ok = __all_sync(0xffffffffu, stored);
                if (!ok) break;
                ++staged;
                stage_busy = true;
            } else {
#pragma unroll
                for (int c = 0; c < D / 2; c += 16) {
                    uint32_t a[16], b[16];
                    tmem_ld16(tmem + lane_base + C::kColDV + h * (D / 2) + c, a);
                    tmem_ld16(tmem + lane_base + C::kColDK + h * (D / 2) + c, b);
                    tmem_ld_wait();
                    float fa[16], fb[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        fa[e] = __uint_as_float(a[e]);
                        fb[e] = __uint_as_float(b[e]);
                    }
                    if (valid) {
                        store_row16<GradT>(dv + c, fa);
                        store_row16<GradT>(dk + c, fb);
                    }
                }
            }
        }
        if (kStageGrad && threadIdx.x == 0 && staged > 0) bulk_wait_all();  // stores done before exit
        if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kBwdWarpMma) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool CAUSAL, typename GradT>
cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t st)
{
    using C = BwdCfg<D>;
    auto kern = fa_bwd_kernel<D, CAUSAL, GradT>;
    static bool configured[64] = {};
    static int regs[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, kern);
        if (e != cudaSuccess) return e;
        regs[dev] = attr.numRegs;
        configured[dev] = true;
    }
    if (regs[dev] * kBwdThreads < 256 * kBwdComputeRegs + 128 * (kBwdControlRegs + kBwdDqRegs))
        return cudaErrorLaunchOutOfResources;  // the register split would not fit
    const long long items = static_cast<long long>(p.BH) * p.Tc;
    if (items <= 0) return cudaSuccess;
    const long long grid = items < p.num_ctas ? items : p.num_ctas;  // persistent: one CTA per SM
    BwdParams q = p;  // the cursor's steps (see first_item / next_item)
    q.step_heads = static_cast<int>(grid / p.Tc);
    q.step_jr = static_cast<int>(grid % p.Tc);
    q.step_rot = q.step_heads % p.Tc;
    return launch_pdl(kern, static_cast<unsigned>(grid), kBwdThreads, C::kSmemBytes, st, q);
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, bool causal, fa_dtype grad_dtype, cudaStream_t st)
{
    if (grad_dtype == FA_F32)
        return causal ? launch_bwd_t<D, true, float>(p, st) : launch_bwd_t<D, false, float>(p, st);
    return causal ? launch_bwd_t<D, true, __nv_bfloat16>(p, st) : launch_bwd_t<D, false, __nv_bfloat16>(p, st);
}

}  // namespace fa
