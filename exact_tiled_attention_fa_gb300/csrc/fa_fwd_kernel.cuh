// fa_fwd_kernel.cuh -- exact attention forward for sm_103a.
//
// Algorithm: "flash_lab.py -- FlashAttention, flash-decoding and megakernel in
// numpy", section 3 `flash_fwd`, FlashAttention-2 loop order: a query tile walks
// the key/value tiles of its head keeping the running row max m and row sum l
// (section 1, `softmax_online`: the old sum is rescaled by exp(m_old - m_new)) and
// an unnormalised O accumulator on chip; O is divided by l once at the end and
// LSE = m + log l.  With a causal mask the walk stops at the first tile lying
// wholly after the tile's last query position (query i sits at position
// Nk - N + i; "02_flash_forward.py", demo 1).
//
// GB300 mapping.  A persistent grid (one CTA per SM) walks work items; an item is
// one head and a pair of 128-row query tiles Q0, Q1 that share every K/V tile.
// Items are ordered head-major (the query pairs of one head run on neighbouring
// CTAs, so that head's K and V are read from HBM once and then hit in L2) and are
// handed out two at a time, a heavy and a light one (see first_item); under a causal
// mask odd items swap which slot takes the upper query tile (d <= 64, decode_item).
// Twelve warps (three warpgroups, as `setmaxnreg` acts on whole warpgroups):
//   warps 0-3 / 4-7  softmax warpgroups for Q0 / Q1: thread t owns query row t
//                    (= TMEM lane t): it reads its score row from TMEM, masks,
//                    updates m and l in base 2 with a log2(e)-prescaled scale,
//                    writes P (bf16) back to TMEM, rescales its O row when the max
//                    grew, and at the end of the item writes LSE and O / l (d <= 64:
//                    through a shared-memory staging tile and one bulk tensor store).
//   warp 8           TMA producer: Q0, Q1 per item (double-buffered for d <= 64),
//                    K_j / V_j into a ring of stages.
//   warps 9, 10      tcgen05 issuers for Q0 and Q1: S_i = Q_i K_j^T (both operands in
//                    shared memory) and O_i += P_i V_j (P from tensor memory, V from
//                    shared memory), each issuing PV_i(j) then S_i(j+1): while one
//                    warpgroup exponentiates, the tensor core runs the other's MMAs.
//                    Every barrier wait or commit stalls the issuing thread for a few
//                    hundred cycles, so each issuer handles only its own query tile,
//                    and K_j / V_j share one barrier.
//   warp 11          idle (completes the control warpgroup).
// For d = 128 without a mask (kernels with long, uniform items whose row-store epilogue is
// costly) a fourth warpgroup, warps 12-15, takes the epilogue of both query tiles: once an
// item's last P V has completed it reads O_i out of TMEM, releases the columns for the next
// item's first P V and stores O / l, while the softmax warps hand over 1 / l and move on to
// the next item at once (its S already computed).  The control warpgroup is then warps 8-11 as
// above.  (For d <= 64, and under a causal mask, this role costs more than it saves: the
// softmax warpgroups lose the registers it takes, and with short causal items one warpgroup
// doing both tiles' epilogues falls behind.)
// Tensor memory (512 columns): S0, S1 (128 fp32 columns each), O0, O1 (d each) and
// P0, P1 (64 columns of packed bf16 each).  For d = 128 there is no room left, so
// P_i overwrites the first half of S_i (already read into registers); S_i(j+1) is
// then issued only after P_i(j) V_j has completed.
// Because every commit tracks all earlier MMAs of the issuing thread, the arrival of
// S_i(j) also means P_i(j-1) V_{j-1} has completed: the softmax can then overwrite
// P_i and rescale O_i without a separate wait.
//
// Precision: the running max moves whenever a tile raises it, so the largest P of a
// row is exactly 1 in bf16.  (Keeping a stale max to skip rescales, with P up to
// 2^k, leaves that dominant weight rounded: with values of magnitude ~8 the O error
// then reaches 2e-2, above the 1e-2 the results must meet.)  A warp rescales its O
// rows only when the max of one of its rows grew.
//
// Split mode (SPLIT = true, fa_fwd_splitkv; "flash_lab.py" section 4 `split_kv_decode` applied
// to query tiles): for few query tiles over many keys the keys are also cut into ranges of whole
// key tiles; an item is (head, query pair, split), its walk covers the split's key tiles (masked
// as usual by their absolute positions), and its epilogue writes each row's normalised fp32
// partial O and natural-log LSE to the split's slot (O = 0, LSE = -inf for a row that sees no key
// of the split); a merge kernel combines the slots.
//
// Every barrier wait is bounded (FwdParams::wait_limit_ns).  A role whose wait runs
// out records FA_ERR_TIMEOUT and raises the CTA's abort flag so the other roles stop
// too; each role then drains what it has in flight (TMA copies, tensor-core
// operations) before the CTA frees its tensor memory and exits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"
#include "ptx.cuh"

namespace fa {

constexpr int kFwdThreads = 384;  // 12 warps = 3 warpgroups
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;       // warps 9 and 10 issue the MMAs of Q0 and Q1; warp 11 idles
constexpr int kWarpCorr = 12;     // warps 12-15: correction warpgroup (kernels with kCorr only)

// Whether the kernel has a correction warpgroup (16 warps) doing the epilogue.
template <int D, bool CAUSAL>
constexpr bool kCorr = D == 128 && !CAUSAL;
template <int D, bool CAUSAL>
constexpr int kThreads = kCorr<D, CAUSAL> ? 512 : kFwdThreads;
// Whether the kernel walks its items in the ordered form (full query pairs first, then the heads'
// one-tile last pairs; see FwdParams::n_full).  Only the d = 128 kernels without a mask, whose
// uniform items make the last round's length matter: the extra cursor code costs the d = 64
// kernels ~0.8 %.
template <int D, bool CAUSAL>
constexpr bool kOrderedWalk = kCorr<D, CAUSAL>;
// Registers per thread after the split: the producer / MMA warpgroup gives registers to the
// two softmax warpgroups.  The split needs kFwdThreads * (registers at launch) >=
// 256 * kSoftmaxRegs + 128 * kControlRegs; the launcher checks this before every launch,
// because an increase that the pool cannot satisfy would wait forever.
// d = 128 keeps the softmax at 224 (its long causal prefill measured 1.6 % faster than with 216);
// for d <= 64 the control warps get 72 (the d = 64 prefill measured 1.6 % faster than with 56).
template <int D>
constexpr int kSoftmaxRegs = D == 128 ? 224 : 216;
template <int D>
constexpr int kControlRegs = D == 128 ? 56 : 72;
// With a correction warpgroup (512 threads, 128 registers each at launch): 256 * 184 + 128 * 72
// + 128 * 72 = 65536, the splits for which ptxas reports no spills in any role.
constexpr int kCorrSoftmaxRegs = 184;
constexpr int kCorrRegs = 72;
constexpr int kCorrControlRegs = 72;

// barrier slots
constexpr int kMaxStages = 8;
enum : int {
    kBarQFull = 0,                         // +2 * buffer + tile (4)
    kBarQEmpty = 4,                        // +2 * buffer + tile (4)
    kBarSFull = 8,                         // +tile (2)
    kBarPFull = 10,                        // +tile (2)
    kBarPVDone = 12,                       // +tile (2)
    kBarOReady = 14,                       // +tile (2)
    kBarDrain = 16,                         // +tile (2)
    kBarSFree = 18,                         // +tile (2): the softmax has read S_i out of TMEM
    kBarKVFull = 20,                        // +stage: K_j and V_j landed
    kBarKVEmpty = kBarKVFull + kMaxStages,  // +stage: both issuers are done with the stage
    kBarLFull = kBarKVEmpty + kMaxStages,   // +tile (2): the softmax wrote the item's 1 / l rows (kCorr)
    kBarOFree = kBarLFull + 2,              // +tile (2): the correction warps read O_i and 1 / l (kCorr)
    kBarCount = kBarOFree + 2
};

template <int D, int OutBytes>
struct FwdCfg {
    static_assert(D == 32 || D == 64 || D == 128, "head size");
    static constexpr int kCB = D < 64 ? D : 64;            // elements per column block (swizzle span)
    static constexpr int kNumCB = D / kCB;                 // column blocks per row
    static constexpr int kRowBytes = kCB * 2;              // 64 or 128 bytes
    static constexpr uint32_t kLayout = kRowBytes == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int kAtomBytes = 8 * kRowBytes;       // 8-row swizzle atom
    static constexpr int kBlkBytes = kBlockM * kRowBytes;  // one 128-row column block
    static constexpr int kTileBytes = kNumCB * kBlkBytes;  // 128 x D bf16
    // K/V ring depth: d = 64 with bf16 output has room for a fourth stage beside its staging tiles
    static constexpr int kStages = D == 128 ? 2 : (D == 64 ? (OutBytes == 2 ? 4 : 3) : 4);
    // Q buffers per query tile: two for d <= 64, so the next item's Q loads while the
    // current item runs (an item there spans few key tiles); one for d = 128 (no room).
    static constexpr int kQBuf = D == 128 ? 1 : 2;
    static constexpr int kOffQ = 0;  // Q buffer (b, i) at kOffQ + (2 * b + i) * kTileBytes
    static constexpr int kOffK = 2 * kQBuf * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    // For d <= 64 the epilogue writes O / l through shared memory and one bulk tensor store per
    // query tile (a thread owns a row, so direct global stores would be 16-byte pieces 2*d bytes
    // apart); one staging tile per query tile, sized for the output type.  d = 128 has no room left
    // and stores rows directly (its items are long, so the epilogue weighs little).
    static constexpr bool kStoreO = D <= 64;
    static constexpr bool kAlternate = D <= 64;  // causal items alternate their query tiles (decode_item)
    static constexpr int kOffStage = kOffV + kStages * kTileBytes;
    static constexpr int kStageTileBytes = kStoreO ? kBlockM * D * OutBytes : 0;
    static constexpr int kOffInvL = kOffStage + 2 * kStageTileBytes;  // fp32 1 / l per row (kCorr)
    static constexpr int kOffBar = kOffInvL + (D == 128 ? 2 * kBlockM * 4 : 0);
    static constexpr int kNumBars = 48;
    static_assert(kStages <= kMaxStages && kBarCount <= kNumBars, "barrier slots");
    static constexpr int kUsedBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + 1 KB alignment slack
    static_assert(kUsedBytes <= 227 * 1024, "shared memory per CTA");
    // At least 120 KB so that a second CTA (which would wait for the 512 TMEM columns
    // this persistent CTA holds) never shares the SM.
    static constexpr int kSmemBytes = kUsedBytes > 120 * 1024 ? kUsedBytes : 120 * 1024;
    static constexpr int kTmemCols = 512;
    static constexpr bool kAliasP = (D == 128);
    __host__ __device__ static constexpr uint32_t col_s(int i) { return 128u * i; }
    __host__ __device__ static constexpr uint32_t col_o(int i) { return 256u + static_cast<uint32_t>(D) * i; }
    __host__ __device__ static constexpr uint32_t col_p(int i)
    {
        return kAliasP ? col_s(i) : 256u + 2u * D + 64u * i;
    }
    static constexpr uint32_t kIdescS = idesc_bf16(kBlockM, kBlockN, false);
    static constexpr uint32_t kIdescO = idesc_bf16(kBlockM, D, true);
};


__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Layout of a staged output tile: column blocks of 128-byte rows (64-byte rows for bf16 with
// d = 32), 128 rows each, swizzled like the tensor map that stores them (the 16-byte chunk
// index of row r XOR r mod 8 for 128-byte rows, XOR (r / 2) mod 4 for 64-byte rows), so that
// the 32 rows a warp writes at once fall on distinct banks.
template <typename OutT, int D>
struct OStage {
    static constexpr int kRowBytes = D * static_cast<int>(sizeof(OutT)) < 128 ? D * static_cast<int>(sizeof(OutT)) : 128;
    static constexpr int kElems = kRowBytes / static_cast<int>(sizeof(OutT));  // elements per block row
    static constexpr int kNumCB = D / kElems;
    static constexpr int kBlkBytes = kBlockM * kRowBytes;
    static constexpr int kChunks = kRowBytes / 16;
};

// Writes row r of a staged output tile: the raw fp32 O words times inv, converted to OutT.
template <typename OutT, int D>
__device__ __forceinline__ void stage_row(uint32_t stg, int r, const uint32_t (&o)[D], float inv)
{
    using OS = OStage<OutT, D>;
    constexpr int kEpc = 16 / static_cast<int>(sizeof(OutT));  // elements per 16-byte chunk
    const uint32_t row_addr = stg + static_cast<uint32_t>(r) * OS::kRowBytes;
    const uint32_t sw = OS::kRowBytes == 128 ? static_cast<uint32_t>(r & 7) : static_cast<uint32_t>((r >> 1) & 3);
#pragma unroll
    for (int g = 0; g < D / kEpc; ++g) {
        const uint32_t addr = row_addr + static_cast<uint32_t>((g / OS::kChunks) * OS::kBlkBytes) +
                              ((static_cast<uint32_t>(g % OS::kChunks) ^ sw) << 4);
        const int e = g * kEpc;
        if constexpr (sizeof(OutT) == 2) {
            st_shared_v4(addr, pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                         pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                         pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                         pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
        } else {
            st_shared_v4(addr, __float_as_uint(__uint_as_float(o[e]) * inv), __float_as_uint(__uint_as_float(o[e + 1]) * inv),
                         __float_as_uint(__uint_as_float(o[e + 2]) * inv), __float_as_uint(__uint_as_float(o[e + 3]) * inv));
        }
    }
}

// Shape of one work item (head bh, query rows [i0, i0 + 256)).  Query tile slot i (warpgroup i,
// issuer i) takes rows [r0[i], r0[i] + 128).
struct Item {
    int bh, i0;
    int split, j0;  // split mode: the item's key range starts at key tile j0 (0 otherwise)
    int r0[2];    // first query row of slot 0 / 1
    int rows[2];  // valid query rows of slot 0 / 1 (0 when the tile lies past N)
    int n[2];     // key/value tiles each query tile visits
    int n_kv;     // max(n[0], n[1])
};

// The work items of a CTA.  Under a causal mask a CTA takes pairs
// of consecutive items (pair blockIdx.x + t * gridDim.x): within a head the query pairs run
// heaviest, lightest, second heaviest, second lightest, ... (see decode_item), so the two
// items of a pair together carry about the same work as any other pair and the static
// assignment stays balanced without a global work counter.  Without a mask every item
// carries the same work and CTA c takes items c, c + G, c + 2G, ...: the last round is then
// one item, not one pair, short (B=64 H=16 N=1024: 27 items on the busiest CTA instead of 28);
// so does a causal launch with no more items than CTAs (each item then has a CTA of its own).
// This CTA's items in that order, with each item's head and position in the head
// advanced by additions: the per-item bookkeeping runs on warps that share their issue slots
// with exponentiating warps, where a 32-bit division and 64-bit index arithmetic cost hundreds
// of cycles at every item boundary.
struct ItemCursor {
    int item, bh, t, k;
};

// `pairs` is the launch's FwdParams::pairs, passed as false by non-causal kernels (never paired).
// Without a mask (`ordered`) t is the query pair itself, and items past BH * n_full are the heads'
// one-tile last pairs (bh = item - BH * n_full, t = n_qp - 1).
__device__ __forceinline__ ItemCursor first_item(const FwdParams& p, bool pairs, bool ordered = false)
{
    ItemCursor c;
    c.item = pairs ? 2 * static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
    c.k = 0;
    if (ordered) {
        const int full = p.BH * p.n_full;
        if (c.item < full) {
            c.bh = c.item / p.n_full;
            c.t = c.item - c.bh * p.n_full;
        } else {
            c.bh = c.item - full;
            c.t = p.n_qp - 1;
        }
        return c;
    }
    c.bh = c.item / p.n_qp;
    c.t = c.item - c.bh * p.n_qp;
    return c;
}

__device__ __forceinline__ void next_item(const FwdParams& p, ItemCursor& c, bool pairs, bool ordered = false)
{
    if (ordered) {  // singly, step G: (head, pair) advanced by additions while in the full pairs
        c.item += static_cast<int>(gridDim.x);
        const int full = p.BH * p.n_full;
        if (c.item < full) {
            c.bh += p.step_heads;
            c.t += p.step_rem;
            if (c.t >= p.n_full) {
                c.t -= p.n_full;
                c.bh += 1;
            }
        } else {
            c.bh = c.item - full;
            c.t = p.n_qp - 1;
        }
        c.k += 1;
        return;
    }
    if (pairs && (c.k & 1) == 0) {  // second item of the pair
        c.item += 1;
        c.t += 1;
    } else {                         // first item of the next round
        c.item += pairs ? 2 * static_cast<int>(gridDim.x) - 1 : static_cast<int>(gridDim.x);
        c.bh += p.step_heads;
        c.t += p.step_rem;
    }
    if (c.t >= p.n_qp) {
        c.t -= p.n_qp;
        c.bh += 1;
    }
    c.k += 1;
}

template <bool SPLIT = false>
__device__ __forceinline__ Item decode_item(const FwdParams& p, const ItemCursor& c, bool causal, bool alternate,
                                            bool ordered = false)
{
    const int item = c.item;
    Item it;
    it.bh = c.bh;
    const int t = c.t;
    int qp;
    it.split = 0;
    it.j0 = 0;
    if constexpr (SPLIT) {  // t = query pair * n_splits + split
        qp = t / p.n_splits;
        it.split = t - qp * p.n_splits;
        it.j0 = it.split * p.split_tiles;
    } else {
        // heavy, light, heavy, light, ...; in the ordered walk (no mask, one-tile last pairs) t is the pair
        qp = ordered ? t : (t & 1) ? (t >> 1) : p.n_qp - 1 - (t >> 1);
    }
    it.i0 = qp * 2 * kBlockM;
    const int n_all = (p.Nk + kBlockN - 1) / kBlockN;
    const int off = p.Nk - p.N;
    // Under a causal mask the upper query tile of a pair sees one key tile more than the lower
    // one, and the slot with fewer tiles can only run ahead as far as the shared K/V ring lets
    // it.  With `alternate`, odd items (every second item of a CTA) swap the halves, so over two
    // items both slots carry the same number of tiles (d <= 64: causal prefill 670 -> 699
    // TFLOP/s; the long d = 128 items measured 10 % slower with it, so they keep the order).
    const int swap = (causal && alternate) ? (item & 1) : 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r0 = it.i0 + (i ^ swap) * kBlockM;
        it.r0[i] = r0;
        it.rows[i] = r0 < p.N ? min(kBlockM, p.N - r0) : 0;
        int n = it.rows[i] > 0 ? n_all : 0;
        if (causal && n > 0) {
            const int last_pos = off + r0 + it.rows[i] - 1;  // position of the tile's last query row
            n = last_pos < 0 ? 0 : min(n_all, last_pos / kBlockN + 1);
        }
        if constexpr (SPLIT) n = max(0, min(n, it.j0 + p.split_tiles) - it.j0);  // tiles j0 .. j0 + n - 1
        it.n[i] = n;
    }
    it.n_kv = max(it.n[0], it.n[1]);
    return it;
}

// Correction warpgroup (kCorr kernels, d = 128): the epilogue of both query tiles.  Warp w reads
// TMEM lanes 32 (w mod 4) .. 32 (w mod 4) + 31, i.e. those rows of O0 and of O1.  For each item
// and query tile with rows: once the item's last P V has completed (OReady) and the softmax has
// written the rows' 1 / l (LFull), it reads O_i 32 columns at a time and stores the rows of
// O / l; then it releases the columns (OFree: the next item's first P V may overwrite them and
// the softmax may write the next 1 / l).
template <int D, bool CAUSAL, typename OutT, bool SPLIT>
__device__ __forceinline__ void fwd_correction(const FwdParams& p, const uint8_t* smem, uint32_t bar0, uint32_t tmem,
                                               volatile int* abort_flag)
{
    using C = FwdCfg<D, static_cast<int>(sizeof(OutT))>;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = 32 * (warp & 3) + lane;  // row within a query tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float* inv_l = reinterpret_cast<const float*>(smem + C::kOffInvL);
    const unsigned long long limit = p.wait_limit_ns;
    int done[2] = {0, 0};  // items whose O_i this warpgroup has read, per query tile
    bool ok = true;
    for (ItemCursor cur = first_item(p, CAUSAL && p.pairs, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp); ok && cur.item < p.n_items; next_item(p, cur, CAUSAL && p.pairs, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp)) {
        const Item it = decode_item<SPLIT>(p, cur, CAUSAL, C::kAlternate, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int rows = it.rows[i];
            if (rows == 0) continue;  // tile lies past N
            const int n = it.n[i];
            if (n > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarOReady + i), done[i] & 1, limit, abort_flag) &&
                                                 mbar_wait(bar(kBarLFull + i), done[i] & 1, limit, abort_flag));
                if (!ok) break;
                tc_fence_after_sync();
            }
            const float inv = n > 0 ? inv_l[i * kBlockM + r] : 0.f;
            const bool valid = r < rows;
            const size_t row = static_cast<size_t>(it.bh) * p.N + static_cast<size_t>(it.r0[i] + r);
            OutT* orow = SPLIT ? reinterpret_cast<OutT*>(p.o_part) + (row * p.n_splits + it.split) * D
                               : reinterpret_cast<OutT*>(p.o) + row * D;
            const uint32_t t_o = tmem + lane_base + C::col_o(i);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                if (n > 0) {
                    uint32_t o[32];
                    tmem_ld32(t_o + 32u * c, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv;
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0.f;
                }
                if (valid) {
                    if constexpr (SPLIT)
                        store_row32_aligned32(reinterpret_cast<float*>(orow) + 32 * c, v);
                    else
                        store_row32<OutT>(orow + 32 * c, v);
                }
            }
            if (n > 0) {
                tc_fence_before_sync();
                mbar_arrive(bar(kBarOFree + i));
                ++done[i];
            }
        }
    }
    if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
}

template <int D, bool CAUSAL, typename OutT, bool SPLIT>
__global__ void __launch_bounds__(kThreads<D, CAUSAL>, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p)
{
    using C = FwdCfg<D, static_cast<int>(sizeof(OutT))>;
    static_assert(!SPLIT || sizeof(OutT) == 4, "split partials are fp32");
    constexpr int S = C::kStages;
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
    const unsigned long long limit = p.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(kBarQFull + i), 1);
            mbar_init(bar(kBarQEmpty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarSFull + i), 1);
            mbar_init(bar(kBarPFull + i), kBlockM);
            mbar_init(bar(kBarPVDone + i), 1);
            mbar_init(bar(kBarOReady + i), 1);
            mbar_init(bar(kBarDrain + i), 1);
            mbar_init(bar(kBarSFree + i), kBlockM);
            mbar_init(bar(kBarLFull + i), kBlockM);
            mbar_init(bar(kBarOFree + i), kBlockM);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(kBarKVFull + s), 1);
            mbar_init(bar(kBarKVEmpty + s), 2);  // one arrival from each MMA issuer
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // Launched with programmatic stream serialization: the setup above may overlap the previous
    // kernel on the stream; every global read and write comes after that kernel has completed.
    // Then the next kernel (the merge of split mode, or the next forward) may begin launching and
    // set itself up while this grid runs; it waits for this grid's completion in the same way.
    grid_dependency_wait();
    grid_launch_dependents();

    constexpr bool kWithCorr = kCorr<D, CAUSAL>;
    if (kWithCorr && warp >= kWarpCorr) {
        if constexpr (kWithCorr) {
            regs_decrease<kCorrRegs>();
            // ============================================================ correction / epilogue
            fwd_correction<D, CAUSAL, OutT, SPLIT>(p, smem, bar0, tmem, abort_flag);
        }
    } else if (warp >= kWarpProducer) {
      regs_decrease<kWithCorr ? kCorrControlRegs : kControlRegs<D>>();
      if (warp == kWarpProducer) {
        // ============================================================ producer
        if (lane == 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
            if (C::kStoreO && !SPLIT) prefetch_tensormap(&p.tm_o);
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            int q_loads[2] = {0, 0};  // loads issued into each Q buffer
            long long g = 0;          // K/V tiles issued so far (ring position)
            bool ok = true;
            for (ItemCursor cur = first_item(p, CAUSAL && p.pairs, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp); ok && cur.item < p.n_items; next_item(p, cur, CAUSAL && p.pairs, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp)) {
                const Item it = decode_item<SPLIT>(p, cur, CAUSAL, C::kAlternate, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp);
                for (int i = 0; i < 2 && ok; ++i) {
                    if (it.n[i] == 0) continue;
                    const int b = q_loads[i] % C::kQBuf;  // buffer of this load
                    const int q_bar = 2 * b + i;
                    if (q_loads[i] >= C::kQBuf &&
                        !mbar_wait(bar(kBarQEmpty + q_bar), (q_loads[i] / C::kQBuf - 1) & 1, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(kBarQFull + q_bar), C::kTileBytes);
#pragma unroll
                    for (int cb = 0; cb < C::kNumCB; ++cb)
                        tma_load_3d(sbase + C::kOffQ + q_bar * C::kTileBytes + cb * C::kBlkBytes, &p.tm_q,
                                    bar(kBarQFull + q_bar), cb * C::kCB, it.r0[i], it.bh, pol_q);
                    ++q_loads[i];
                }
                for (int j = 0; ok && j < it.n_kv; ++j, ++g) {
                    const int s = static_cast<int>(g % S);
                    const uint32_t round = static_cast<uint32_t>(g / S);
                    if (g >= S && !mbar_wait(bar(kBarKVEmpty + s), (round - 1) & 1, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(kBarKVFull + s), 2 * C::kTileBytes);
#pragma unroll
                    for (int cb = 0; cb < C::kNumCB; ++cb)
                        tma_load_3d(sbase + C::kOffK + s * C::kTileBytes + cb * C::kBlkBytes, &p.tm_k,
                                    bar(kBarKVFull + s), cb * C::kCB, (it.j0 + j) * kBlockN, it.bh, pol_kv);
#pragma unroll
                    for (int cb = 0; cb < C::kNumCB; ++cb)
                        tma_load_3d(sbase + C::kOffV + s * C::kTileBytes + cb * C::kBlkBytes, &p.tm_v,
                                    bar(kBarKVFull + s), cb * C::kCB, (it.j0 + j) * kBlockN, it.bh, pol_kv);
                }
            }
            if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            // Every issued copy must land before the CTA may exit (its last phase per barrier).
            for (int i = 0; i < 2; ++i)
                for (int t = q_loads[i] - C::kQBuf < 0 ? 0 : q_loads[i] - C::kQBuf; t < q_loads[i]; ++t)
                    mbar_wait(bar(kBarQFull + 2 * (t % C::kQBuf) + i), (t / C::kQBuf) & 1, kDrainLimitNs, nullptr);
            for (long long t = g - S < 0 ? 0 : g - S; t < g; ++t) {
                const int s = static_cast<int>(t % S);
                const uint32_t par = static_cast<uint32_t>(t / S) & 1;
                mbar_wait(bar(kBarKVFull + s), par, kDrainLimitNs, nullptr);
            }
        }
      } else if (warp == kWarpMma || warp == kWarpMma + 1) {
        // ============================================================ MMA issuers
        // Warp 9 issues every MMA of query tile 0, warp 10 those of query tile 1, so the
        // fixed cost of barrier waits and commits on the issuing thread is split in two.
        if (lane == 0) {
            const int i = warp - kWarpMma;  // query tile of this issuer
            int q_uses = 0;                 // items in which this query tile had key tiles
            int tiles = 0;                  // (query tile, key tile) pairs processed
            int s_issued = 0;               // S_i tiles issued so far
            long long g = 0;                // K/V ring position
            bool ok = true;
            const uint32_t d_s = tmem + C::col_s(i);
            const uint32_t d_o = tmem + C::col_o(i);
            const uint32_t a_p = tmem + C::col_p(i);

            // S_i = Q_i K^T from Q buffer q_bar and K stage `stage`.  Descriptors are built
            // once per group and advanced by the byte offset (>> 4) of each 16-wide K step.
            auto issue_s = [&](int q_bar, int stage) {
                const uint64_t a0 = smem_desc(sbase + C::kOffQ + q_bar * C::kTileBytes, 16, C::kAtomBytes, C::kLayout);
                const uint64_t b0 = smem_desc(sbase + C::kOffK + stage * C::kTileBytes, 16, C::kAtomBytes, C::kLayout);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk * 16) / C::kCB * C::kBlkBytes + ((kk * 16) % C::kCB) * 2) >> 4;
                    umma_ss(d_s, a0 + off, b0 + off, C::kIdescS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int stage, bool accumulate) {
                const uint64_t b0 = smem_desc(sbase + C::kOffV + stage * C::kTileBytes, C::kBlkBytes, C::kAtomBytes,
                                              C::kLayout);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    umma_ts(d_o, a_p + 8u * kk, b0 + ((kk * 16 * C::kRowBytes) >> 4), C::kIdescO,
                            (accumulate || kk > 0) ? 1u : 0u);
            };
            // Next S_i.  The S_i columns must have been read by the softmax; with P aliased
            // into them the previous P_i V must also have completed.
            auto do_s = [&](int q_bar, int stage, bool last) -> bool {
                if (C::kAliasP) {
                    if (tiles > 0 && !mbar_wait(bar(kBarPVDone + i), (tiles - 1) & 1, limit, abort_flag)) return false;
                } else {
                    if (s_issued > 0 && !mbar_wait(bar(kBarSFree + i), (s_issued - 1) & 1, limit, abort_flag))
                        return false;
                }
                ++s_issued;
                tc_fence_after_sync();
                issue_s(q_bar, stage);
                umma_commit(bar(kBarSFull + i));
                if (last) umma_commit(bar(kBarQEmpty + q_bar));  // Q_i no longer read
                return true;
            };

            for (ItemCursor cur = first_item(p, CAUSAL && p.pairs, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp); ok && cur.item < p.n_items; next_item(p, cur, CAUSAL && p.pairs, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp)) {
                const Item it = decode_item<SPLIT>(p, cur, CAUSAL, C::kAlternate, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp);
                const int n = i ? it.n[1] : it.n[0];
                const int q_bar = 2 * (q_uses % C::kQBuf) + i;
                if (n > 0 && !mbar_wait(bar(kBarQFull + q_bar), (q_uses / C::kQBuf) & 1, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                for (int j = 0; ok && j < it.n_kv; ++j) {
                    const long long gj = g + j;
                    const int sj = static_cast<int>(gj % S);
                    if (j >= n) {
                        // key tile this query tile does not visit: release the stage once it is loaded
                        if (!mbar_wait(bar(kBarKVFull + sj), static_cast<uint32_t>(gj / S) & 1, limit, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive(bar(kBarKVEmpty + sj));
                        continue;
                    }
                    if (j == 0) {
                        if (!mbar_wait(bar(kBarKVFull + sj), static_cast<uint32_t>(gj / S) & 1, limit, abort_flag) ||
                            !do_s(q_bar, sj, n == 1)) {
                            ok = false;
                            break;
                        }
                    }
                    // Without aliasing, S_i(j+1) only needs S_i(j) read: issue it before P_i(j) V_j,
                    // so that it runs while the softmax of tile j is still exponentiating.
                    if (!C::kAliasP && j + 1 < n) {
                        const long long gn = gj + 1;
                        const int sn = static_cast<int>(gn % S);
                        if (!mbar_wait(bar(kBarKVFull + sn), static_cast<uint32_t>(gn / S) & 1, limit, abort_flag) ||
                            !do_s(q_bar, sn, j + 1 == n - 1)) {
                            ok = false;
                            break;
                        }
                    }
                    // With a correction warpgroup, the first P V of an item (which overwrites O_i)
                    // waits until the correction warps have read the previous item's O_i.
                    if (kWithCorr && j == 0 && q_uses > 0 &&
                        !mbar_wait(bar(kBarOFree + i), (q_uses - 1) & 1, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(bar(kBarPFull + i), tiles & 1, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    issue_pv(sj, j > 0);
                    umma_commit(bar(kBarPVDone + i));
                    if (j == n - 1) umma_commit(bar(kBarOReady + i));
                    umma_commit(bar(kBarKVEmpty + sj));
                    ++tiles;
                    if (C::kAliasP && j + 1 < n) {
                        const long long gn = gj + 1;
                        const int sn = static_cast<int>(gn % S);
                        if (!mbar_wait(bar(kBarKVFull + sn), static_cast<uint32_t>(gn / S) & 1, limit, abort_flag) ||
                            !do_s(q_bar, sn, j + 1 == n - 1)) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (n > 0) ++q_uses;
                g += it.n_kv;
            }
            if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
            // Wait for every tensor-core operation this thread issued.
            umma_commit(bar(kBarDrain + i));
            mbar_wait(bar(kBarDrain + i), 0, kDrainLimitNs, nullptr);
        }
      }
    } else {
        regs_increase<kWithCorr ? kCorrSoftmaxRegs : kSoftmaxRegs<D>>();
        // ============================================================ softmax + epilogue
        const int wg = warp >> 2;               // query tile of this warpgroup
        const int r = threadIdx.x & 127;        // row within the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t t_s = tmem + lane_base + C::col_s(wg);
        const uint32_t t_o = tmem + lane_base + C::col_o(wg);
        const uint32_t t_p = tmem + lane_base + C::col_p(wg);
        const float sl2 = p.scale_log2;
        const int off = p.Nk - p.N;
        int tiles = 0;   // (query tile, key tile) pairs processed by this warpgroup
        int items = 0;   // items in which this warpgroup had key tiles
        int staged = 0;  // output tiles this warpgroup wrote through the staging tile
        bool ok = true;

        for (ItemCursor cur = first_item(p, CAUSAL && p.pairs, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp); ok && cur.item < p.n_items; next_item(p, cur, CAUSAL && p.pairs, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp)) {
            const Item it = decode_item<SPLIT>(p, cur, CAUSAL, C::kAlternate, kOrderedWalk<D, CAUSAL> && p.n_full != p.n_qp);
            const int n = wg ? it.n[1] : it.n[0];
            const int rows = wg ? it.rows[1] : it.rows[0];
            const int row0 = wg ? it.r0[1] : it.r0[0];  // first query row of this tile
            const int qpos = off + row0 + r;
            float m_run = -INFINITY;  // running max of scale*log2(e)*S over visible keys
            float l = 0.f;
            for (int j = 0; j < n; ++j) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + wg), tiles & 1, limit, abort_flag));
                if (!ok) break;
                tc_fence_after_sync();
                uint32_t u[kBlockN];
                // The row's maximum comes reduced by the TMEM loads themselves.  d = 128 loads the
                // row in two 64-column loads (C3-shaped prefill 1000 -> 1036 TFLOP/s against four
                // 32-column ones); d <= 64 keeps four (two measured 0.7 % slower there).
                float mrow;
                float mql[4];  // the load's per-chunk maxima (causal d <= 64)
                if constexpr (D == 128) {
                    float mh[2];
                    tmem_ld64_max(t_s + 0, *reinterpret_cast<uint32_t(*)[64]>(&u[0]), mh[0]);
                    tmem_ld64_max(t_s + 64, *reinterpret_cast<uint32_t(*)[64]>(&u[64]), mh[1]);
                    tmem_ld_wait();
                    mrow = fmaxf(mh[0], mh[1]);
                } else {
                    float mq[4];
                    tmem_ld32_max(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&u[0]), mq[0]);
                    tmem_ld32_max(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]), mq[1]);
                    tmem_ld32_max(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&u[64]), mq[2]);
                    tmem_ld32_max(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&u[96]), mq[3]);
                    tmem_ld_wait();
                    mrow = max3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
                    if constexpr (CAUSAL) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) mql[q] = mq[q];
                    }
                }
                if constexpr (!C::kAliasP) {  // S_i is in registers: its columns may be overwritten
                    tc_fence_before_sync();
                    mbar_arrive(bar(kBarSFree + wg));
                }
                float s[kBlockN];
#pragma unroll
                for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(u[c]);
                const int k0 = (it.j0 + j) * kBlockN;
                const bool need_mask = (k0 + kBlockN > p.Nk) || (CAUSAL && k0 + kBlockN - 1 > off + row0);
                if (CAUSAL && D <= 64 && need_mask) {
                    // Causal, d <= 64: the mask is taken per 32-column chunk, decided for the whole
                    // warp.  A chunk every row of the warp sees keeps its load maximum; a chunk no row
                    // sees is set to -inf (one select per column on the warp-wide test, no maximum);
                    // only the chunk the warp's rows cut is tested column by column.  On a diagonal
                    // tile every warp then masks one chunk instead of four (B=64 H=16 N=1024 d=64
                    // causal prefill 707 -> 716 TFLOP/s).  Hidden scores become -inf rather than being offset, so a
                    // non-finite score in a key a row cannot see never reaches that row; a constant
                    // store in place of the select made the compiler spill the score row.
                    const int lim = min(qpos, p.Nk - 1) - k0;  // columns 0 .. lim visible to this row
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (__all_sync(0xffffffffu, lim < 32 * q)) {
                            float* t = s + 32 * q;
#pragma unroll
                            for (int c = 0; c < 32; ++c) t[c] = lim < 32 * q ? -INFINITY : t[c];
                            mql[q] = -INFINITY;
                        } else if (!__all_sync(0xffffffffu, lim >= 32 * q + 31)) {
                            float* t = s + 32 * q;
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                if (32 * q + c > lim) t[c] = -INFINITY;
                            float a = max3(t[0], t[1], t[2]);
#pragma unroll
                            for (int c = 3; c < 31; c += 2) a = max3(a, t[c], t[c + 1]);
                            mql[q] = fmaxf(a, t[31]);
                        }
                    }
                    mrow = max3(mql[0], mql[1], fmaxf(mql[2], mql[3]));
                } else if (need_mask) {  // diagonal or ragged tile: mask, then take the max in registers
                    const int last = CAUSAL ? min(qpos, p.Nk - 1) : p.Nk - 1;  // last visible key
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        if (k0 + c > last) s[c] = -INFINITY;
                    float mq[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float* t = s + 32 * q;
                        float a = max3(t[0], t[1], t[2]);
#pragma unroll
                        for (int c = 3; c < 31; c += 2) a = max3(a, t[c], t[c + 1]);
                        mq[q] = fmaxf(a, t[31]);
                    }
                    mrow = max3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
                }
                const float mt = mrow * sl2;
                const bool grow = mt > m_run;
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2(m_run - mt);  // 0 when m_run = -inf
                    m_run = mt;
                }
                const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
                // Test now whether P_i(j-1) V_{j-1} has completed; the answer is needed only
                // after the exponentials, so the barrier's latency overlaps them.
                const bool pv_ready = C::kAliasP || j == 0 || mbar_test(bar(kBarPVDone + wg), (tiles - 1) & 1);
                // Packed two-wide FP32 arithmetic (scale-and-subtract, row sums) halves the
                // non-exponential instructions of this loop.
                const float2 sl2x2 = make_float2(sl2, sl2);
                const float2 negm = make_float2(-m_use, -m_use);
                // Four running pairs for the row sum keep its dependency chains short.
                float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                uint32_t pk[kBlockN / 2];
#pragma unroll
                for (int c = 0; c < kBlockN; c += 8) {
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 x = __ffma2_rn(make_float2(s[c + 2 * h], s[c + 2 * h + 1]), sl2x2, negm);
                        const float2 e = make_float2(ex2(x.x), ex2(x.y));
                        rs[h] = __fadd2_rn(rs[h], e);
                        pk[c / 2 + h] = pack_bf16x2(e.x, e.y);
                    }
                }
                // O_i and the P_i columns are free once P_i(j-1) V_{j-1} has completed.  With P
                // aliased into S_i this is implied by the arrival of S_i(j); otherwise wait for it.
                if (!C::kAliasP && j > 0) {
                    ok = __all_sync(0xffffffffu,
                                    pv_ready || mbar_wait(bar(kBarPVDone + wg), (tiles - 1) & 1, limit, abort_flag));
                    if (!ok) break;
                    tc_fence_after_sync();
                }
                if (j > 0 && __any_sync(0xffffffffu, grow)) {
                    // O row times alpha in chunks of kRescale columns: all of them at once for
                    // d <= 64 (one TMEM round trip), 32 at a time for d = 128 (registers).
                    constexpr int kRescale = D <= 64 ? D : 32;
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += kRescale) {
                        uint32_t oc[kRescale];
#pragma unroll
                        for (int c = 0; c < kRescale; c += 32)
                            tmem_ld32(t_o + static_cast<uint32_t>(c0 + c), *reinterpret_cast<uint32_t(*)[32]>(&oc[c]));
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < kRescale; e += 2) {
                            const float2 v = __fmul2_rn(make_float2(__uint_as_float(oc[e]), __uint_as_float(oc[e + 1])), a2);
                            oc[e] = __float_as_uint(v.x);
                            oc[e + 1] = __float_as_uint(v.y);
                        }
#pragma unroll
                        for (int c = 0; c < kRescale; c += 32)
                            tmem_st32(t_o + static_cast<uint32_t>(c0 + c), *reinterpret_cast<uint32_t(*)[32]>(&oc[c]));
                    }
                }
                tmem_st32(t_p + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
                tmem_st32(t_p + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(bar(kBarPFull + wg));
                l = l * alpha + (((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y)) + ((rs[2].x + rs[2].y) + (rs[3].x + rs[3].y)));
                ++tiles;
            }
            if (!ok) break;
            if (rows == 0) continue;  // tile lies past N: nothing to write
            if constexpr (kWithCorr) {
                // Hand 1 / l to the correction warps (once they have read the previous item's),
                // write LSE and move on: the correction warps store O / l.
                if (n > 0) {
                    if (items > 0) {
                        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarOFree + wg), (items - 1) & 1, limit, abort_flag));
                        if (!ok) break;
                    }
                    reinterpret_cast<float*>(smem + C::kOffInvL)[wg * kBlockM + r] = l > 0.f ? 1.f / l : 0.f;
                    mbar_arrive(bar(kBarLFull + wg));
                    ++items;
                }
                if (r < rows) {
                    const size_t row = static_cast<size_t>(it.bh) * p.N + static_cast<size_t>(row0 + r);
                    const float lse = l > 0.f ? (m_run + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
                    if constexpr (SPLIT)
                        p.lse_part[row * p.n_splits + it.split] = lse;
                    else if (p.lse != nullptr)
                        p.lse[row] = lse;
                }
                continue;
            }
            if (n > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarOReady + wg), items & 1, limit, abort_flag));
                if (!ok) break;
                ++items;
                tc_fence_after_sync();
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const size_t row = static_cast<size_t>(it.bh) * p.N + static_cast<size_t>(row0 + r);
            const bool valid = r < rows;
            if constexpr (C::kStoreO && !SPLIT) {
                using OS = OStage<OutT, D>;
                const uint32_t stg = sbase + C::kOffStage + static_cast<uint32_t>(wg) * C::kStageTileBytes;
                // Each warp stages its 32 rows and stores them itself (a 32-row box), so the epilogue
                // needs no barrier across the warpgroup: lane 0 first waits until the warp's previous
                // store has read its rows (issued one item ago, long done).
                const int wq = warp & 3;
                if (lane == 0 && staged > 0) bulk_wait_read_all();
                __syncwarp();
                uint32_t o[D];
                if (n > 0) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld32(t_o + 32u * c, *reinterpret_cast<uint32_t(*)[32]>(&o[32 * c]));
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < D; ++e) o[e] = 0u;
                }
                stage_row<OutT, D>(stg, r, o, inv);
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0 && row0 + 32 * wq < p.N) {  // rows past N lie outside the map and are skipped
#pragma unroll
                    for (int cb = 0; cb < OS::kNumCB; ++cb)
                        tma_store_3d(&p.tm_o, stg + cb * OS::kBlkBytes + wq * 32 * OS::kRowBytes, cb * OS::kElems,
                                     row0 + 32 * wq, it.bh);
                    bulk_commit_group();
                }
                ++staged;
            } else {
                // split mode: this split's slot of the row's fp32 partials
                OutT* orow = SPLIT ? reinterpret_cast<OutT*>(p.o_part) + (row * p.n_splits + it.split) * D
                                   : reinterpret_cast<OutT*>(p.o) + row * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
                    if (n > 0) {
                        uint32_t o[32];
                        tmem_ld32(t_o + 32u * c, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv;
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0.f;
                    }
                    if (valid) {
                        if constexpr (SPLIT)  // partial slots are 512-byte multiples into the aligned workspace
                            store_row32_aligned32(reinterpret_cast<float*>(orow) + 32 * c, v);
                        else
                            store_row32<OutT>(orow + 32 * c, v);
                    }
                }
            }
            if (valid) {
                const float lse = l > 0.f ? (m_run + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
                if constexpr (SPLIT)
                    p.lse_part[row * p.n_splits + it.split] = lse;
                else if (p.lse != nullptr)
                    p.lse[row] = lse;
            }
        }
        // Bulk stores must finish before the CTA's shared memory goes away.
        if (C::kStoreO && lane == 0 && staged > 0) bulk_wait_all();
        if (!ok && !*abort_flag) record_failure(p.status, abort_flag, FA_ERR_TIMEOUT);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool CAUSAL, typename OutT, bool SPLIT = false>
cudaError_t launch_fwd_t(const FwdParams& p, cudaStream_t st)
{
    using C = FwdCfg<D, static_cast<int>(sizeof(OutT))>;
    auto kern = fa_fwd_kernel<D, CAUSAL, OutT, SPLIT>;
    static bool configured[64] = {};  // the shared-memory attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    static int regs[64] = {};  // registers per thread at launch, per device
    if (dev >= 0 && dev < 64 && regs[dev] == 0) {
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, kern);
        if (e != cudaSuccess) return e;
        regs[dev] = attr.numRegs;
    }
    const int launch_regs = (dev >= 0 && dev < 64) ? regs[dev] : 0;
    constexpr bool kWithCorr = kCorr<D, CAUSAL>;
    constexpr int kNeed = kWithCorr ? 256 * kCorrSoftmaxRegs + 128 * (kCorrRegs + kCorrControlRegs)
                                    : 256 * kSoftmaxRegs<D> + 128 * kControlRegs<D>;
    if (launch_regs * kThreads<D, CAUSAL> < kNeed)
        return cudaErrorLaunchOutOfResources;  // the register split would not fit
    FwdParams q = p;
    // Pairs balance causal work over several rounds; with no more items than CTAs every item gets
    // a CTA of its own.  Split items go out singly, in (head, query pair, split) order.
    q.pairs = (!SPLIT && CAUSAL && p.n_items > p.num_ctas) ? 1 : 0;
    const int units = q.pairs ? (p.n_items + 1) / 2 : p.n_items;  // pairs of items, or items
    const int grid = units < p.num_ctas ? units : p.num_ctas;
    const long long step = q.pairs ? 2LL * grid - 1 : grid;  // see next_item
    const int rem_rows = p.N % (2 * kBlockM);
    q.n_full = (!SPLIT && rem_rows > 0 && rem_rows <= kBlockM) ? p.n_qp - 1 : p.n_qp;
    // pairs per head of the walk: n_full in the ordered walk (no mask, one-tile last pairs), else n_qp
    const int per_head = (kOrderedWalk<D, CAUSAL> && q.n_full != p.n_qp) ? (q.n_full > 0 ? q.n_full : 1) : p.n_qp;
    q.step_heads = static_cast<int>(step / per_head);
    q.step_rem = static_cast<int>(step % per_head);
    return launch_pdl(kern, static_cast<unsigned>(grid), kThreads<D, CAUSAL>, C::kSmemBytes, st, q);
}

template <int D>
cudaError_t launch_fwd_d(const FwdParams& p, bool causal, fa_dtype o_dtype, cudaStream_t st)
{
    if (o_dtype == FA_F32)
        return causal ? launch_fwd_t<D, true, float>(p, st) : launch_fwd_t<D, false, float>(p, st);
    return causal ? launch_fwd_t<D, true, __nv_bfloat16>(p, st) : launch_fwd_t<D, false, __nv_bfloat16>(p, st);
}

template <int D>
cudaError_t launch_fwd_split_d(const FwdParams& p, bool causal, cudaStream_t st)
{
    return causal ? launch_fwd_t<D, true, float, true>(p, st) : launch_fwd_t<D, false, float, true>(p, st);
}

}  // namespace fa
