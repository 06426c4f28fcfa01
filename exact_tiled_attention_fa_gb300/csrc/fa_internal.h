// fa_internal.h -- parameter blocks and launchers shared by the C-ABI layer and
// the kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Forward kernel tile: 128 query rows (the tcgen05 M) x 128 keys.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;

struct FwdParams {
    CUtensorMap tm_q;  // bf16 [B*H][N][d], box {min(d,64), 128, 1}
    CUtensorMap tm_k;  // bf16 [B*H][Nk][d]
    CUtensorMap tm_v;  // bf16 [B*H][Nk][dv]
    CUtensorMap tm_o;  // O [B*H][N][dv] (bf16 or fp32), box {128 bytes of a row (64 for bf16 d = 32), 32, 1}
    void* o;           // [B*H][N][dv], bf16 or fp32
    float* lse;        // [B*H][N] or nullptr
    int* status;       // device status word
    int BH, N, Nk;
    int n_qp;           // query tile pairs per head: ceil(N / 256)
    int n_items;        // BH * n_qp work items
    int num_ctas;       // persistent CTAs (one per SM)
    float scale_log2;   // scale * log2(e)
    unsigned long long wait_limit_ns;
    // set by the launcher from its grid size G: the step between a CTA's item rounds (G items
    // without a causal mask, 2G - 1 from the second item of a pair under one) as whole heads
    // and a remainder, so that the kernel advances (head, position) without a division
    int step_heads, step_rem;
    int pairs;          // items go out in heavy/light pairs (causal, more items than CTAs) or singly
    // Without a mask: pairs per head with rows in both query tiles (all but a last pair of at most
    // 128 rows).  Items 0 .. BH * n_full - 1 are those pairs, head-major; the BH one-tile last
    // pairs (if any) come after them, so that they fill the last round instead of lengthening it.
    int n_full;
    // Split mode (fa_fwd_splitkv): the keys are cut into n_splits ranges of split_tiles key
    // tiles, an item is (head, query pair, split), n_qp counts the (query pair, split) items of a
    // head (pair-major), and each item writes its rows' normalised partial O (fp32) and natural-log
    // LSE to o_part [B*H*N][n_splits][dv] and lse_part [B*H*N][n_splits] instead of o / lse.
    int n_splits, split_tiles;
    float* o_part;
    float* lse_part;
};

// Launch the forward kernel for head size d (= dv), causal flag and output type.
cudaError_t launch_fwd(const FwdParams& p, int d, bool causal, fa_dtype o_dtype, cudaStream_t st);
// The same kernel in split mode (fp32 partials; FwdParams::n_splits, split_tiles, o_part, lse_part).
cudaError_t launch_fwd_split(const FwdParams& p, int d, bool causal, cudaStream_t st);

// Backward.  Work item: one head and one 128-key tile; the CTA walks every query tile
// that sees a key of it.  Per-row vectors and the dQ accumulator are padded to whole
// query tiles (Tr * 128 rows per head).
struct BwdParams {
    CUtensorMap tm_q;   // bf16 [B*H][N][d], box {min(d,64), 128, 1}
    CUtensorMap tm_k;   // bf16 [B*H][Nk][d]
    CUtensorMap tm_v;   // bf16 [B*H][Nk][d]
    CUtensorMap tm_do;  // bf16 [B*H][N][d]
    CUtensorMap tm_dk;  // dK [B*H][Nk][d] (gradient dtype), box {128 bytes of a row (64 for bf16 d = 32), 128, 1}
    CUtensorMap tm_dv;  // dV, the same
    const float* lse2;  // [B*H][Tr*128]: LSE * log2(e); +inf past N and where no key is visible
    const float* dsc;   // [B*H][Tr*128]: scale * sum_c dO[c] O[c]; 0 past N
    float* dq_acc;      // [B*H][Tr] tiles of 128 x d fp32 (layout: see dq_bulk), zeroed before the kernel
    void* dk;           // [B*H][Nk][d], gradient dtype
    void* dv;           // [B*H][Nk][d]
    int* status;
    int BH, N, Nk, Tr, Tc;
    int num_ctas;       // persistent CTAs (one per SM)
    float scale_log2;   // scale * log2(e)
    float scale;
    unsigned long long wait_limit_ns;
    // set by the launcher from its grid size G: G = step_heads * Tc + step_jr, and step_heads mod Tc
    // (the causal rotation), so that the kernel advances its items without a division
    int step_heads, step_jr, step_rot;
};

#ifndef FA_DQ_BULK
#define FA_DQ_BULK 1
#endif
// d <= 64: the tensor-core kernel adds its dQ tiles into the accumulator with bulk reductions from
// shared memory, and the accumulator of a (head, query tile) is laid out [row quarter w][d/4][32][4]
// (row q: w = q / 32, lane q mod 32), so that each warp's 16-column block is 2 KB contiguous.
// d = 128 (no shared memory left for the staging) keeps vector atomics and the [d/4][128][4] layout.
constexpr bool dq_bulk(int d) { return FA_DQ_BULK != 0 && d <= 64; }

struct BwdPrepParams {
    const void* o;      // [B*H][N][d], bf16 or fp32 (forward output)
    const void* d_o;    // bf16 [B*H][N][d]
    const float* lse;   // [B*H][N] (forward output, natural log)
    float* lse2;
    float* dsc;
    float* dq_acc;
    int BH, N, Tr, d;
    float scale;
};

struct BwdDqParams {
    const float* dq_acc;
    void* dq;           // [B*H][N][d], gradient dtype
    int BH, N, Tr, d;
};

cudaError_t launch_bwd(const BwdParams& p, int d, bool causal, fa_dtype grad_dtype, cudaStream_t st);
cudaError_t launch_bwd_prep(const BwdPrepParams& p, fa_dtype o_dtype, cudaStream_t st);
cudaError_t launch_bwd_dq(const BwdDqParams& p, fa_dtype grad_dtype, cudaStream_t st);

// Split-KV on the tensor core: one CTA per (key split, 128-row query tile, group).  A group is
// a head (prefill: its N query rows) or a key/value head with its R packed query heads (decode).
struct SplitParams {
    CUtensorMap tm_q;   // bf16 [n_groups][rows_per_group][d], box {min(d,64), 128, 1}
    CUtensorMap tm_k;   // bf16 [n_groups][Nk][d]
    CUtensorMap tm_v;   // bf16 [n_groups][Nk][d]
    float* o_part;      // [n_groups * rows_per_group][n_splits][d] fp32
    float* lse_part;    // [n_groups * rows_per_group][n_splits] fp32
    const int* seqlens; // decode: keys per sequence (group / groups_per_batch); nullptr: Nk for all
    int* status;
    int n_groups, rows_per_group, n_qtiles, groups_per_batch;
    int Nk, n_splits, chunk;  // chunk: keys per split, a multiple of 128
    int causal_off;           // Nk - N: query row i sits at position causal_off + i
    float scale_log2;
    unsigned long long wait_limit_ns;
};

cudaError_t launch_splitkv(const SplitParams& p, int d, bool causal, bool varlen, cudaStream_t st);

// Decode: keys per block of the split kernel's inner loop; a split is a whole
// number of such blocks.
constexpr int kDecodeKeyBlock = 64;

struct DecodeParams {
    const void* q;        // bf16 [B*H][d]
    const void* k;        // bf16 [B*Hkv][Nk_max][d]
    const void* v;        // bf16 [B*Hkv][Nk_max][dv]
    const int* seqlens;   // int32 [B]
    float* o_part;        // fp32 [B*H][n_splits][dv]
    float* lse_part;      // fp32 [B*H][n_splits]
    void* o;              // [B*H][dv]
    float* lse;           // [B*H] or nullptr
    int* status;
    int B, H, Nk_max, n_splits, chunk;
    int Hkv;              // key/value heads; query head h reads key/value head h / (H / Hkv)
    float scale_log2;
    // Fused combine: non-null = per-(b, key/value head) arrival counters (zero on entry, left
    // zero); the last split CTA of a (b, key/value head) merges its rows into o / lse.
    unsigned int* counters;
    fa_dtype o_dtype;
};

cudaError_t launch_decode(const DecodeParams& p, int d, fa_dtype o_dtype, cudaStream_t st);

struct MergeParams {
    const float* o_parts;   // partial outputs
    const float* lse_parts; // partial log-sum-exps
    long long o_part_stride, o_row_stride;     // elements between parts / rows of o_parts
    long long lse_part_stride, lse_row_stride; // elements between parts / rows of lse_parts
    int n_parts, rows, dv;
    // optional per-row count of valid parts: ceil(clamp(seqlens[row / H]) / chunk)
    const int* seqlens;
    int H, chunk, Nk_max;
    void* o;     // [rows][dv]
    float* lse;  // [rows] or nullptr
    int* status;
};

cudaError_t launch_merge(const MergeParams& p, fa_dtype o_dtype, cudaStream_t st);

// Status word helpers (device side records the first failure only).
enum : int { kStatusOk = 0 };

}  // namespace fa
