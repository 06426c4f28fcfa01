/*
 * fa.h -- C ABI of libfa: exact tiled attention on GB300 (sm_103a).
 *
 * Operations (page titles and sections they follow):
 *   fa_fwd              exact attention forward, tiled with an online softmax
 *                       ("flash_lab.py -- FlashAttention, flash-decoding and
 *                       megakernel in numpy", section 3 `flash_fwd`, FlashAttention-2
 *                       loop order; the value it reaches is section 2
 *                       `standard_attention`).
 *   fa_decode_splitkv   single-query decode split over the key/value length, each
 *                       split's normalised output and log-sum-exp merged afterwards
 *                       ("flash_lab.py", section 4 `split_kv_decode`).
 *   fa_bwd              gradients dQ, dK, dV of exact attention, P recomputed tile by
 *                       tile from the forward's log-sum-exp ("flash_lab.py", section 3
 *                       `flash_bwd`, FlashAttention-2 form; the value it reaches is
 *                       section 2 `standard_attention_bwd`).
 *   fa_decode_splitkv_gqa  the same with the query heads of a key/value group packed
 *                       together ("flash_lab.py", section 4: GQA packs a group's query heads
 *                       as the rows of q; `decode_attention_time` method "fd").
 *   fa_fwd_splitkv      the forward with the keys split and merged, for few query tiles
 *                       ("flash_lab.py", section 4 applied to a query tile).
 *   fa_decode_splitkv_fused  the decode with the combine done by the last split of each
 *                       (b, h) instead of a second kernel.
 *   fa_merge_states     the log-sum-exp combine of partial states on its own
 *                       ("flash_lab.py", section 4 `split_kv_decode` combine, the
 *                       lse form of section 1 `merge_states`).
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense, row-major, last dimension contiguous, in the layouts
 *     stated per argument ([B,H,rows,cols]).  Device pointers must be 16-byte aligned.
 *   - q, k, v and the caches are bf16.  Arithmetic is fp32 (tensor-core accumulation in
 *     fp32; softmax statistics in fp32).  O is written as bf16 (FA_BF16) or fp32 (FA_F32);
 *     LSE is always fp32, natural log, scale included:
 *       LSE[i] = log sum_{visible j} exp(scale * q_i . k_j).
 *   - Causal masking places query i at position Nk - N + i and key j at position j
 *     ("02_flash_forward.py -- FlashAttention forward", demo 1; "flash_lab.py"
 *     `_causal_mask`).  A query row with no visible key (only when causal and N > Nk)
 *     gets O = 0 and LSE = -inf.
 *   - Ownership: the caller allocates and owns every buffer; the library allocates
 *     nothing.  Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and never synchronise, except
 *     fa_get_device_error.
 *   - Stream order is kept: every kernel is launched with programmatic stream
 *     serialization, so it may start its setup (barriers, tensor memory) while the kernel
 *     before it on `stream` finishes, but it reads and writes global memory only after that
 *     kernel has completed and its writes are visible.  A caller's kernel launched after a
 *     call without that attribute starts once the call's kernels have completed, as usual.
 *   - CUDA graphs: after the first call on a device (which caches kernel attributes and
 *     device addresses), a call launches kernels on `stream` and does nothing else on the
 *     device, so every entry point but fa_get_device_error may be captured into a CUDA
 *     graph and replayed; the tensor maps are encoded at capture time from the pointers
 *     and sizes given, so a replay reads and writes the same buffers.
 *   - Errors: every argument is checked on the host before any launch; a bad argument
 *     returns a status and launches nothing.  A launch failure returns FA_ERR_CUDA.
 *     Failures the device detects (a bounded wait that ran out, a sequence length out
 *     of range) are recorded in a device status word read by fa_get_device_error.
 *   - Supported head sizes: d = dv, d in {32, 64, 128}.  Other sizes return
 *     FA_ERR_UNSUPPORTED.  Heads are independent; the number of key/value heads equals
 *     the number of query heads except in fa_decode_splitkv_gqa.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, misaligned pointer, bad enum */
    FA_ERR_UNSUPPORTED = 2, /* valid arguments this build has no kernel for (head size) */
    FA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    FA_ERR_WORKSPACE = 4,   /* caller-provided workspace smaller than required */
    FA_ERR_TIMEOUT = 5      /* a device-side bounded wait ran out (kernel returned early) */
} fa_status;

typedef enum { FA_BF16 = 0, FA_F32 = 1 } fa_dtype;

/*
 * Exact attention forward ("flash_lab.py" section 3, FlashAttention-2 order): for each
 * (b, h) and query row i,
 *   O[b,h,i,:] = sum_j softmax_j(scale * Q[b,h,i,:] . K[b,h,j,:]) V[b,h,j,:]
 * over the visible keys j (all Nk keys, or j <= Nk - N + i when causal), and
 *   lse[b,h,i] = log sum_j exp(scale * Q[b,h,i,:] . K[b,h,j,:]).
 * The N x Nk score matrix never reaches memory.
 *
 *   q    bf16 [B, H, N,  d]        (device)
 *   k    bf16 [B, H, Nk, d]        (device)
 *   v    bf16 [B, H, Nk, dv]       (device)
 *   o    o_dtype [B, H, N, dv]     (device, written)
 *   lse  fp32 [B, H, N]            (device, written; may be NULL to skip it)
 *   B, H, N, Nk >= 1; d = dv in {32, 64, 128}; causal 0 or 1; scale > 0 and finite
 *   (1/sqrt(d) is the usual value); B*H*ceil(N/256) < 2^30 (else FA_ERR_INVALID_ARG).
 * Returns FA_OK after enqueueing the kernel on `stream`.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int Nk, int d, int dv, int causal, float scale, fa_dtype o_dtype,
                 void* stream);

/*
 * Bytes of workspace fa_bwd needs: with Tr = ceil(N / 128), an fp32 dQ accumulator of
 * B*H*Tr*128*d values, then fp32 base-2 log-sum-exps and fp32 scaled row terms of
 * B*H*Tr*128 values each, every region 256-byte aligned.  Returns 0 on invalid arguments.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Exact attention backward ("flash_lab.py" section 3 `flash_bwd`).  For the upstream
 * gradient dO of the forward's output O, with P the attention weights of fa_fwd (same
 * mask and scale) and D_i = sum_c dO[i,c] O[i,c]:
 *   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dQ = dS K scale,  dK = dS^T Q scale
 * for every (b, h).  P is recomputed tile by tile as exp(scale q.k - lse); it never reaches
 * memory.  Rows with no visible key (lse = -inf) contribute nothing.
 *
 *   q, k, v      bf16 [B, H, N, d], [B, H, Nk, d], [B, H, Nk, dv]  (device; the forward inputs)
 *   o            o_dtype [B, H, N, dv]   (device; the forward output, used only for D)
 *   lse          fp32 [B, H, N]          (device; the forward's log-sum-exp)
 *   grad_o       bf16 [B, H, N, dv]      (device; dO)
 *   grad_q, grad_k, grad_v   grad_dtype [B, H, N, d], [B, H, Nk, d], [B, H, Nk, dv]
 *                (device, written; every element is written)
 *   workspace    device scratch of ws_bytes >= fa_bwd_workspace_size(B, H, N, d) bytes,
 *                256-byte aligned; its contents on entry do not matter.
 *   B, H, N, Nk >= 1; d = dv in {32, 64, 128}; causal 0 or 1; scale > 0 and finite, the
 *   value the forward used; B*H*ceil(Nk/128) < 2^30 (else FA_ERR_INVALID_ARG).
 * Three kernels are enqueued on `stream`: a preparation pass (D, lse in base 2, zeroing the
 * dQ accumulator), the tensor-core pass (a persistent grid, one CTA per SM, walking the
 * (b, h, 128-key tile) items; each item's dK and dV written when its walk ends, dQ added into
 * the accumulator) and the dQ conversion.
 * The key tiles' shares of dQ are added into the fp32 accumulator by the memory system in
 * whatever order the CTAs reach it, so grad_q can differ in its last bits from run to run;
 * grad_k and grad_v are summed on chip in a fixed order and are reproducible.
 * Returns FA_ERR_WORKSPACE if ws_bytes is too small (nothing launched).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* grad_o, void* grad_q, void* grad_k, void* grad_v, void* workspace,
                 size_t ws_bytes, int B, int H, int N, int Nk, int d, int dv, int causal,
                 float scale, fa_dtype o_dtype, fa_dtype grad_dtype, void* stream);

/*
 * Split count fa_decode_splitkv uses when asked for n_splits = 0, for a device with
 * `num_sms` streaming multiprocessors: enough splits of the longest sequence that the
 * non-empty (b, h, split) work items fill the device several times over, each split at
 * least one key block long.  Pure host function.  Returns 0 on invalid arguments.
 */
int fa_decode_default_splits(int B, int H, int Nk_max, int num_sms);

/*
 * Bytes of workspace fa_decode_splitkv needs for `n_splits` splits (n_splits >= 1):
 * fp32 partial outputs [B, H, n_splits, dv] followed by fp32 partial log-sum-exps
 * [B, H, n_splits], each region 256-byte aligned.  Returns 0 on invalid arguments.
 */
size_t fa_decode_workspace_size(int B, int H, int dv, int n_splits);

/*
 * Split-KV single-query decode ("flash_lab.py" section 4 `split_kv_decode`).  For each
 * (b, h), the first seqlens_k[b] cached keys are cut into n_splits consecutive chunks of
 * c = ceil(Nk_max / n_splits) keys (rounded up to the kernel's key block); split s covers
 * keys [s*c, min((s+1)*c, seqlens_k[b])) and is empty when that range is.  Each non-empty
 * split writes its normalised output o_s and lse_s to the workspace; a second kernel merges
 *   lse = log sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s.
 * The single query sits at position seqlens_k[b] - 1 and sees every cached key.
 *
 *   q          bf16 [B, H, 1, d]          (device)
 *   k_cache    bf16 [B, H, Nk_max, d]     (device; rows past seqlens_k[b] are never read)
 *   v_cache    bf16 [B, H, Nk_max, dv]    (device; idem)
 *   seqlens_k  int32 [B]                  (device; 0 <= seqlens_k[b] <= Nk_max.  Values
 *              outside that range are clamped into it and recorded as FA_ERR_INVALID_ARG in
 *              the device status word.  A length of 0 gives O = 0, LSE = -inf.)
 *   o          o_dtype [B, H, 1, dv]      (device, written)
 *   lse        fp32 [B, H, 1]             (device, written; may be NULL)
 *   workspace  device scratch of ws_bytes >= fa_decode_workspace_size(B, H, dv, n) bytes,
 *              256-byte aligned, where n is n_splits or, for n_splits = 0, the automatic
 *              count fa_decode_default_splits(B, H, Nk_max, <SMs of the current device>).
 *   n_splits   >= 0; 0 picks the automatic count.  Values above Nk_max are reduced to it.
 * Returns FA_ERR_WORKSPACE if ws_bytes is too small (nothing launched).
 */
fa_status fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                            const int* seqlens_k, void* o, float* lse, void* workspace,
                            size_t ws_bytes, int B, int H, int Nk_max, int d, int dv, float scale,
                            int n_splits, fa_dtype o_dtype, void* stream);

/*
 * Split count fa_decode_splitkv_gqa uses when asked for n_splits = 0, for Hq query heads over Hkv
 * key/value heads of head size d on a device with `num_sms` multiprocessors.  Groups of
 * R = Hq / Hkv = 1 or 2 heads, and of 4 heads at d != 128, run on CUDA cores and take
 * fa_decode_default_splits(B, Hq, Nk_max, num_sms).  Other groups (tensor core) take
 * floor(1.7 * c * num_sms / (B * Hkv)) splits, where c = 2 for 3 to 8 heads at d = 128 (two CTAs
 * per multiprocessor) and 1 otherwise; raised to 2 while B * Hkv < 2 * num_sms, then to
 * ceil(ceil(Nk_max / 128) / T) with T = 64 key tiles for R <= 4 and 32 otherwise (no split
 * longer than T tiles), then clamped to [1, ceil(Nk_max / 128)].  Pure host function.  Returns 0
 * on invalid arguments (a non-positive size, or Hkv not dividing Hq).
 */
int fa_decode_gqa_default_splits(int B, int Hq, int Hkv, int Nk_max, int d, int num_sms);

/*
 * Split-KV decode with grouped key/value heads (GQA): Hq query heads share Hkv key/value heads,
 * query head h reading key/value head h / R with R = Hq / Hkv.  The R query heads of a group are
 * packed together ("flash_lab.py" section 4 `split_kv_decode`, q of shape [R, d]; section 4
 * `decode_attention_time`, method "fd": one work item per (b, key/value head, split), K and V read
 * once per group), so each cached key and value is read from memory once for all R heads.  The
 * split, merge, arguments and errors are those of fa_decode_splitkv, with:
 *
 *   q          bf16 [B, Hq, 1, d]          (device)
 *   k_cache    bf16 [B, Hkv, Nk_max, d]    (device)
 *   v_cache    bf16 [B, Hkv, Nk_max, dv]   (device)
 *   o          o_dtype [B, Hq, 1, dv]      (device, written)
 *   lse        fp32 [B, Hq, 1]             (device, written; may be NULL)
 *   workspace  ws_bytes >= fa_decode_workspace_size(B, Hq, dv, n) bytes, where n is n_splits or,
 *              for n_splits = 0, fa_decode_gqa_default_splits(B, Hq, Hkv, Nk_max, d, <SMs of the
 *              device>).
 *   Hkv >= 1 dividing Hq, R = Hq / Hkv <= 128 (larger groups return FA_ERR_UNSUPPORTED).
 *   Hkv = Hq is fa_decode_splitkv.  Groups of 1 or 2 heads, and of 4 heads at d != 128, run on
 *   CUDA cores; other group sizes on the tensor core (3 to 32 heads at d = 128 with the product
 *   transposed, keys on the tensor-memory lanes; otherwise the R query rows are the rows of a
 *   128-row tile), where splits are whole 128-key tiles (the chunk is rounded up to a multiple of
 *   128 instead of the key block) and cache rows past a sequence's length are never used,
 *   whatever they hold.
 */
fa_status fa_decode_splitkv_gqa(const void* q, const void* k_cache, const void* v_cache,
                                const int* seqlens_k, void* o, float* lse, void* workspace,
                                size_t ws_bytes, int B, int Hq, int Hkv, int Nk_max, int d, int dv,
                                float scale, int n_splits, fa_dtype o_dtype, void* stream);

/*
 * Bytes of workspace fa_decode_splitkv_fused needs: fa_decode_workspace_size(B, H, dv, n_splits)
 * followed by B*H 32-bit arrival counters (256-byte aligned).  0 on invalid arguments.
 */
size_t fa_decode_fused_workspace_size(int B, int H, int dv, int n_splits);

/*
 * fa_decode_splitkv with the combine fused into the split kernel: every non-empty split of a
 * (b, h) writes its o_s, lse_s and then counts itself on a per-(b, h) counter; the split that
 * arrives last merges the row ("flash_lab.py" section 4 combine), so one kernel is launched
 * instead of two (the launch gap is a decode cost the pages single out, section 5).  Same
 * arguments, checks and result as fa_decode_splitkv, except:
 *   workspace  ws_bytes >= fa_decode_fused_workspace_size(B, H, dv, n) bytes.  Its counter region
 *              (the last B*H*4 bytes of that size) must be zero before the first call that uses
 *              this workspace; every call that completes leaves it zero again.  After a call that
 *              failed on the device (fa_get_device_error != FA_OK) zero it again.  Calls sharing a
 *              workspace must not overlap on the GPU.
 */
fa_status fa_decode_splitkv_fused(const void* q, const void* k_cache, const void* v_cache,
                                  const int* seqlens_k, void* o, float* lse, void* workspace,
                                  size_t ws_bytes, int B, int H, int Nk_max, int d, int dv, float scale,
                                  int n_splits, fa_dtype o_dtype, void* stream);

/*
 * Split count fa_fwd_splitkv uses for n_splits = 0 on a device with `num_sms` multiprocessors:
 * the largest count for which the B*H*ceil(N/256) pairs of query tiles times the splits fit one
 * persistent CTA per multiprocessor (one round), at least 1 and at most ceil(Nk/128) (each split
 * at least one 128-key tile).  Pure host function; 0 on invalid arguments.
 */
int fa_fwd_splitkv_default_splits(int B, int H, int N, int Nk, int num_sms);

/*
 * Bytes of workspace fa_fwd_splitkv needs for n_splits splits: fp32 partial outputs
 * [B, H, N, n_splits, dv] then fp32 partial log-sum-exps [B, H, N, n_splits], each region
 * 256-byte aligned.  0 on invalid arguments.
 */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int dv, int n_splits);

/*
 * Exact attention forward with the keys split ("flash_lab.py" section 4 `split_kv_decode`
 * applied to a query tile): for workloads with few 128-row query tiles (B*H*ceil(N/256) pairs
 * of them below the number of multiprocessors) the keys are cut into chunks of whole 128-key
 * tiles (ceil(ceil(Nk/128) / n_splits) tiles each; chunks past the keys are dropped); the
 * forward kernel computes each (head, query tile pair, chunk)'s normalised output and
 * log-sum-exp, and a second kernel merges them.  Same arguments, masks, result and output
 * conventions as fa_fwd, plus:
 *   workspace  ws_bytes >= fa_fwd_splitkv_workspace_size(B, H, N, dv, n) bytes, 256-byte aligned,
 *              where n is n_splits or, for 0, fa_fwd_splitkv_default_splits(B, H, N, Nk, <SMs>);
 *   n_splits   >= 0; values above Nk are reduced to it.
 * B*H*N must be below 2^31 and B*H*ceil(N/256)*chunks below 2^30.  Returns FA_ERR_WORKSPACE if
 * ws_bytes is too small (nothing launched).
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         void* workspace, size_t ws_bytes, int B, int H, int N, int Nk, int d, int dv,
                         int causal, float scale, int n_splits, fa_dtype o_dtype, void* stream);

/*
 * Bytes of device scratch that fa_decode_splitkv_noalloc owns (8 MiB): room for the split
 * partials of B*H*n_splits*(dv+1) fp32 values, e.g. B=16, H=32, dv=128 with up to 30 splits.
 */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * fa_decode_splitkv without a workspace argument: the same computation, arguments, checks and
 * result, but the split partials go to a fixed scratch array of FA_DECODE_NOALLOC_SCRATCH_BYTES
 * that the library keeps in device memory (every GPU that loads the library holds it until the
 * process exits).  The pages have no counterpart; it exists for callers that cannot allocate
 * device memory: code whose memory belongs to another allocator (a framework's caching allocator,
 * a serving engine's fixed pool) and may not call cudaMalloc behind its back, code under a hard
 * per-process memory budget, and code that must not risk the device-wide synchronisation that
 * cudaMalloc and cudaFree can cause.  It allocates nothing and calls no allocating routine.
 *
 *   - Size limit: returns FA_ERR_WORKSPACE, launching nothing, when
 *     fa_decode_workspace_size(B, H, dv, n) exceeds FA_DECODE_NOALLOC_SCRATCH_BYTES, where n is
 *     n_splits or, for n_splits = 0, the automatic count.  Use fewer splits, or
 *     fa_decode_splitkv with a workspace of your own, for larger problems.
 *   - Set-up: the first call on each device looks up the scratch array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make that first call
 *     before any stream capture.  A failed look-up returns FA_ERR_CUDA.
 *   - Sharing: every call on a device uses the same array, which keeps the last call's contents.
 *     Nothing in it needs to start at zero (each non-empty split writes its slot before the
 *     combine reads it, and empty splits are never read).  Calls whose kernels overlap on the GPU
 *     (concurrent streams, or several host threads) race on the array: order them on one stream.
 */
fa_status fa_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    const int* seqlens_k, void* o, float* lse, int B, int H,
                                    int Nk_max, int d, int dv, float scale, int n_splits,
                                    fa_dtype o_dtype, void* stream);

/*
 * Log-sum-exp combine of n_parts partial attention states per row ("flash_lab.py"
 * section 4 combine; section 1 `merge_states`, where a state with lse = -inf is empty and
 * gets weight 0):
 *   lse[r] = log sum_p exp(lse_parts[p, r]),  o[r, :] = sum_p exp(lse_parts[p, r] - lse[r]) o_parts[p, r, :]
 * A row whose every part is empty gets o = 0, lse = -inf.
 *
 *   o_parts    fp32 [n_parts, rows, dv]   (device)
 *   lse_parts  fp32 [n_parts, rows]       (device)
 *   o          o_dtype [rows, dv]         (device, written)
 *   lse        fp32 [rows]                (device, written; may be NULL)
 *   n_parts >= 1, rows >= 1, 1 <= dv <= 512.
 */
fa_status fa_merge_states(const float* o_parts, const float* lse_parts, int n_parts, int rows,
                          int dv, void* o, float* lse, fa_dtype o_dtype, void* stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of the current
 * device: FA_OK if no kernel recorded a failure since the last call, else the first
 * recorded status (FA_ERR_TIMEOUT, FA_ERR_INVALID_ARG).  FA_ERR_CUDA if the synchronisation
 * itself failed.
 */
fa_status fa_get_device_error(void* stream);

/*
 * Upper bound, in nanoseconds of the GPU global timer, on every wait for a barrier inside
 * the forward and backward tensor-core kernels (default 2e9).  When a wait runs out the kernel records FA_ERR_TIMEOUT,
 * drains its own copies in flight, frees its tensor memory and returns.  0 restores the
 * default.  Applies to launches made after the call.
 */
void fa_set_wait_timeout_ns(unsigned long long ns);

/* Static description of a status code. */
const char* fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
