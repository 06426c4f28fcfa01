// fa_api.cu -- the C ABI (include/fa.h): argument checks, TMA tensor maps,
// workspace layout and kernel dispatch.  Host code only.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_internal.h"

namespace fa {
cudaError_t launch_fwd_32(const FwdParams& p, bool causal, fa_dtype o_dtype, cudaStream_t st);
cudaError_t launch_fwd_64(const FwdParams& p, bool causal, fa_dtype o_dtype, cudaStream_t st);
cudaError_t launch_fwd_128(const FwdParams& p, bool causal, fa_dtype o_dtype, cudaStream_t st);

cudaError_t launch_fwd(const FwdParams& p, int d, bool causal, fa_dtype o_dtype, cudaStream_t st)
{
    switch (d) {
    case 32: return launch_fwd_32(p, causal, o_dtype, st);
    case 64: return launch_fwd_64(p, causal, o_dtype, st);
    case 128: return launch_fwd_128(p, causal, o_dtype, st);
    default: return cudaErrorInvalidValue;
    }
}
cudaError_t launch_fwd_split_32(const FwdParams& p, bool causal, cudaStream_t st);
cudaError_t launch_fwd_split_64(const FwdParams& p, bool causal, cudaStream_t st);
cudaError_t launch_fwd_split_128(const FwdParams& p, bool causal, cudaStream_t st);

cudaError_t launch_fwd_split(const FwdParams& p, int d, bool causal, cudaStream_t st)
{
    switch (d) {
    case 32: return launch_fwd_split_32(p, causal, st);
    case 64: return launch_fwd_split_64(p, causal, st);
    case 128: return launch_fwd_split_128(p, causal, st);
    default: return cudaErrorInvalidValue;
    }
}
cudaError_t launch_splitkv_32(const SplitParams& p, bool causal, bool varlen, cudaStream_t st);
cudaError_t launch_splitkv_64(const SplitParams& p, bool causal, bool varlen, cudaStream_t st);
cudaError_t launch_splitkv_128(const SplitParams& p, bool causal, bool varlen, cudaStream_t st);

cudaError_t launch_gqa_tc(const SplitParams& p, cudaStream_t st);

cudaError_t launch_splitkv(const SplitParams& p, int d, bool causal, bool varlen, cudaStream_t st)
{
    switch (d) {
    case 32: return launch_splitkv_32(p, causal, varlen, st);
    case 64: return launch_splitkv_64(p, causal, varlen, st);
    case 128: return launch_splitkv_128(p, causal, varlen, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_32(const BwdParams& p, bool causal, fa_dtype grad_dtype, cudaStream_t st);
cudaError_t launch_bwd_64(const BwdParams& p, bool causal, fa_dtype grad_dtype, cudaStream_t st);
cudaError_t launch_bwd_128(const BwdParams& p, bool causal, fa_dtype grad_dtype, cudaStream_t st);

cudaError_t launch_bwd(const BwdParams& p, int d, bool causal, fa_dtype grad_dtype, cudaStream_t st)
{
    switch (d) {
    case 32: return launch_bwd_32(p, causal, grad_dtype, st);
    case 64: return launch_bwd_64(p, causal, grad_dtype, st);
    case 128: return launch_bwd_128(p, causal, grad_dtype, st);
    default: return cudaErrorInvalidValue;
    }
}
}  // namespace fa

namespace {

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

// Device status word: kernels record the first failure they detect here.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

cudaError_t current_device(int* dev)
{
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
    return cudaSuccess;
}

// Per-device facts looked up once (under a lock) and then read from a per-thread copy, so that
// a call takes no lock.
thread_local int* t_status_ptr[kMaxDevices] = {};
thread_local int t_num_sms[kMaxDevices] = {};

// Device address of the status word on the current device (looked up once per device).
cudaError_t status_word(int** out)
{
    int dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    if (t_status_ptr[dev] == nullptr) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_status_ptr[dev] == nullptr) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_device_status);
            if (e != cudaSuccess) return e;
            g_status_ptr[dev] = static_cast<int*>(p);
        }
        t_status_ptr[dev] = g_status_ptr[dev];
    }
    *out = t_status_ptr[dev];
    return cudaSuccess;
}

cudaError_t sm_count(int* out)
{
    int dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    if (t_num_sms[dev] == 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_num_sms[dev] == 0) {
            e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
        }
        t_num_sms[dev] = g_num_sms[dev];
    }
    *out = t_num_sms[dev];
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A tensor map is a pure function of (address, sizes, element type, box): encoding one costs on
// the order of a microsecond of host time, a visible share of a short call.  Each host thread
// keeps the last kMapCache maps it encoded and reuses one whose key matches (device addresses are
// unique across the process's devices, so the key needs no device).
struct MapKey {
    const void* ptr;
    int BH, rows, d, kind, box_rows;  // kind: 0 bf16 input, 1 bf16 output, 2 fp32 output
    bool operator==(const MapKey& o) const
    {
        return ptr == o.ptr && BH == o.BH && rows == o.rows && d == o.d && kind == o.kind && box_rows == o.box_rows;
    }
};
constexpr int kMapCache = 16;
struct MapCache {
    MapKey key[kMapCache];
    CUtensorMap map[kMapCache];
    bool used[kMapCache] = {};
    int next = 0;
    bool find(const MapKey& k, CUtensorMap* m) const
    {
        for (int i = 0; i < kMapCache; ++i)
            if (used[i] && key[i] == k) {
                *m = map[i];
                return true;
            }
        return false;
    }
    void put(const MapKey& k, const CUtensorMap& m)
    {
        key[next] = k;
        map[next] = m;
        used[next] = true;
        next = (next + 1) % kMapCache;
    }
};
thread_local MapCache t_maps;

bool encode_map(CUtensorMap* m, const void* ptr, int BH, int rows, int d, int box_rows);
bool encode_out_map(CUtensorMap* m, void* ptr, int BH, int rows, int d, fa_dtype t, int box_rows);

// bf16 input tensor [BH][rows][d] (see encode_map), from the thread's cache when possible.
bool make_map(CUtensorMap* m, const void* ptr, int BH, int rows, int d, int box_rows = fa::kBlockM)
{
    const MapKey k{ptr, BH, rows, d, 0, box_rows};
    if (t_maps.find(k, m)) return true;
    if (!encode_map(m, ptr, BH, rows, d, box_rows)) return false;
    t_maps.put(k, *m);
    return true;
}

// Output tensor map (see encode_out_map), from the thread's cache when possible.
bool make_out_map(CUtensorMap* m, void* ptr, int BH, int rows, int d, fa_dtype t, int box_rows)
{
    const MapKey k{ptr, BH, rows, d, t == FA_F32 ? 2 : 1, box_rows};
    if (t_maps.find(k, m)) return true;
    if (!encode_out_map(m, ptr, BH, rows, d, t, box_rows)) return false;
    t_maps.put(k, *m);
    return true;
}

// bf16 tensor [BH][rows][d] as a 3-D tiled map with a {min(d,64), box_rows, 1} box,
// swizzled so that each box row is one swizzle span (64 or 128 bytes).
bool encode_map(CUtensorMap* m, const void* ptr, int BH, int rows, int d, int box_rows)
{
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    const int cb = d < 64 ? d : 64;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows) * d * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(cb), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     cb == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output tensor [BH][rows][d] of bf16 or fp32 as a 3-D tiled map for bulk stores: the box is
// box_rows rows of one column block (128 bytes of a row, or the whole 64-byte row of bf16 d = 32),
// swizzled to match the staging tiles the kernels write (the forward stores 32-row quarters, one
// per warp; the backward whole 128-row tiles).
bool encode_out_map(CUtensorMap* m, void* ptr, int BH, int rows, int d, fa_dtype t, int box_rows)
{
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    const int es = t == FA_F32 ? 4 : 2;
    const int blk = d * es < 128 ? d : 128 / es;  // elements per box row
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es, static_cast<cuuint64_t>(rows) * d * es};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(blk), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, t == FA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     blk * es == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool head_ok(int d) { return d == 32 || d == 64 || d == 128; }
bool dtype_ok(fa_dtype t) { return t == FA_BF16 || t == FA_F32; }
bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

constexpr size_t kAlign = 256;
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s)
{
    switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_WORKSPACE: return "workspace too small";
    case FA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

void fa_set_wait_timeout_ns(unsigned long long ns) { g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns); }

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int Nk,
                 int d, int dv, int causal, float scale, fa_dtype o_dtype, void* stream)
{
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || N <= 0 || Nk <= 0 || d <= 0 || dv <= 0) return FA_ERR_INVALID_ARG;
    if ((causal != 0 && causal != 1) || !dtype_ok(o_dtype) || !scale_ok(scale)) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return FA_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    const long long n_qp = (static_cast<long long>(N) + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
    // the kernels index items with 32-bit ints and step past the last one by up to 2 * SMs
    if (BH * n_qp > 0x3fffffffLL) return FA_ERR_INVALID_ARG;
    if (!head_ok(d) || dv != d) return FA_ERR_UNSUPPORTED;

    fa::FwdParams p{};
    p.n_splits = 1;
    if (!make_map(&p.tm_q, q, static_cast<int>(BH), N, d) || !make_map(&p.tm_k, k, static_cast<int>(BH), Nk, d) ||
        !make_map(&p.tm_v, v, static_cast<int>(BH), Nk, dv) ||
        !make_out_map(&p.tm_o, o, static_cast<int>(BH), N, dv, o_dtype, 32))
        return FA_ERR_CUDA;
    int* status = nullptr;
    if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return FA_ERR_CUDA;
    p.o = o;
    p.lse = lse;
    p.status = status;
    p.BH = static_cast<int>(BH);
    p.N = N;
    p.Nk = Nk;
    p.n_qp = static_cast<int>(n_qp);
    p.n_items = static_cast<int>(BH * n_qp);
    p.num_ctas = sms;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit_ns = g_wait_ns.load();
    cudaError_t e = fa::launch_fwd(p, d, causal != 0, o_dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d)
{
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
    const size_t rows = static_cast<size_t>(B) * H * ((static_cast<size_t>(N) + fa::kBlockM - 1) / fa::kBlockM) *
                        fa::kBlockM;
    return round_up(rows * d * sizeof(float), kAlign) + 2 * round_up(rows * sizeof(float), kAlign);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* grad_o,
                 void* grad_q, void* grad_k, void* grad_v, void* workspace, size_t ws_bytes, int B, int H, int N,
                 int Nk, int d, int dv, int causal, float scale, fa_dtype o_dtype, fa_dtype grad_dtype, void* stream)
{
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse == nullptr || grad_o == nullptr ||
        grad_q == nullptr || grad_k == nullptr || grad_v == nullptr || workspace == nullptr)
        return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || N <= 0 || Nk <= 0 || d <= 0 || dv <= 0) return FA_ERR_INVALID_ARG;
    if ((causal != 0 && causal != 1) || !dtype_ok(o_dtype) || !dtype_ok(grad_dtype) || !scale_ok(scale))
        return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(grad_o, 16) || !aligned(grad_q, 16) || !aligned(grad_k, 16) || !aligned(grad_v, 16) ||
        !aligned(workspace, kAlign))
        return FA_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    const long long Tr = (static_cast<long long>(N) + fa::kBlockM - 1) / fa::kBlockM;
    const long long Tc = (static_cast<long long>(Nk) + fa::kBlockN - 1) / fa::kBlockN;
    if (BH * Tc > 0x3fffffffLL) return FA_ERR_INVALID_ARG;  // 32-bit item indices with headroom for the cursor's step
    if (!head_ok(d) || dv != d) return FA_ERR_UNSUPPORTED;
    if (ws_bytes < fa_bwd_workspace_size(B, H, N, d)) return FA_ERR_WORKSPACE;

    int* status = nullptr;
    if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
    const size_t rows = static_cast<size_t>(BH) * Tr * fa::kBlockM;
    char* ws = static_cast<char*>(workspace);
    float* dq_acc = reinterpret_cast<float*>(ws);
    float* lse2 = reinterpret_cast<float*>(ws + round_up(rows * d * sizeof(float), kAlign));
    float* dsc = reinterpret_cast<float*>(reinterpret_cast<char*>(lse2) + round_up(rows * sizeof(float), kAlign));
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    fa::BwdPrepParams pp;
    pp.o = o;
    pp.d_o = grad_o;
    pp.lse = lse;
    pp.lse2 = lse2;
    pp.dsc = dsc;
    pp.dq_acc = dq_acc;
    pp.BH = static_cast<int>(BH);
    pp.N = N;
    pp.Tr = static_cast<int>(Tr);
    pp.d = d;
    pp.scale = scale;
    if (fa::launch_bwd_prep(pp, o_dtype, st) != cudaSuccess) return FA_ERR_CUDA;

    fa::BwdParams p;
    if (!make_map(&p.tm_q, q, static_cast<int>(BH), N, d) || !make_map(&p.tm_k, k, static_cast<int>(BH), Nk, d) ||
        !make_map(&p.tm_v, v, static_cast<int>(BH), Nk, dv) ||
        !make_map(&p.tm_do, grad_o, static_cast<int>(BH), N, dv) ||
        !make_out_map(&p.tm_dk, grad_k, static_cast<int>(BH), Nk, d, grad_dtype, fa::kBlockM) ||
        !make_out_map(&p.tm_dv, grad_v, static_cast<int>(BH), Nk, dv, grad_dtype, fa::kBlockM))
        return FA_ERR_CUDA;
    p.lse2 = lse2;
    p.dsc = dsc;
    p.dq_acc = dq_acc;
    p.dk = grad_k;
    p.dv = grad_v;
    p.status = status;
    p.BH = static_cast<int>(BH);
    p.N = N;
    p.Nk = Nk;
    p.Tr = static_cast<int>(Tr);
    p.Tc = static_cast<int>(Tc);
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return FA_ERR_CUDA;
    p.num_ctas = sms;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.scale = scale;
    p.wait_limit_ns = g_wait_ns.load();
    if (fa::launch_bwd(p, d, causal != 0, grad_dtype, st) != cudaSuccess) return FA_ERR_CUDA;

    fa::BwdDqParams dp;
    dp.dq_acc = dq_acc;
    dp.dq = grad_q;
    dp.BH = static_cast<int>(BH);
    dp.N = N;
    dp.Tr = static_cast<int>(Tr);
    dp.d = d;
    return fa::launch_bwd_dq(dp, grad_dtype, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_decode_default_splits(int B, int H, int Nk_max, int num_sms)
{
    if (B <= 0 || H <= 0 || Nk_max <= 0 || num_sms <= 0) return 0;
    // Enough (b, h, split) items for several full waves of 4-warp CTAs, but no
    // split shorter than a few key blocks.
    const long long heads = static_cast<long long>(B) * H;
    const long long target = 64LL * num_sms;
    long long n = (target + heads - 1) / heads;
    const long long max_n = (static_cast<long long>(Nk_max) + 4 * fa::kDecodeKeyBlock - 1) / (4 * fa::kDecodeKeyBlock);
    if (n > max_n) n = max_n;
    if (n < 1) n = 1;
    return static_cast<int>(n);
}

size_t fa_decode_workspace_size(int B, int H, int dv, int n_splits)
{
    if (B <= 0 || H <= 0 || dv <= 0 || n_splits <= 0) return 0;
    const size_t slots = static_cast<size_t>(B) * H * n_splits;
    return round_up(slots * dv * sizeof(float), kAlign) + round_up(slots * sizeof(float), kAlign);
}

}  // extern "C"

namespace {

// Merge n_splits partial states per row (every slot written by the split kernel).
cudaError_t merge_rows(const float* o_part, const float* lse_part, int rows, int n_splits, int dv, void* o,
                       float* lse, int* status, fa_dtype o_dtype, cudaStream_t st)
{
    fa::MergeParams m{};
    m.o_parts = o_part;
    m.lse_parts = lse_part;
    m.o_part_stride = dv;
    m.o_row_stride = static_cast<long long>(n_splits) * dv;
    m.lse_part_stride = 1;
    m.lse_row_stride = n_splits;
    m.n_parts = n_splits;
    m.rows = rows;
    m.dv = dv;
    m.seqlens = nullptr;
    m.o = o;
    m.lse = lse;
    m.status = status;
    return fa::launch_merge(m, o_dtype, st);
}

// Groups of 1 or 2 query heads per key/value head run on the CUDA-core split kernel (the packed
// rows' dot products are cheap there and it keeps more loads in flight), and so do groups of 4
// at d != 128; every other group size up to 128 runs on the tensor core.  Measured on GB300 with
// 32 query heads, d = 128 and 1-32K cached tokens: 4 heads per group 5.1 TB/s on CUDA cores
// against 6.4-6.7 on the transposed tensor-core kernel; 2 heads 7.0 TB/s on CUDA cores.
bool gqa_on_cuda_cores(int R, int d) { return R == 1 || R == 2 || (R == 4 && d != 128); }

// d = 128 with 3-32 query heads per group: the transposed kernel (keys on the TMEM lanes, the
// group's heads on 16 or 32 columns); otherwise the heads are rows of a 128-row tile
bool gqa_transposed(int R, int d) { return d == 128 && R >= 3 && R <= 32; }

// Tensor-core groups: one CTA per (b, key/value head, split); the transposed kernel runs two CTAs
// per SM for 3 to 8 heads, the others one.  A CTA's time goes to the per-tile softmax chain more
// than to the bytes, and the lengths vary (many of the later splits are short or empty), so the
// count aims at about 1.7 CTAs per CTA slot; splits longer than T key tiles are cut down further,
// so that many groups still spread evenly over the slots: T = 32 for more than 4 heads, 64 for up
// to 4 (their tiles are cheaper, so a CTA's fixed cost weighs more).  Measured on GB300, d = 128,
// 1-32K cached tokens, 24-64 query heads over 1-8 key/value heads, 4-64 sequences: within 3 %
// of the best count swept for 3-, 4-, 8-, 16- and 32-head groups; 8-head groups of 64 sequences x
// 4 key/value heads with 2 splits of 32K keys 6.2 TB/s, with 8 splits 6.8.
// At least two splits while the groups alone leave SMs idle; each split at least one 128-key tile.
int gqa_tc_default_splits(int B, int R, int Hkv, int Nk_max, int d, int sms)
{
    const long long groups = static_cast<long long>(B) * Hkv;
    const long long slots = static_cast<long long>(sms) * (gqa_transposed(R, d) && R <= 8 ? 2 : 1);
    long long n = 17LL * slots / (10LL * groups);
    if (n < 2 && groups < 2LL * sms) n = 2;
    const long long max_n = (static_cast<long long>(Nk_max) + fa::kBlockN - 1) / fa::kBlockN;
    const long long tiles_per_split = R <= 4 ? 64 : 32;
    const long long min_n = (max_n + tiles_per_split - 1) / tiles_per_split;
    if (n < min_n) n = min_n;
    if (n > max_n) n = max_n;
    if (n < 1) n = 1;
    return static_cast<int>(n);
}

// Split-KV decode for Hq query heads over Hkv key/value heads (Hkv = Hq: multi-head).
fa_status decode_impl(const void* q, const void* k_cache, const void* v_cache, const int* seqlens_k, void* o,
                      float* lse, void* workspace, size_t ws_bytes, int B, int Hq, int Hkv, int Nk_max, int d, int dv,
                      float scale, int n_splits, fa_dtype o_dtype, void* stream, bool fused = false)
{
    if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seqlens_k == nullptr || o == nullptr ||
        workspace == nullptr)
        return FA_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nk_max <= 0 || d <= 0 || dv <= 0 || n_splits < 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!dtype_ok(o_dtype) || !scale_ok(scale)) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
        !aligned(lse, 4) || !aligned(seqlens_k, 4) || !aligned(workspace, kAlign))
        return FA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * Hq > 0x7fffffffLL || B > 65535 || Hkv > 65535) return FA_ERR_INVALID_ARG;
    const int R = Hq / Hkv;
    const bool tc = !gqa_on_cuda_cores(R, d);
    if (!head_ok(d) || dv != d || R > fa::kBlockM) return FA_ERR_UNSUPPORTED;

    int n = n_splits;
    if (n == 0) {
        int sms = 0;
        if (sm_count(&sms) != cudaSuccess) return FA_ERR_CUDA;
        n = fa_decode_gqa_default_splits(B, Hq, Hkv, Nk_max, d, sms);
    }
    if (n > Nk_max) n = Nk_max;
    const size_t part_bytes = fa_decode_workspace_size(B, Hq, dv, n);
    const size_t counter_bytes = fused ? round_up(static_cast<size_t>(B) * Hkv * sizeof(unsigned int), kAlign) : 0;
    if (ws_bytes < part_bytes + counter_bytes) return FA_ERR_WORKSPACE;
    if (fused && tc) return FA_ERR_UNSUPPORTED;
    if (tc) {
        // packed groups on the tensor core: splits are whole 128-key tiles
        long long chunk = (static_cast<long long>(Nk_max) + n - 1) / n;
        chunk = (chunk + fa::kBlockN - 1) / fa::kBlockN * fa::kBlockN;
        const int n_eff = static_cast<int>((Nk_max + chunk - 1) / chunk);
        int* status = nullptr;
        if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
        fa::SplitParams sp;
        const long long groups = static_cast<long long>(B) * Hkv;
        const bool transposed = gqa_transposed(R, d);
        const int q_box = transposed ? (R <= 16 ? 16 : 32) : fa::kBlockM;
        if (!transposed && groups > 65535) return FA_ERR_UNSUPPORTED;  // grid z
        if (!make_map(&sp.tm_q, q, static_cast<int>(groups), R, d, q_box) ||
            !make_map(&sp.tm_k, k_cache, static_cast<int>(groups), Nk_max, d) ||
            !make_map(&sp.tm_v, v_cache, static_cast<int>(groups), Nk_max, dv))
            return FA_ERR_CUDA;
        const size_t slots = static_cast<size_t>(B) * Hq * n_eff;
        sp.o_part = static_cast<float*>(workspace);
        sp.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(slots * dv * sizeof(float), kAlign));
        sp.seqlens = seqlens_k;
        sp.status = status;
        sp.n_groups = static_cast<int>(groups);
        sp.rows_per_group = R;
        sp.n_qtiles = 1;
        sp.groups_per_batch = Hkv;
        sp.Nk = Nk_max;
        sp.n_splits = n_eff;
        sp.chunk = static_cast<int>(chunk);
        sp.causal_off = 0;
        sp.scale_log2 = scale * 1.4426950408889634f;
        sp.wait_limit_ns = g_wait_ns.load();
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        if ((transposed ? fa::launch_gqa_tc(sp, st) : fa::launch_splitkv(sp, d, false, true, st)) != cudaSuccess)
            return FA_ERR_CUDA;
        return merge_rows(sp.o_part, sp.lse_part, B * Hq, n_eff, dv, o, lse, status, o_dtype, st) == cudaSuccess
                   ? FA_OK
                   : FA_ERR_CUDA;
    }
    // Fixed chunk per split, a whole number of key blocks; trailing splits may be empty.
    long long chunk = (static_cast<long long>(Nk_max) + n - 1) / n;
    chunk = (chunk + fa::kDecodeKeyBlock - 1) / fa::kDecodeKeyBlock * fa::kDecodeKeyBlock;
    const int n_eff = static_cast<int>((Nk_max + chunk - 1) / chunk);

    int* status = nullptr;
    if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
    fa::DecodeParams p;
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.seqlens = seqlens_k;
    const size_t slots = static_cast<size_t>(B) * Hq * n_eff;
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(slots * dv * sizeof(float), kAlign));
    p.o = o;
    p.lse = lse;
    p.status = status;
    p.B = B;
    p.H = Hq;
    p.Hkv = Hkv;
    p.Nk_max = Nk_max;
    p.n_splits = n_eff;
    p.chunk = static_cast<int>(chunk);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.counters = fused ? reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + part_bytes) : nullptr;
    p.o_dtype = o_dtype;
    cudaError_t e = fa::launch_decode(p, d, o_dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_decode_gqa_default_splits(int B, int Hq, int Hkv, int Nk_max, int d, int num_sms)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nk_max <= 0 || d <= 0 || num_sms <= 0 || Hq % Hkv != 0) return 0;
    // On CUDA cores a CTA's arithmetic grows with the R heads it carries, so the count follows the
    // B * Hq query heads (R = 4: 4.3 -> 4.8 TB/s against counting B * Hkv items).
    return gqa_on_cuda_cores(Hq / Hkv, d) ? fa_decode_default_splits(B, Hq, Nk_max, num_sms)
                                          : gqa_tc_default_splits(B, Hq / Hkv, Hkv, Nk_max, d, num_sms);
}

fa_status fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, const int* seqlens_k, void* o,
                            float* lse, void* workspace, size_t ws_bytes, int B, int H, int Nk_max, int d, int dv,
                            float scale, int n_splits, fa_dtype o_dtype, void* stream)
{
    return decode_impl(q, k_cache, v_cache, seqlens_k, o, lse, workspace, ws_bytes, B, H, H, Nk_max, d, dv, scale,
                       n_splits, o_dtype, stream);
}

int fa_fwd_splitkv_default_splits(int B, int H, int N, int Nk, int num_sms)
{
    if (B <= 0 || H <= 0 || N <= 0 || Nk <= 0 || num_sms <= 0) return 0;
    // A split item is (head, pair of 128-row query tiles, split) on the persistent forward kernel,
    // one CTA per SM, and an item costs a few key tiles beyond its own (Q load, pipeline fill,
    // partial write, its share of the merge), so a second round of shorter items loses to one
    // round of longer ones: the count is the largest for which every item runs at once, each
    // split at least one 128-key tile.  Measured on GB300, B=1 H=8 N=512 Nk=32K d=128 causal
    // (16 query pairs): 9 splits (144 items) 790 TFLOP/s, 8 753, 12 (192 items, a short second
    // round) 557, 19 (two full rounds) 770.
    const long long pairs = static_cast<long long>(B) * H * ((N + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM));
    const long long max_n = (static_cast<long long>(Nk) + fa::kBlockN - 1) / fa::kBlockN;
    long long n = num_sms / pairs;
    if (n > max_n) n = max_n;
    if (n < 1) n = 1;
    return static_cast<int>(n);
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int dv, int n_splits)
{
    if (B <= 0 || H <= 0 || N <= 0 || dv <= 0 || n_splits <= 0) return 0;
    const size_t slots = static_cast<size_t>(B) * H * N * n_splits;
    return round_up(slots * dv * sizeof(float), kAlign) + round_up(slots * sizeof(float), kAlign);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                         size_t ws_bytes, int B, int H, int N, int Nk, int d, int dv, int causal, float scale,
                         int n_splits, fa_dtype o_dtype, void* stream)
{
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || workspace == nullptr) return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || N <= 0 || Nk <= 0 || d <= 0 || dv <= 0 || n_splits < 0) return FA_ERR_INVALID_ARG;
    if ((causal != 0 && causal != 1) || !dtype_ok(o_dtype) || !scale_ok(scale)) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(workspace, kAlign))
        return FA_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    const long long n_qp = (static_cast<long long>(N) + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
    if (BH * N > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    if (!head_ok(d) || dv != d) return FA_ERR_UNSUPPORTED;
    int sms = 0;
    int n = n_splits;
    if (n == 0) {
        if (sm_count(&sms) != cudaSuccess) return FA_ERR_CUDA;
        n = fa_fwd_splitkv_default_splits(B, H, N, Nk, sms);
    }
    if (n > Nk) n = Nk;
    if (ws_bytes < fa_fwd_splitkv_workspace_size(B, H, N, dv, n)) return FA_ERR_WORKSPACE;
    if (sms == 0 && sm_count(&sms) != cudaSuccess) return FA_ERR_CUDA;
    // whole 128-key tiles per split; trailing splits past the keys are dropped
    const long long key_tiles = (static_cast<long long>(Nk) + fa::kBlockN - 1) / fa::kBlockN;
    const long long split_tiles = (key_tiles + n - 1) / n;
    const long long n_eff = (key_tiles + split_tiles - 1) / split_tiles;
    // the kernels index items with 32-bit ints and step past the last one by up to the grid size
    if (BH * n_qp * n_eff > 0x3fffffffLL) return FA_ERR_INVALID_ARG;

    int* status = nullptr;
    if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
    fa::FwdParams p{};
    if (!make_map(&p.tm_q, q, static_cast<int>(BH), N, d) || !make_map(&p.tm_k, k, static_cast<int>(BH), Nk, d) ||
        !make_map(&p.tm_v, v, static_cast<int>(BH), Nk, dv))
        return FA_ERR_CUDA;
    const size_t slots = static_cast<size_t>(BH) * N * static_cast<size_t>(n_eff);
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(slots * dv * sizeof(float), kAlign));
    p.o = nullptr;
    p.lse = nullptr;
    p.status = status;
    p.BH = static_cast<int>(BH);
    p.N = N;
    p.Nk = Nk;
    p.n_splits = static_cast<int>(n_eff);
    p.split_tiles = static_cast<int>(split_tiles);
    p.n_qp = static_cast<int>(n_qp * n_eff);  // (query pair, split) items per head
    p.n_items = static_cast<int>(BH * n_qp * n_eff);
    p.num_ctas = sms;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit_ns = g_wait_ns.load();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (fa::launch_fwd_split(p, d, causal != 0, st) != cudaSuccess) return FA_ERR_CUDA;
    return merge_rows(p.o_part, p.lse_part, static_cast<int>(BH * N), static_cast<int>(n_eff), dv, o, lse, status,
                      o_dtype, st) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
}

size_t fa_decode_fused_workspace_size(int B, int H, int dv, int n_splits)
{
    const size_t parts = fa_decode_workspace_size(B, H, dv, n_splits);
    return parts == 0 ? 0 : parts + round_up(static_cast<size_t>(B) * H * sizeof(unsigned int), kAlign);
}

fa_status fa_decode_splitkv_fused(const void* q, const void* k_cache, const void* v_cache, const int* seqlens_k,
                                  void* o, float* lse, void* workspace, size_t ws_bytes, int B, int H, int Nk_max,
                                  int d, int dv, float scale, int n_splits, fa_dtype o_dtype, void* stream)
{
    return decode_impl(q, k_cache, v_cache, seqlens_k, o, lse, workspace, ws_bytes, B, H, H, Nk_max, d, dv, scale,
                       n_splits, o_dtype, stream, true);
}

fa_status fa_decode_splitkv_gqa(const void* q, const void* k_cache, const void* v_cache, const int* seqlens_k,
                                void* o, float* lse, void* workspace, size_t ws_bytes, int B, int Hq, int Hkv,
                                int Nk_max, int d, int dv, float scale, int n_splits, fa_dtype o_dtype, void* stream)
{
    return decode_impl(q, k_cache, v_cache, seqlens_k, o, lse, workspace, ws_bytes, B, Hq, Hkv, Nk_max, d, dv, scale,
                       n_splits, o_dtype, stream);
}

fa_status fa_merge_states(const float* o_parts, const float* lse_parts, int n_parts, int rows, int dv, void* o,
                          float* lse, fa_dtype o_dtype, void* stream)
{
    if (o_parts == nullptr || lse_parts == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
    if (n_parts <= 0 || rows <= 0 || dv <= 0 || dv > 512 || !dtype_ok(o_dtype)) return FA_ERR_INVALID_ARG;
    if (!aligned(o_parts, 4) || !aligned(lse_parts, 4) || !aligned(o, 4) || !aligned(lse, 4))
        return FA_ERR_INVALID_ARG;
    int* status = nullptr;
    if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
    fa::MergeParams m{};
    m.o_parts = o_parts;
    m.lse_parts = lse_parts;
    m.o_part_stride = static_cast<long long>(rows) * dv;
    m.o_row_stride = dv;
    m.lse_part_stride = rows;
    m.lse_row_stride = 1;
    m.n_parts = n_parts;
    m.rows = rows;
    m.dv = dv;
    m.seqlens = nullptr;
    m.o = o;
    m.lse = lse;
    m.status = status;
    cudaError_t e = fa::launch_merge(m, o_dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_get_device_error(void* stream)
{
    int* status = nullptr;
    if (status_word(&status) != cudaSuccess) return FA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemcpyAsync(&h, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
    return static_cast<fa_status>(h);
}

}  // extern "C"
