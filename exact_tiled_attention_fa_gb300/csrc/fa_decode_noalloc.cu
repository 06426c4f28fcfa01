// fa_decode_noalloc.cu -- fa_decode_splitkv_noalloc: split-KV decode whose split
// partials live in a scratch array owned by the library, so the caller never has
// to provide (and therefore never has to allocate) device workspace.
//
// Some callers cannot allocate device memory: code whose device memory belongs to
// another allocator (a framework's caching allocator, a serving engine's fixed pool)
// and may not call cudaMalloc behind its back, code under a hard per-process memory
// budget, and code that must not risk the device-wide synchronisation cudaMalloc and
// cudaFree can cause.  This entry point gives them the same result as
// fa_decode_splitkv while allocating nothing.
#include <mutex>

#include "fa_internal.h"

namespace {

// The scratch array.  Every GPU that loads the library holds these bytes until the
// process exits.  The host cannot use the symbol itself as a device address; the
// address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[FA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use).
fa_status scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                               const int* seqlens_k, void* o, float* lse, int B, int H,
                                               int Nk_max, int d, int dv, float scale, int n_splits,
                                               fa_dtype o_dtype, void* stream)
{
    // Reject problems whose partials do not fit before touching the device.
    if (B > 0 && H > 0 && dv > 0 && n_splits > 0) {
        const int n = n_splits < Nk_max ? n_splits : (Nk_max > 0 ? Nk_max : 1);
        if (fa_decode_workspace_size(B, H, dv, n) > FA_DECODE_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    const fa_status st = scratch_address(&scratch);
    if (st != FA_OK) return st;
    // Same checks and kernels as fa_decode_splitkv; it reports FA_ERR_WORKSPACE when the
    // automatic split count needs more partial storage than the scratch array holds.
    return fa_decode_splitkv(q, k_cache, v_cache, seqlens_k, o, lse, scratch, FA_DECODE_NOALLOC_SCRATCH_BYTES, B,
                             H, Nk_max, d, dv, scale, n_splits, o_dtype, stream);
}
