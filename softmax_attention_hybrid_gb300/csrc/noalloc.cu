// Forward pass for callers that cannot allocate device memory.
//
// saf_attn_fwd needs a caller-provided device workspace. Some callers cannot
// provide one: code running where cudaMalloc is off limits (inside a
// stream-ordered region that must not allocate, a host framework that owns
// every allocation and hands out only input and output buffers, or a plugin
// called from a context where allocation could deadlock or fragment a
// caching allocator). saf_attn_fwd_noalloc serves them: it runs the same
// forward kernels as saf_attn_fwd, with the workspace taken from a fixed
// array in device memory that this library declares statically. No call
// allocates or frees anything.
//
// The array is kNoallocScratchBytes (8 MiB) per device, held by every GPU
// that loads the library until the process exits. Problems whose forward
// workspace would exceed it are rejected with SAF_ESCRATCH.
#include <mutex>

#include "saf_internal.h"

namespace saf {
namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

// File-scope device scratch. In host code this name is only a stand-in for
// the symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. The first call
// on each device looks it up (with that device current) and caches it.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SAF_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SAF_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return SAF_ECUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SAF_OK;
}

}  // namespace
}  // namespace saf

extern "C" int saf_attn_fwd_noalloc(const void* q, const void* k, const void* v, const float* a, const float* r,
                                    int ld_prior, const uint8_t* frozen, int B, int H, int T, int d,
                                    saf_dtype_t dt, void* o, float* lse, void* stream) {
    using namespace saf;
    const size_t need = saf_attn_workspace_bytes(B, H, T, d, dt, 0);
    if (need == 0) return (dt == SAF_BF16 || dt == SAF_FP32) && !head_dim_supported(d, dt) ? SAF_EUNSUPPORTED : SAF_EINVAL;
    if (need > kNoallocScratchBytes) return SAF_ESCRATCH;
    void* ws = nullptr;
    const int st = scratch_address(&ws);
    if (st != SAF_OK) return st;
    // The forward pass clears the status words and per-head flags it uses (its
    // first kernel, on `stream`) before anything reads them, so stale contents
    // left by an earlier call do not leak into this one.
    return saf_attn_fwd(q, k, v, a, r, ld_prior, frozen, B, H, T, d, dt, o, lse, ws, kNoallocScratchBytes, stream);
}
