// Internal declarations shared by the host entry points and the kernels of
// the SAF hybrid attention library. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "saf.h"

namespace saf {

// Head dimension of every kernel in this library.
constexpr int kHeadDim = 64;

// Per-head frozen flags as a bitmask, passed by value to every kernel so that
// no host-to-device copy is needed per call (H <= SAF_MAX_HEADS).
struct HeadMask {
    uint64_t w[SAF_MAX_HEADS / 64];
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__host__ __device__ inline bool head_frozen(const HeadMask& m, int h) {
    return (m.w[h >> 6] >> (h & 63)) & 1ull;
}

// Error word layout at the start of every workspace (256 bytes reserved).
//   status[0]: bitwise OR of kStatus* flags raised by kernels of the last call
//   status[1]: first work item whose bounded wait expired (diagnostic)
enum : uint32_t {
    kStatusRange = 1u << 0,     // info: a frozen head left the factorised form's range and
                                // is computed in the exact exp form (not an error)
    kStatusTimeout = 1u << 1,   // a bounded mbarrier wait expired
};
constexpr size_t kStatusBytes = 256;

// Byte offsets of the workspace regions for one call.
struct WorkspaceLayout {
    size_t status = 0;   // uint32[64]
    size_t lz = 0;       // fp32 [H, T]   log Z of frozen heads (batch independent)
    size_t hflag = 0;    // uint32 [H]    per-head flags raised by the normaliser prep
    size_t delta = 0;    // fp32 [B, H, T] D_i = sum_c dO_ic O_ic (backward only)
    size_t dq_acc = 0;   // fp32 [B, H, T, 64] dQ accumulator of the tensor-core backward (bf16 only)
    size_t total = 0;
};
WorkspaceLayout workspace_layout(int B, int H, int T, int backward, int bf16);

// Everything a kernel needs about one call. Pointers are device pointers.
struct LayerArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* o;       // backward: forward output
    const void* dO;      // backward: output gradient
    const float* lse;    // backward: forward lse
    const float* a;
    const float* r;
    void* out;           // forward: o
    float* lse_out;      // forward: lse
    void* dq;
    void* dk;
    void* dv;
    float* lz;           // workspace: log Z [H, T]
    uint32_t* hflag;     // workspace: per-head flags [H]
    float* delta;        // workspace: D [B, H, T]
    float* dq_acc;       // workspace: fp32 dQ accumulator [B, H, T, 64]
    uint32_t* status;    // workspace: error words
    int B, H, T, ld_prior;
    HeadMask mask;
};

// Launch bookkeeping (saf_api.cu): call before_launch(kernel id, stream)
// right before a launch and after_launch(...) right after it; they count
// the launch and record the trace events of saf_set_trace_events.
void before_launch(int kernel, cudaStream_t s);
void after_launch(int kernel, cudaStream_t s);

// prep.cu
cudaError_t launch_lognorm(const LayerArgs& p, cudaStream_t s);
cudaError_t launch_bwd_delta(const LayerArgs& p, bool bf16, cudaStream_t s);

// fwd_tc.cu: tensor-core forward (bf16)
cudaError_t launch_tc_fwd(const LayerArgs& p, cudaStream_t s);

// bwd_tc.cu: tensor-core backward (bf16), including the dQ finishing kernel
cudaError_t launch_tc_bwd(const LayerArgs& p, cudaStream_t s);

// simt.cu: fp32-arithmetic path (any dtype), used for SAF_FP32
cudaError_t launch_simt_fwd(const LayerArgs& p, bool bf16, cudaStream_t s);
cudaError_t launch_simt_bwd(const LayerArgs& p, bool bf16, cudaStream_t s);

}  // namespace saf
