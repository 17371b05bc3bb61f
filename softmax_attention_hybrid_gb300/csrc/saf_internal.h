// Internal declarations shared by the host entry points and the kernels of
// the SAF hybrid attention library. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "saf.h"

namespace saf {

// Head dimension of the main tensor-core kernels (bf16). dh_tc.cu serves bf16
// at 96 and 128 (multi-head layout, per-call normalisers); the fp32 CUDA-core
// path takes 64, 96 and 128.
constexpr int kHeadDim = 64;
inline bool head_dim_supported(int d, saf_dtype_t dt) {
    (void)dt;
    return d == kHeadDim || d == 96 || d == 128;
}

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

// Programmatic dependent launch. Every kernel of the tensor-core path starts
// with grid_dep_wait(): it returns once the kernels before it on the stream
// have completed and their memory is visible (at once when the kernel was
// launched without the attribute), so a kernel that was scheduled early never
// touches data that is still being written. Every CTA runs it, early exits
// included, so that a kernel's completion implies its predecessors'.
// grid_dep_launch() then lets the next kernel on the stream be scheduled while
// this one runs; that kernel's own grid_dep_wait() holds it back until this
// one has completed.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with cudaLaunchKernelEx: pdl allows programmatic dependent launch
// after the previous kernel on the stream (the kernel must call
// grid_dep_wait() first); cluster > 1 groups consecutive CTAs of the x
// dimension into thread-block clusters of that size.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      int cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    unsigned n = 0;
    if (pdl) {
        at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = (unsigned)cluster;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = at;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Error word layout at the start of every workspace (256 bytes reserved,
// cleared by the first kernel of every call).
//   status[0]: bitwise OR of kStatus* flags raised by kernels of the last call
//   status[8]: work-item counter of the tensor-core backward
//   status[9]: work-item counter of the tensor-core forward
enum : uint32_t {
    kStatusRange = 1u << 0,     // info: a frozen head left the factorised form's range and
                                // is computed in the exact exp form (not an error)
// per-head flags (hflag[h]): bit 0 the normaliser prep needed its exact
// fallback, bit 1 the tensor-core kernels must use the exact form
    kStatusTimeout = 1u << 1,   // a bounded mbarrier wait expired
};
constexpr size_t kStatusBytes = 256;
constexpr int kCounterBwd = 8;
constexpr int kCounterFwd = 9;

// Byte offsets of the workspace regions for one call.
// Tp = T rounded up to a multiple of 128 (query and key blocks).
struct WorkspaceLayout {
    size_t status = 0;   // uint32[64]
    size_t lz = 0;       // fp32 [H, T]   log Z of frozen heads (batch independent)
    size_t hflag = 0;    // uint32 [H]    per-head flags raised by the normaliser prep
    size_t amax = 0;     // fp32 [2, H]   max a, max r of frozen heads
    size_t a2p = 0;      // fp32 [H, Tp]  a * log2(e), -inf padded (bf16 path)
    size_t r2p = 0;      // fp32 [H, Tp + 256]  r * log2(e) shifted by 127, -inf padded (bf16 path)
    size_t eap = 0;      // fp32 [H, Tp]  exp(a - max a), 0 padded (bf16 path)
    size_t erp = 0;      // fp32 [H, Tp + 256]  exp(r - max r) shifted by 127, 0 padded (bf16 path)
    size_t invz = 0;     // fp32 [H, Tp]  1 / Z' of the factorised form, 0 padded (bf16 path)
    size_t delta = 0;    // fp32 [B, H, T] D_i = sum_c dO_ic O_ic (fp32 backward)
    size_t rowvec = 0;   // fp32 [B, H, Tp / 128, 256] lse * log2(e) and D per query block (bf16 backward)
    size_t dq_acc = 0;   // fp32 [B, H, T, 64] dQ accumulator (bf16 backward)
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
    float* amax;         // workspace: max a [H], max r [H]
    float* delta;        // workspace: D [B, H, T]
    float* dq_acc;       // workspace: fp32 dQ accumulator [B, H, T, 64]
    float* a2p;          // workspace: padded a * log2(e) [H, Tp]
    float* r2p;          // workspace: padded r * log2(e) [H, Tp + 256]
    float* eap;          // workspace: exp(a - max a) [H, Tp]
    float* erp;          // workspace: exp(r - max r), shifted by 127 [H, Tp + 256]
    float* invz;         // workspace: 1 / Z' [H, Tp]
    float* rowvec;       // workspace: per-block row vectors [B, H, Tp / 128, 256]
    uint32_t* status;    // workspace: error words
    int B, H, T, ld_prior;
    int Hkv;             // key/value heads: query head h reads key/value head h / (H / Hkv)
    int d;               // head dimension
    HeadMask mask;
    // diagnostic forward only (saf_attn_fwd_diag): a shorter limit for every bounded
    // wait (0: the default), and a producer that withholds every work item
    unsigned long long diag_wait_ns;
    int diag_withhold;
};

// Launch bookkeeping (saf_api.cu): call before_launch(kernel id, stream)
// right before a launch and after_launch(...) right after it; they count
// the launch and record the trace events of saf_set_trace_events.
void before_launch(int kernel, cudaStream_t s);
// the start event only (launches counted separately with note_launch)
void trace_begin(int kernel, cudaStream_t s);
// a further launch inside a group bracketed by before_launch / after_launch
void note_launch();
void after_launch(int kernel, cudaStream_t s);

// prep.cu
// First kernel of every call: clears the status words and per-head flags; for
// the frozen heads, max a and max r, and with pad (tensor-core path) the
// padded a, r slices in both forms of Eq. 3. 1 launch, counted.
cudaError_t launch_call_init(const LayerArgs& p, bool pad, bool pdl, cudaStream_t s);
// log Z of the frozen heads (and with pre, tensor-core path: from the padded
// exp slices of launch_call_init, also 1 / Z' and the exact-form flag).
// 1 launch, counted.
cudaError_t launch_lognorm(const LayerArgs& p, bool pre, bool pdl, cudaStream_t s);
// Tensor-core backward prep: per-tile lse and D rows, the zeroed dQ
// accumulator of ordinary heads, and 1 / Z' of frozen heads from lse.
// frozen_part: also 1 / Z' and the exact-form flags of the frozen heads, from the
// log Z rows of lse (false when a prepared frozen-pattern state already holds them).
cudaError_t launch_bwd_prep(const LayerArgs& p, cudaStream_t s, bool frozen_part = true);
cudaError_t launch_bwd_delta(const LayerArgs& p, bool bf16, cudaStream_t s);

// fwd_tc.cu: tensor-core forward (bf16)
cudaError_t launch_tc_fwd(const LayerArgs& p, cudaStream_t s);

// bwd_tc.cu: tensor-core backward (bf16), including the dQ finishing kernel
cudaError_t launch_tc_bwd(const LayerArgs& p, cudaStream_t s);

// dh_tc.cu: tensor-core forward and backward (bf16) at head dimensions 96 and 128
// (one key/value head per query head). The forward needs the layer's call_init
// and lognorm launches before it; the backward call_init, and launches its own prep.
cudaError_t launch_dh_fwd(const LayerArgs& p, cudaStream_t s);
cudaError_t launch_dh_bwd(const LayerArgs& p, cudaStream_t s);

// simt.cu: fp32-arithmetic path (any dtype), used for SAF_FP32
cudaError_t launch_simt_fwd(const LayerArgs& p, bool bf16, cudaStream_t s);
cudaError_t launch_simt_bwd(const LayerArgs& p, bool bf16, cudaStream_t s);

}  // namespace saf
