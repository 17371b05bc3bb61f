// Host entry points of the C ABI declared in include/saf.h: argument
// validation, workspace carving, and the launch sequence of each pass.
#include <string.h>

#include "saf_internal.h"

namespace saf {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WorkspaceLayout workspace_layout(int B, int H, int T, int backward, int bf16) {
    WorkspaceLayout L;
    const size_t Tp = (size_t)(T + 127) / 128 * 128;
    size_t off = 0;
    L.status = off;
    off += kStatusBytes;
    L.lz = off;
    off = align_up(off + (size_t)H * T * sizeof(float), 256);
    L.hflag = off;
    off = align_up(off + (size_t)H * sizeof(uint32_t), 256);
    L.amax = off;
    off = align_up(off + (size_t)2 * H * sizeof(float), 256);
    if (bf16) {
        L.a2p = off;
        off = align_up(off + (size_t)H * Tp * sizeof(float), 256);
        L.r2p = off;
        off = align_up(off + (size_t)H * (Tp + 256) * sizeof(float), 256);
        L.eap = off;
        off = align_up(off + (size_t)H * Tp * sizeof(float), 256);
        L.erp = off;
        off = align_up(off + (size_t)H * (Tp + 256) * sizeof(float), 256);
        L.invz = off;
        off = align_up(off + (size_t)H * Tp * sizeof(float), 256);
    }
    if (backward) {
        if (bf16) {
            L.rowvec = off;
            off = align_up(off + (size_t)B * H * (Tp / 128) * 256 * sizeof(float), 256);
            L.dq_acc = off;
            off = align_up(off + (size_t)B * H * T * kHeadDim * sizeof(float), 256);
        } else {
            L.delta = off;
            off = align_up(off + (size_t)B * H * T * sizeof(float), 256);
        }
    }
    L.total = off;
    return L;
}

namespace {
constexpr int kNumKernelIds = SAF_KERNEL_PATTERN_GRAD + 1;
cudaEvent_t g_trace_start[kNumKernelIds] = {};
cudaEvent_t g_trace_stop[kNumKernelIds] = {};
unsigned long long g_launches = 0;
}  // namespace

void trace_begin(int kernel, cudaStream_t s) {
    if (g_trace_start[kernel]) cudaEventRecord(g_trace_start[kernel], s);
}

void before_launch(int kernel, cudaStream_t s) {
    ++g_launches;
    trace_begin(kernel, s);
}

void note_launch() { ++g_launches; }

void after_launch(int kernel, cudaStream_t s) {
    if (g_trace_stop[kernel]) cudaEventRecord(g_trace_stop[kernel], s);
}

namespace {

int g_device_ok = -1;  // cached: 1 = sm_103 device present, 0 = not

int check_device() {
    if (g_device_ok >= 0) return g_device_ok ? SAF_OK : SAF_EUNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SAF_ECUDA;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        return SAF_ECUDA;
    }
    g_device_ok = (prop.major == 10 && prop.minor == 3) ? 1 : 0;
    return g_device_ok ? SAF_OK : SAF_EUNSUPPORTED;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

struct Common {
    HeadMask mask;
    int nfrozen;
};

// Shape, pointer and workspace checks shared by both passes.
int validate(const void* q, const void* k, const void* v, const float* a, const float* r, int ld_prior,
             const uint8_t* frozen, int B, int H, int T, int d, saf_dtype_t dt, void* workspace,
             size_t ws_bytes, int backward, Common* c) {
    if (B < 0 || H <= 0 || T < 0) return SAF_EINVAL;
    if (H > SAF_MAX_HEADS) return SAF_EINVAL;
    if (dt != SAF_BF16 && dt != SAF_FP32) return SAF_EINVAL;
    if (!head_dim_supported(d, dt)) return SAF_EUNSUPPORTED;
    if ((long long)B * H * T * d > (1ll << 40)) return SAF_EINVAL;
    memset(c, 0, sizeof(*c));
    for (int h = 0; h < H; ++h) {
        if (frozen && frozen[h]) {
            c->mask.w[h >> 6] |= 1ull << (h & 63);
            c->nfrozen++;
        }
    }
    if (B == 0 || T == 0) return SAF_OK;  // empty call: nothing to check further
    if (!v) return SAF_EINVAL;
    if (c->nfrozen < H && (!q || !k)) return SAF_EINVAL;
    if (c->nfrozen > 0 && (!a || !r || ld_prior < T)) return SAF_EINVAL;
    if (!aligned16(v) || (q && !aligned16(q)) || (k && !aligned16(k))) return SAF_EALIGN;
    if ((a && ((uintptr_t)a & 3u)) || (r && ((uintptr_t)r & 3u))) return SAF_EALIGN;
    if (!workspace) return SAF_EWORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return SAF_EALIGN;
    if (ws_bytes < workspace_layout(B, H, T, backward, dt == SAF_BF16).total) return SAF_EWORKSPACE;
    return SAF_OK;
}

LayerArgs make_args(const void* q, const void* k, const void* v, const float* a, const float* r, int ld_prior,
                    int B, int H, int T, const Common& c, void* workspace, int backward, int bf16) {
    LayerArgs p;
    memset(&p, 0, sizeof(p));
    const WorkspaceLayout L = workspace_layout(B, H, T, backward, bf16);
    char* ws = (char*)workspace;
    p.q = q;
    p.k = k;
    p.v = v;
    p.a = a;
    p.r = r;
    p.B = B;
    p.H = H;
    p.T = T;
    p.ld_prior = ld_prior;
    p.Hkv = H;
    p.mask = c.mask;
    p.status = (uint32_t*)(ws + L.status);
    p.lz = (float*)(ws + L.lz);
    p.hflag = (uint32_t*)(ws + L.hflag);
    p.amax = (float*)(ws + L.amax);
    p.delta = (backward && !bf16) ? (float*)(ws + L.delta) : nullptr;
    p.dq_acc = (backward && bf16) ? (float*)(ws + L.dq_acc) : nullptr;
    p.rowvec = (backward && bf16) ? (float*)(ws + L.rowvec) : nullptr;
    p.a2p = bf16 ? (float*)(ws + L.a2p) : nullptr;
    p.r2p = bf16 ? (float*)(ws + L.r2p) : nullptr;
    p.eap = bf16 ? (float*)(ws + L.eap) : nullptr;
    p.erp = bf16 ? (float*)(ws + L.erp) : nullptr;
    p.invz = bf16 ? (float*)(ws + L.invz) : nullptr;
    return p;
}

int launch_status(cudaError_t e) {
    if (e == cudaSuccess) return SAF_OK;
    cudaGetLastError();
    return SAF_ELAUNCH;
}

// The kernels that run before the main kernel of a pass. The first one
// (call_init) clears the error words, work counters and per-head flags and,
// for the frozen heads, finds max a, max r and (tensor-core path) writes the
// padded a, r slices. The forward then computes log Z (and on the tensor-core
// path 1 / Z'); the tensor-core backward reads log Z back from lse in its prep
// kernel (launched by saf_attn_bwd), the fp32 backward recomputes it. The
// tensor-core path launches every kernel with programmatic dependent launch.
cudaError_t begin_call(const LayerArgs& p, const Common& c, bool backward, bool bf16, cudaStream_t s) {
    const int kid = backward ? SAF_KERNEL_PATTERN_PREP : SAF_KERNEL_LOGNORM;
    trace_begin(kid, s);
    cudaError_t e = launch_call_init(p, bf16, bf16, s);
    if (e == cudaSuccess && c.nfrozen > 0 && !(backward && bf16)) e = launch_lognorm(p, bf16, bf16, s);
    after_launch(kid, s);
    return e;
}

}  // namespace
}  // namespace saf

using namespace saf;

extern "C" {

int saf_version(void) { return 100; }

int saf_set_trace_events(int kernel, void* start, void* stop) {
    if (kernel < SAF_KERNEL_NONE || kernel >= kNumKernelIds) return SAF_EINVAL;
    if (kernel == SAF_KERNEL_NONE) {
        for (int i = 0; i < kNumKernelIds; ++i) g_trace_start[i] = g_trace_stop[i] = nullptr;
        return SAF_OK;
    }
    const bool on = start && stop;
    g_trace_start[kernel] = on ? (cudaEvent_t)start : nullptr;
    g_trace_stop[kernel] = on ? (cudaEvent_t)stop : nullptr;
    return SAF_OK;
}

unsigned long long saf_launch_count(void) { return g_launches; }

size_t saf_attn_workspace_bytes(int B, int H, int T, int d, saf_dtype_t dt, int backward) {
    if (B < 0 || H <= 0 || T < 0 || H > SAF_MAX_HEADS) return 0;
    if (dt != SAF_BF16 && dt != SAF_FP32) return 0;
    if (!head_dim_supported(d, dt)) return 0;
    return workspace_layout(B, H, T, backward ? 1 : 0, dt == SAF_BF16).total;
}

int saf_attn_fwd_gqa(const void* q, const void* k, const void* v, const float* a, const float* r, int ld_prior,
                     const uint8_t* frozen, int B, int H, int Hkv, int T, int d, saf_dtype_t dt, void* o, float* lse,
                     void* workspace, size_t ws_bytes, void* stream) {
    if (Hkv <= 0 || H <= 0 || H % Hkv != 0) return SAF_EINVAL;
    Common c;
    int st = validate(q, k, v, a, r, ld_prior, frozen, B, H, T, d, dt, workspace, ws_bytes, 0, &c);
    if (st != SAF_OK) return st;
    if (B == 0 || T == 0) return SAF_OK;
    if (!o || !lse) return SAF_EINVAL;
    if (!aligned16(o) || !aligned16(lse)) return SAF_EALIGN;
    if ((st = check_device()) != SAF_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    LayerArgs p = make_args(q, k, v, a, r, ld_prior, B, H, T, c, workspace, 0, dt == SAF_BF16);
    p.Hkv = Hkv;
    p.d = d;
    p.out = o;
    p.lse_out = lse;
    const bool bf16 = dt == SAF_BF16;
    cudaError_t e = begin_call(p, c, false, bf16, s);
    if (e == cudaSuccess)
        e = !bf16 ? launch_simt_fwd(p, false, s) : d == kHeadDim ? launch_tc_fwd(p, s) : launch_dh_fwd(p, s);
    return launch_status(e);
}

int saf_attn_fwd_diag(const void* q, const void* k, const void* v, const float* a, const float* r, int ld_prior,
                      const uint8_t* frozen, int B, int H, int T, int d, saf_dtype_t dt, void* o, float* lse,
                      void* workspace, size_t ws_bytes, void* stream, int withhold, unsigned wait_limit_us) {
    if (dt != SAF_BF16 || d != kHeadDim) return SAF_EUNSUPPORTED;   // the forward kernel with the test switches
    if (withhold != 0 && withhold != 1) return SAF_EINVAL;
    Common c;
    int st = validate(q, k, v, a, r, ld_prior, frozen, B, H, T, d, dt, workspace, ws_bytes, 0, &c);
    if (st != SAF_OK) return st;
    if (B == 0 || T == 0) return SAF_OK;
    if (!o || !lse) return SAF_EINVAL;
    if (!aligned16(o) || !aligned16(lse)) return SAF_EALIGN;
    if ((st = check_device()) != SAF_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    LayerArgs p = make_args(q, k, v, a, r, ld_prior, B, H, T, c, workspace, 0, 1);
    p.d = d;
    p.out = o;
    p.lse_out = lse;
    p.diag_wait_ns = (unsigned long long)wait_limit_us * 1000ull;
    p.diag_withhold = withhold;
    cudaError_t e = begin_call(p, c, false, true, s);
    if (e == cudaSuccess) e = launch_tc_fwd(p, s);
    return launch_status(e);
}

int saf_attn_fwd(const void* q, const void* k, const void* v, const float* a, const float* r, int ld_prior,
                 const uint8_t* frozen, int B, int H, int T, int d, saf_dtype_t dt, void* o, float* lse,
                 void* workspace, size_t ws_bytes, void* stream) {
    return saf_attn_fwd_gqa(q, k, v, a, r, ld_prior, frozen, B, H, H, T, d, dt, o, lse, workspace, ws_bytes, stream);
}

int saf_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                     const float* a, const float* r, int ld_prior, const uint8_t* frozen, int B, int H, int Hkv, int T,
                     int d, saf_dtype_t dt, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                     void* stream) {
    if (Hkv <= 0 || H <= 0 || H % Hkv != 0) return SAF_EINVAL;
    Common c;
    int st = validate(q, k, v, a, r, ld_prior, frozen, B, H, T, d, dt, workspace, ws_bytes, 1, &c);
    if (st != SAF_OK) return st;
    if (B == 0 || T == 0) return SAF_OK;
    if (!o || !dO || !lse || !dq || !dk || !dv) return SAF_EINVAL;
    if (!aligned16(o) || !aligned16(dO) || !aligned16(lse) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
        return SAF_EALIGN;
    if ((st = check_device()) != SAF_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    LayerArgs p = make_args(q, k, v, a, r, ld_prior, B, H, T, c, workspace, 1, dt == SAF_BF16);
    p.Hkv = Hkv;
    p.d = d;
    p.o = o;
    p.dO = dO;
    p.lse = lse;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    const bool bf16 = dt == SAF_BF16;
    cudaError_t e = begin_call(p, c, true, bf16, s);
    if (bf16 && d != kHeadDim) {
        if (e == cudaSuccess) e = launch_dh_bwd(p, s);
    } else if (bf16) {
        if (e == cudaSuccess) e = launch_bwd_prep(p, s);
        if (e == cudaSuccess) e = launch_tc_bwd(p, s);
    } else {
        if (e == cudaSuccess && c.nfrozen < H) e = launch_bwd_delta(p, false, s);
        if (e == cudaSuccess) e = launch_simt_bwd(p, false, s);
    }
    return launch_status(e);
}

int saf_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 const float* a, const float* r, int ld_prior, const uint8_t* frozen, int B, int H, int T, int d,
                 saf_dtype_t dt, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, void* stream) {
    return saf_attn_bwd_gqa(q, k, v, o, dO, lse, a, r, ld_prior, frozen, B, H, H, T, d, dt, dq, dk, dv, workspace,
                            ws_bytes, stream);
}

// ---------------------------------------------------------------------------
// Prepared frozen-pattern state: the normalisers and padded slices of the frozen
// heads, computed once for fixed (a, r) and reused by every call.
// ---------------------------------------------------------------------------

size_t saf_frozen_state_bytes(int H, int T, saf_dtype_t dt) {
    if (H <= 0 || H > SAF_MAX_HEADS || T <= 0) return 0;
    if (dt != SAF_BF16 && dt != SAF_FP32) return 0;
    return workspace_layout(0, H, T, 0, dt == SAF_BF16).total;
}

int saf_frozen_prepare(const float* a, const float* r, int ld_prior, const uint8_t* frozen, int H, int T,
                       saf_dtype_t dt, void* state, size_t state_bytes, void* stream) {
    if (H <= 0 || H > SAF_MAX_HEADS || T <= 0) return SAF_EINVAL;
    if (dt != SAF_BF16 && dt != SAF_FP32) return SAF_EINVAL;
    Common c;
    memset(&c, 0, sizeof(c));
    for (int h = 0; h < H; ++h)
        if (frozen && frozen[h]) {
            c.mask.w[h >> 6] |= 1ull << (h & 63);
            c.nfrozen++;
        }
    if (c.nfrozen > 0 && (!a || !r || ld_prior < T)) return SAF_EINVAL;
    if ((a && ((uintptr_t)a & 3u)) || (r && ((uintptr_t)r & 3u))) return SAF_EALIGN;
    if (!state) return SAF_EWORKSPACE;
    if (((uintptr_t)state & 255u) != 0) return SAF_EALIGN;
    if (state_bytes < saf_frozen_state_bytes(H, T, dt)) return SAF_EWORKSPACE;
    int st = check_device();
    if (st != SAF_OK) return st;
    const bool bf16 = dt == SAF_BF16;
    LayerArgs p = make_args(nullptr, nullptr, nullptr, a, r, ld_prior, 0, H, T, c, state, 0, bf16);
    return launch_status(begin_call(p, c, false, bf16, (cudaStream_t)stream));
}

namespace saf {
namespace {
// The frozen-pattern fields of p point into a prepared state instead of the workspace.
void use_state(LayerArgs& p, const void* state, int H, int T, bool bf16) {
    const WorkspaceLayout L = workspace_layout(0, H, T, 0, bf16);
    char* st = (char*)state;
    p.lz = (float*)(st + L.lz);
    p.hflag = (uint32_t*)(st + L.hflag);
    p.amax = (float*)(st + L.amax);
    p.a2p = bf16 ? (float*)(st + L.a2p) : nullptr;
    p.r2p = bf16 ? (float*)(st + L.r2p) : nullptr;
    p.eap = bf16 ? (float*)(st + L.eap) : nullptr;
    p.erp = bf16 ? (float*)(st + L.erp) : nullptr;
    p.invz = bf16 ? (float*)(st + L.invz) : nullptr;
}
// First kernel of a prepared call: clears the workspace's status words (error word
// and work counters) and nothing else: with no frozen head in its mask the init
// kernel touches no frozen-pattern data, and its per-head flags go to the
// workspace's own (unused) flag region.
cudaError_t clear_call(const LayerArgs& ws_view, bool bf16, cudaStream_t s) {
    LayerArgs q = ws_view;
    memset(&q.mask, 0, sizeof(q.mask));
    return launch_call_init(q, false, bf16, s);
}
}  // namespace
}  // namespace saf

int saf_attn_fwd_prepared(const void* q, const void* k, const void* v, const float* a, const float* r,
                          int ld_prior, const uint8_t* frozen, const void* state, int B, int H, int Hkv, int T, int d,
                          saf_dtype_t dt, void* o, float* lse, void* workspace, size_t ws_bytes, void* stream) {
    if (Hkv <= 0 || H <= 0 || H % Hkv != 0) return SAF_EINVAL;
    Common c;
    int st = validate(q, k, v, a, r, ld_prior, frozen, B, H, T, d, dt, workspace, ws_bytes, 0, &c);
    if (st != SAF_OK) return st;
    if (B == 0 || T == 0) return SAF_OK;
    if (!o || !lse) return SAF_EINVAL;
    if (!aligned16(o) || !aligned16(lse)) return SAF_EALIGN;
    if (!state) return SAF_EWORKSPACE;
    if (((uintptr_t)state & 255u) != 0) return SAF_EALIGN;
    if ((st = check_device()) != SAF_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const bool bf16 = dt == SAF_BF16;
    LayerArgs p = make_args(q, k, v, a, r, ld_prior, B, H, T, c, workspace, 0, bf16);
    p.Hkv = Hkv;
    p.d = d;
    p.out = o;
    p.lse_out = lse;
    cudaError_t e = clear_call(p, bf16, s);
    use_state(p, state, H, T, bf16);
    if (e == cudaSuccess)
        e = !bf16 ? launch_simt_fwd(p, false, s) : d == kHeadDim ? launch_tc_fwd(p, s) : launch_dh_fwd(p, s);
    return launch_status(e);
}

int saf_attn_bwd_prepared(const void* q, const void* k, const void* v, const void* o, const void* dO,
                          const float* lse, const float* a, const float* r, int ld_prior, const uint8_t* frozen,
                          const void* state, int B, int H, int Hkv, int T, int d, saf_dtype_t dt, void* dq, void* dk,
                          void* dv, void* workspace, size_t ws_bytes, void* stream) {
    if (Hkv <= 0 || H <= 0 || H % Hkv != 0) return SAF_EINVAL;
    Common c;
    int st = validate(q, k, v, a, r, ld_prior, frozen, B, H, T, d, dt, workspace, ws_bytes, 1, &c);
    if (st != SAF_OK) return st;
    if (B == 0 || T == 0) return SAF_OK;
    if (!o || !dO || !lse || !dq || !dk || !dv) return SAF_EINVAL;
    if (!aligned16(o) || !aligned16(dO) || !aligned16(lse) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
        return SAF_EALIGN;
    if (!state) return SAF_EWORKSPACE;
    if (((uintptr_t)state & 255u) != 0) return SAF_EALIGN;
    if ((st = check_device()) != SAF_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const bool bf16 = dt == SAF_BF16;
    LayerArgs p = make_args(q, k, v, a, r, ld_prior, B, H, T, c, workspace, 1, bf16);
    p.Hkv = Hkv;
    p.d = d;
    p.o = o;
    p.dO = dO;
    p.lse = lse;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    cudaError_t e = clear_call(p, bf16, s);
    use_state(p, state, H, T, bf16);
    if (bf16 && d != kHeadDim) {
        if (e == cudaSuccess) e = launch_dh_bwd(p, s);
    } else if (bf16) {
        if (e == cudaSuccess) e = launch_bwd_prep(p, s, false);
        if (e == cudaSuccess) e = launch_tc_bwd(p, s);
    } else {
        if (e == cudaSuccess && c.nfrozen < H) e = launch_bwd_delta(p, false, s);
        if (e == cudaSuccess) e = launch_simt_bwd(p, false, s);
    }
    return launch_status(e);
}

int saf_device_status(const void* workspace, void* stream) {
    if (!workspace) return SAF_EWORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t words[2] = {0, 0};
    if (cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return SAF_ECUDA;
    }
    if (words[0] & kStatusTimeout) return SAF_ETIMEOUT;
    return SAF_OK;
}

const char* saf_error_string(int status) {
    switch (status) {
        case SAF_OK: return "ok";
        case SAF_EINVAL: return "invalid argument (null pointer, bad shape, ld_prior < T or too many heads)";
        case SAF_EALIGN: return "misaligned pointer (tensors need 16-byte, workspace 256-byte alignment)";
        case SAF_EUNSUPPORTED: return "unsupported device, head dimension or dtype";
        case SAF_ELAUNCH: return "kernel launch or asynchronous CUDA call failed";
        case SAF_EWORKSPACE: return "workspace missing or smaller than saf_attn_workspace_bytes";
        case SAF_ETIMEOUT: return "a bounded device wait expired";
        case SAF_ECUDA: return "CUDA runtime error";
        case SAF_ESCRATCH: return "problem too large for the 8 MiB fixed scratch of saf_attn_fwd_noalloc";
        default: return "unknown status";
    }
}

}  // extern "C"
