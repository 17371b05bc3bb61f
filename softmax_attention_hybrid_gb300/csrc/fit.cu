// Compact fitting of a frozen pattern on the GPU ("When Can Attention Heads Be
// Statically Defined?", §3.2 "Fitting", Eq. 4; App. D.1, Eq. 20; the fitting
// steps of the selection algorithm; settings in App. C.1).
//
// Given a target's sufficient statistics, the key-column sums eta_abs(j) and
// the diagonal sums eta_rel(delta), the fitter minimises Eq. 4,
//     L(a, r) = (1/T) [sum_i log Z(i) - sum_j eta_abs(j) a(j) - sum_d eta_rel(d) r(d)],
// whose gradient (Eq. 20 and its analogue for r) is the fitted pattern's
// marginals minus the target's, over T. Every Adam step therefore needs log Z
// of the current (a, r), which the normaliser kernels of the attention layer
// compute (call_init_kernel for the maxima, lognorm_kernel for the causal
// convolution), and the fitted marginals
//     fa(j) = sum_{i >= j} W(i, j),   fr(d) = sum_{i >= d} W(i, i - d),
// W(i, j) = exp(a(j) + r(i - j) - log Z(i)) from Eq. 3. Each term is a
// probability (at most 1), so the sums are formed in the exact exp form.
#include <math.h>
#include <string.h>

#include "saf_internal.h"

namespace saf {
namespace {

constexpr float kFitFloor = 1e-9f;

// a = 0, r(d) = log max(eta_rel(d) / (T - d), 1e-9), Adam moments 0.
// Grid (ceil(T / 256), H), 256 threads.
__global__ void __launch_bounds__(256)
fit_init_kernel(const float* __restrict__ eta_rel, int T, int H, float* __restrict__ a, float* __restrict__ r,
                float* __restrict__ mom) {
    const int h = blockIdx.y;
    const int j = blockIdx.x * 256 + threadIdx.x;
    if (j >= T) return;
    const size_t o = (size_t)h * T + j;
    a[o] = 0.f;
    r[o] = logf(fmaxf(eta_rel[o] / (float)(T - j), kFitFloor));
    const size_t n = (size_t)H * T;
    for (int k = 0; k < 4; ++k) mom[k * n + o] = 0.f;
}

// out(x) = sum_{i >= x} exp(c(x) + u(i - x) - lz(i)): with (c, u) = (a, r) the
// key-column marginal fa, with (c, u) = (r, a) the diagonal marginal fr.
// Eq. 3 factorises as in the layer's kernels: with C = max c, U = max u,
//     exp(c(x) + u(i - x) - lz(i)) = exp(c(x) - C) * exp(u(i - x) - U) * exp(C + U - lz(i)),
// so a term costs one multiply-add once the factors are staged. Rows with
// lz(i) - C - U < -64 would push the last factor past e^64; their terms are
// formed in the exact exp form instead (the choice is per row i, so every
// thread of the block takes the same branch). Elsewhere a term lost to
// underflow of the first two factors is below e^-23 of its row's total.
// Grid (ceil(T / 128), H, 2) (z = 0: fa, z = 1: fr), 128 threads: thread t of
// block x sums output x = 128 bx + t over i in chunks of 128; the chunk's
// factors and the 255 values of u it meets are staged in shared memory.
__global__ void __launch_bounds__(128)
fit_marginals_kernel(const float* __restrict__ a, const float* __restrict__ r, const float* __restrict__ lz,
                     const float* __restrict__ amax, int T, int H, float* __restrict__ fa, float* __restrict__ fr) {
    const int h = blockIdx.y;
    const bool rel = blockIdx.z != 0;
    const size_t row = (size_t)h * T;
    const float* c = (rel ? r : a) + row;
    const float* u = (rel ? a : r) + row;
    const float* l = lz + row;
    const float C = amax[rel ? H + h : h], U = amax[rel ? h : H + h];
    __shared__ float ls[128], izs[128];
    __shared__ float us[256], eus[256];
    __shared__ int exact_any;
    const int x0 = blockIdx.x * 128;
    const int x = x0 + threadIdx.x;
    const float cx = x < T ? c[x] : 0.f;
    float acc_f = 0.f, acc_x = 0.f;   // factorised terms (without exp(c(x) - C)), exact terms
    for (int i0 = x0; i0 < T; i0 += 128) {
        if (threadIdx.x == 0) exact_any = 0;
        __syncthreads();
        {
            const int i = i0 + threadIdx.x;
            const float li = i < T ? l[i] : INFINITY;
            const float sh = li - C - U;
            const bool ex = i < T && !(sh >= -64.f);
            ls[threadIdx.x] = li;
            izs[threadIdx.x] = (i < T && !ex) ? expf(-sh) : 0.f;
            if (ex) exact_any = 1;
        }
        for (int k = threadIdx.x; k < 255; k += 128) {
            const int d = i0 - x0 - 127 + k;
            const bool in = d >= 0 && d < T;
            us[k] = in ? u[d] : -INFINITY;
            eus[k] = in ? expf(u[d] - U) : 0.f;
        }
        __syncthreads();
        if (x < T) {
            const float* ep = eus + 127 - (int)threadIdx.x;
            if (!exact_any) {
#pragma unroll 8
                for (int t = 0; t < 128; ++t)
                    if (i0 + t >= x) acc_f = fmaf(ep[t], izs[t], acc_f);
            } else {
                const float* up = us + 127 - (int)threadIdx.x;
                for (int t = 0; t < 128; ++t) {
                    const int i = i0 + t;
                    if (i < x || i >= T) continue;
                    if (izs[t] != 0.f)
                        acc_f = fmaf(ep[t], izs[t], acc_f);
                    else
                        acc_x += expf(cx + up[t] - ls[t]);
                }
            }
        }
        __syncthreads();
    }
    if (x < T) (rel ? fr : fa)[row + x] = expf(cx - C) * acc_f + acc_x;
}

// One Adam step (Kingma and Ba, bias-corrected moments) on a and r with the
// gradient of Eq. 4: (fa - eta_abs) / T and (fr - eta_rel) / T.
// mom: [4][H][T] = m_a, v_a, m_r, v_r. c1 = 1 - b1^t, c2 = 1 - b2^t.
__global__ void __launch_bounds__(256)
fit_adam_kernel(const float* __restrict__ eta_abs, const float* __restrict__ eta_rel, const float* __restrict__ fa,
                const float* __restrict__ fr, int T, int H, float lr, float b1, float b2, float eps, float c1,
                float c2, float* __restrict__ a, float* __restrict__ r, float* __restrict__ mom) {
    const int h = blockIdx.y;
    const int j = blockIdx.x * 256 + threadIdx.x;
    if (j >= T) return;
    const size_t o = (size_t)h * T + j;
    const size_t n = (size_t)H * T;
    const float inv_t = 1.f / (float)T;
    const float g[2] = {(fa[o] - eta_abs[o]) * inv_t, (fr[o] - eta_rel[o]) * inv_t};
    float* p[2] = {a, r};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float& m = mom[(2 * k) * n + o];
        float& v = mom[(2 * k + 1) * n + o];
        m = b1 * m + (1.f - b1) * g[k];
        v = b2 * v + (1.f - b2) * g[k] * g[k];
        p[k][o] -= lr * (m / c1) / (sqrtf(v / c2) + eps);
    }
}

// loss[h] = Eq. 4 at the current (a, r), from log Z. One block per head,
// 256 threads; the per-thread strided sums meet in a fixed-order tree.
__global__ void __launch_bounds__(256)
fit_loss_kernel(const float* __restrict__ lz, const float* __restrict__ eta_abs, const float* __restrict__ eta_rel,
                const float* __restrict__ a, const float* __restrict__ r, int T, float* __restrict__ loss) {
    const int h = blockIdx.x;
    const size_t row = (size_t)h * T;
    float s = 0.f;
    for (int i = threadIdx.x; i < T; i += 256)
        s += lz[row + i] - eta_abs[row + i] * a[row + i] - eta_rel[row + i] * r[row + i];
    __shared__ float red[256];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) loss[h] = red[0] / (float)T;
}

// ---------------------------------------------------------------------------
// Target statistics: from a measured mean attention matrix A (dense, [T, T]
// per head) to the fit's inputs. The selection algorithm floors the causal
// entries at 1e-9 and normalises every row (P = floor-and-normalise(A)); the
// fit then needs only the marginals eta_abs(j) = sum_{i >= j} P(i, j) and
// eta_rel(d) = sum_{i >= d} P(i, i - d) (Eq. 4), and the acceptance test needs
// (1/T) sum_i sum_j P log P, since
//     kappa = (1/T) sum_i KL(P(i, .) || W(i, .)) = (1/T) sum P log P + L(a, r)
// with L the Eq. 4 loss at the fitted (a, r) (the cross term is
// sum_ij P(i, j) (a(j) + r(i - j)) - sum_i log Z(i) = T (-L)). P is never stored.
// ---------------------------------------------------------------------------

// One warp per row i of head h: s(i) = sum_{j <= i} f(i, j) with f = max(A, 1e-9),
// and the row's sum_j P log P = (sum_j f log f) / s - log s.
// Grid (ceil(T / 8), H), 256 threads.
__global__ void __launch_bounds__(256)
target_rows_kernel(const float* __restrict__ A, int T, float* __restrict__ rs, float* __restrict__ rplogp) {
    const int h = blockIdx.y;
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (i >= T) return;
    const float* row = A + ((size_t)h * T + i) * T;
    float sum = 0.f, flf = 0.f;
    for (int j = lane; j <= i; j += 32) {
        const float f = fmaxf(row[j], kFitFloor);
        sum += f;
        flf = fmaf(f, logf(f), flf);
    }
    for (int o = 16; o > 0; o >>= 1) {
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
        flf += __shfl_xor_sync(0xffffffffu, flf, o);
    }
    if (lane == 0) {
        rs[(size_t)h * T + i] = sum;
        rplogp[(size_t)h * T + i] = flf / sum - logf(sum);
    }
}

// Marginals of P: thread x of block (bx, h, z) sums column x (z = 0, eta_abs) or
// diagonal x (z = 1, eta_rel) over rows i >= x in a fixed order, so the result
// is the same on every run. Consecutive threads read consecutive addresses of a
// row (column x, or i - x). Grid (ceil(T / 256), H, 2), 256 threads.
__global__ void __launch_bounds__(256)
target_marginals_kernel(const float* __restrict__ A, const float* __restrict__ rs, int T,
                        float* __restrict__ eta_abs, float* __restrict__ eta_rel) {
    const int h = blockIdx.y;
    const bool rel = blockIdx.z != 0;
    const int x = blockIdx.x * 256 + threadIdx.x;
    if (x >= T) return;
    const float* Ah = A + (size_t)h * T * T;
    const float* sh = rs + (size_t)h * T;
    float acc = 0.f;
    for (int i = x; i < T; ++i) {
        const float f = fmaxf(Ah[(size_t)i * T + (rel ? i - x : x)], kFitFloor);
        acc += f / sh[i];
    }
    (rel ? eta_rel : eta_abs)[(size_t)h * T + x] = acc;
}

// negent[h] = (1/T) sum_i rplogp(i); one block per head, fixed-order tree.
__global__ void __launch_bounds__(256)
target_negent_kernel(const float* __restrict__ rplogp, int T, float* __restrict__ negent) {
    const int h = blockIdx.x;
    float s = 0.f;
    for (int i = threadIdx.x; i < T; i += 256) s += rplogp[(size_t)h * T + i];
    __shared__ float red[256];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) negent[h] = red[0] / (float)T;
}

// kappa = negent + L at the fitted parameters; accepted when kappa <= tol.
__global__ void target_kappa_kernel(const float* __restrict__ negent, const float* __restrict__ loss, int H,
                                    float tol, float* __restrict__ kappa, uint8_t* __restrict__ accept) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    const float k = negent[h] + loss[h];
    kappa[h] = k;
    accept[h] = k <= tol ? 1 : 0;
}

struct StatsLayout {
    size_t rs, rplogp, total;
};

struct FitLayout {
    size_t status, hflag, amax, lz, fa, fr, mom, total;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

StatsLayout stats_layout(int H, int T) {
    StatsLayout L;
    const size_t n = (size_t)H * T * sizeof(float);
    L.rs = 0;
    L.rplogp = align256(n);
    L.total = align256(L.rplogp + n);
    return L;
}

FitLayout fit_layout(int H, int T) {
    FitLayout L;
    const size_t n = (size_t)H * T * sizeof(float);
    size_t off = 0;
    L.status = off;
    off = align256(off + kStatusBytes);
    L.hflag = off;
    off = align256(off + (size_t)H * sizeof(uint32_t));
    L.amax = off;
    off = align256(off + 2 * (size_t)H * sizeof(float));
    L.lz = off;
    off = align256(off + n);
    L.fa = off;
    off = align256(off + n);
    L.fr = off;
    off = align256(off + n);
    L.mom = off;
    off = align256(off + 4 * n);
    L.total = off;
    return L;
}

}  // namespace
}  // namespace saf

using namespace saf;

extern "C" size_t saf_fit_workspace_bytes(int H, int T) {
    if (H <= 0 || H > SAF_MAX_HEADS || T <= 0) return 0;
    return fit_layout(H, T).total;
}

namespace saf {
namespace {

int check_fit_device() {
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        return SAF_ECUDA;
    }
    return (prop.major == 10 && prop.minor == 3) ? SAF_OK : SAF_EUNSUPPORTED;
}

// The fit itself, arguments already checked: `steps` Adam steps from the
// start point, then the Eq. 4 loss at the result.
int run_fit(const float* eta_abs, const float* eta_rel, int H, int T, int steps, float lr, float* a, float* r,
            float* loss, char* ws, cudaStream_t s) {
    const FitLayout L = fit_layout(H, T);
    float* lz = (float*)(ws + L.lz);
    float* fa = (float*)(ws + L.fa);
    float* fr = (float*)(ws + L.fr);
    float* mom = (float*)(ws + L.mom);

    // the normaliser kernels of the layer see every head as frozen, with the
    // current parameters as their a and r (row stride T)
    LayerArgs p;
    memset(&p, 0, sizeof(p));
    p.a = a;
    p.r = r;
    p.ld_prior = T;
    p.B = 1;
    p.H = H;
    p.Hkv = H;
    p.T = T;
    for (int h = 0; h < H; ++h) p.mask.w[h >> 6] |= 1ull << (h & 63);
    p.status = (uint32_t*)(ws + L.status);
    p.hflag = (uint32_t*)(ws + L.hflag);
    p.amax = (float*)(ws + L.amax);
    p.lz = lz;

    const dim3 g256((unsigned)((T + 255) / 256), (unsigned)H);
    const dim3 gm((unsigned)((T + 127) / 128), (unsigned)H, 2);
    const float b1 = 0.9f, b2 = 0.999f, eps = 1e-8f;
    cudaError_t e;
    note_launch();
    fit_init_kernel<<<g256, 256, 0, s>>>(eta_rel, T, H, a, r, mom);
    e = cudaGetLastError();
    double p1 = 1.0, p2 = 1.0;
    for (int t = 1; t <= steps && e == cudaSuccess; ++t) {
        e = launch_call_init(p, false, false, s);
        if (e == cudaSuccess) e = launch_lognorm(p, false, false, s);
        if (e != cudaSuccess) break;
        note_launch();
        fit_marginals_kernel<<<gm, 128, 0, s>>>(a, r, lz, p.amax, T, H, fa, fr);
        p1 *= b1;
        p2 *= b2;
        note_launch();
        fit_adam_kernel<<<g256, 256, 0, s>>>(eta_abs, eta_rel, fa, fr, T, H, lr, b1, b2, eps, (float)(1.0 - p1),
                                             (float)(1.0 - p2), a, r, mom);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = launch_call_init(p, false, false, s);
    if (e == cudaSuccess) e = launch_lognorm(p, false, false, s);
    if (e == cudaSuccess) {
        note_launch();
        fit_loss_kernel<<<H, 256, 0, s>>>(lz, eta_abs, eta_rel, a, r, T, loss);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) return SAF_OK;
    cudaGetLastError();
    return SAF_ELAUNCH;
}

// Target statistics into eta_abs, eta_rel [H, T] and negent [H].
int run_stats(const float* A, int H, int T, float* eta_abs, float* eta_rel, float* negent, char* ws,
              cudaStream_t s) {
    const StatsLayout L = stats_layout(H, T);
    float* rs = (float*)(ws + L.rs);
    float* rplogp = (float*)(ws + L.rplogp);
    note_launch();
    target_rows_kernel<<<dim3((unsigned)((T + 7) / 8), (unsigned)H), 256, 0, s>>>(A, T, rs, rplogp);
    note_launch();
    target_marginals_kernel<<<dim3((unsigned)((T + 255) / 256), (unsigned)H, 2), 256, 0, s>>>(A, rs, T, eta_abs,
                                                                                              eta_rel);
    note_launch();
    target_negent_kernel<<<H, 256, 0, s>>>(rplogp, T, negent);
    if (cudaGetLastError() != cudaSuccess) return SAF_ELAUNCH;
    return SAF_OK;
}

// Workspace of saf_fit_from_target: statistics, eta_abs, eta_rel, negent, loss, fit.
struct PipeLayout {
    size_t stats, eta_abs, eta_rel, negent, loss, fit, total;
};
PipeLayout pipe_layout(int H, int T) {
    PipeLayout L;
    const size_t n = (size_t)H * T * sizeof(float);
    size_t off = 0;
    L.stats = off;
    off = align256(off + stats_layout(H, T).total);
    L.eta_abs = off;
    off = align256(off + n);
    L.eta_rel = off;
    off = align256(off + n);
    L.negent = off;
    off = align256(off + (size_t)H * sizeof(float));
    L.loss = off;
    off = align256(off + (size_t)H * sizeof(float));
    L.fit = off;
    off = align256(off + fit_layout(H, T).total);
    L.total = off;
    return L;
}

bool bad_align4(const void* p) { return ((uintptr_t)p & 3u) != 0; }

}  // namespace
}  // namespace saf

extern "C" int saf_fit_compact(const float* eta_abs, const float* eta_rel, int H, int T, int steps, float lr,
                               float* a, float* r, float* loss, void* workspace, size_t ws_bytes, void* stream) {
    if (H <= 0 || H > SAF_MAX_HEADS || T <= 0 || steps < 0 || !(lr > 0.f) || !isfinite(lr)) return SAF_EINVAL;
    if (!eta_abs || !eta_rel || !a || !r || !loss) return SAF_EINVAL;
    const uintptr_t any = (uintptr_t)eta_abs | (uintptr_t)eta_rel | (uintptr_t)a | (uintptr_t)r | (uintptr_t)loss;
    if (any & 3u) return SAF_EALIGN;
    if (!workspace) return SAF_EWORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return SAF_EALIGN;
    if (ws_bytes < fit_layout(H, T).total) return SAF_EWORKSPACE;
    const int st = check_fit_device();
    if (st != SAF_OK) return st;
    return run_fit(eta_abs, eta_rel, H, T, steps, lr, a, r, loss, (char*)workspace, (cudaStream_t)stream);
}

extern "C" size_t saf_fit_stats_workspace_bytes(int H, int T) {
    if (H <= 0 || H > SAF_MAX_HEADS || T <= 0) return 0;
    return stats_layout(H, T).total;
}

extern "C" int saf_fit_target_stats(const float* A, int H, int T, float* eta_abs, float* eta_rel, float* negent,
                                    void* workspace, size_t ws_bytes, void* stream) {
    if (H <= 0 || H > SAF_MAX_HEADS || T <= 0) return SAF_EINVAL;
    if (!A || !eta_abs || !eta_rel || !negent) return SAF_EINVAL;
    if (bad_align4(A) || bad_align4(eta_abs) || bad_align4(eta_rel) || bad_align4(negent)) return SAF_EALIGN;
    if (!workspace) return SAF_EWORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return SAF_EALIGN;
    if (ws_bytes < stats_layout(H, T).total) return SAF_EWORKSPACE;
    const int st = check_fit_device();
    if (st != SAF_OK) return st;
    return run_stats(A, H, T, eta_abs, eta_rel, negent, (char*)workspace, (cudaStream_t)stream);
}

extern "C" size_t saf_fit_from_target_workspace_bytes(int H, int T) {
    if (H <= 0 || H > SAF_MAX_HEADS || T <= 0) return 0;
    return pipe_layout(H, T).total;
}

extern "C" int saf_fit_from_target(const float* A, int H, int T, int steps, float lr, float tol, float* a, float* r,
                                   float* kappa, uint8_t* accept, void* workspace, size_t ws_bytes, void* stream) {
    if (H <= 0 || H > SAF_MAX_HEADS || T <= 0 || steps < 0 || !(lr > 0.f) || !isfinite(lr) || !(tol >= 0.f))
        return SAF_EINVAL;
    if (!A || !a || !r || !kappa || !accept) return SAF_EINVAL;
    if (bad_align4(A) || bad_align4(a) || bad_align4(r) || bad_align4(kappa)) return SAF_EALIGN;
    if (!workspace) return SAF_EWORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return SAF_EALIGN;
    const PipeLayout L = pipe_layout(H, T);
    if (ws_bytes < L.total) return SAF_EWORKSPACE;
    int st = check_fit_device();
    if (st != SAF_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)workspace;
    float* ea = (float*)(ws + L.eta_abs);
    float* er = (float*)(ws + L.eta_rel);
    float* ng = (float*)(ws + L.negent);
    float* ls = (float*)(ws + L.loss);
    if ((st = run_stats(A, H, T, ea, er, ng, ws + L.stats, s)) != SAF_OK) return st;
    if ((st = run_fit(ea, er, H, T, steps, lr, a, r, ls, ws + L.fit, s)) != SAF_OK) return st;
    note_launch();
    target_kappa_kernel<<<(H + 127) / 128, 128, 0, s>>>(ng, ls, H, tol, kappa, accept);
    if (cudaGetLastError() != cudaSuccess) return SAF_ELAUNCH;
    return SAF_OK;
}
