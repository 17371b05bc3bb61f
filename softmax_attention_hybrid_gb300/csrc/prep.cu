// Per-call preparation kernels of the hybrid attention layer.
//
//  * lognorm: the row normalisers log Z(i) of every frozen head
//    ("When Can Attention Heads Be Statically Defined?", §3.2 Eq. 3; §3.3
//    "precomputed normalisers"). They do not depend on the batch.
//  * frozen_prep: per frozen head, a and r in the exact (log2) and the
//    factorised form of Eq. 3, padded so that every tile of the tensor-core
//    kernels reads its slice with one aligned bulk copy.
//  * bwd_delta / bwd_rowvec: D_i = sum_c dO_ic O_ic for the ordinary-head
//    backward (the softmax Jacobian term of Eqs. 5-7 differentiated; App. D.2),
//    the latter together with lse * log2(e) in the per-tile layout of the
//    tensor-core backward.
#include <math.h>

#include "saf_internal.h"

namespace saf {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ float block_max(float x, float* red) {
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = x;
    __syncthreads();
    if (warp == 0) {
        x = lane < (int)(blockDim.x >> 5) ? red[lane] : -INFINITY;
        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) red[0] = x;
    }
    __syncthreads();
    x = red[0];
    __syncthreads();
    return x;
}

// max a and max r of every frozen head (the A and R of the factorised form).
// Grid (H), 1024 threads.
__global__ void __launch_bounds__(1024)
frozen_max_kernel(const float* __restrict__ a_all, const float* __restrict__ r_all, int ld, HeadMask mask, int T,
                  int H, float* __restrict__ amax) {
    const int h = blockIdx.x;
    if (!head_frozen(mask, h)) return;
    const float* a = a_all + (size_t)h * ld;
    const float* r = r_all + (size_t)h * ld;
    __shared__ float red[32];
    float ma = -INFINITY, mr = -INFINITY;
    // 16 loads of a and 16 of r per thread go out before any is used, so that a
    // row of up to 16 K entries costs one memory latency
    constexpr int kPer = 16;
    for (int base = 0; base < T; base += kPer * 1024) {
        float va[kPer], vr[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int j = base + threadIdx.x + 1024 * k;
            va[k] = j < T ? a[j] : -INFINITY;
            vr[k] = j < T ? r[j] : -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            ma = fmaxf(ma, va[k]);
            mr = fmaxf(mr, vr[k]);
        }
    }
    const float A = block_max(ma, red);
    const float R = block_max(mr, red);
    if (threadIdx.x == 0) {
        amax[h] = A;
        amax[H + h] = R;
    }
}

// Eq. 3 factorises: exp(a[j] + r[i-j]) = e^{A+R} * ea[j] * er[i-j] with
// ea = exp(a - A), er = exp(r - R), A = max a, R = max r. So
//     Z(i) = e^{A+R} * sum_{j<=i} ea[j] er[i-j],
// a causal convolution that needs no exp per term. Every factor lies in
// (0, 1]. If the shifted sum falls below 1e-28, terms that matter may have
// left the normal fp32 range; that row is recomputed exactly by a running
// log-sum-exp and the head is flagged (kStatusRange, informational).
//
// lognorm_kernel: one CTA per (frozen head, 128-row tile), numbered so that
// the tiles with the most keys come first: the block scheduler then hands the
// long tiles out early and fills in with short ones. 256 threads. Thread
// (warp w, lane l) sums rows i0 = 128 t + 8 (l % 16) .. +7 over key run
// 2 w + l / 16 of each chunk (16 runs of kLnRun keys), eight keys per step: the
// 15 er values that a step's 8 x 8 products need slide along the band in
// registers, so a step costs 8 er and 8 ea shared loads for 64 FMAs. The er
// staging is padded (one word every 8): a half-warp's rows, 8 apart, and the two
// half-warps' runs, kLnRun apart, then fall on 32 distinct banks. The 16 runs
// meet in shared memory and are added in a fixed order, so the result does not
// depend on scheduling; a row whose sum underflows is recomputed by a running
// log-sum-exp in the exact domain and its head is flagged.
// kPre: ea and er come precomputed (eap, erp of the tensor-core path) and are
// copied into shared memory asynchronously, the next chunk while the current
// one is summed; otherwise every chunk stages exp(a - A), exp(r - R) itself.
constexpr int kLnRows = 128, kLnThreads = 256, kLnRuns = 16, kLnRun = 128, kLnChunk = kLnRuns * kLnRun;
constexpr int kLnBand = kLnChunk + kLnRows;   // er offsets a chunk needs
constexpr int kLnBandPad = kLnBand + kLnBand / 8 + 8;
__device__ __forceinline__ int lz_pad(int x) { return x + (x >> 3); }

__device__ __forceinline__ uint32_t shared_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(shared_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(shared_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <bool kPre>
__global__ void __launch_bounds__(kLnThreads)
lognorm_kernel(const float* __restrict__ a_all, const float* __restrict__ r_all, int ld, HeadMask mask, int T, int H,
               int F, int nrt, int Tp, const float* __restrict__ eap, const float* __restrict__ erp,
               const float* __restrict__ amax, float* __restrict__ lz, uint32_t* __restrict__ hflag,
               uint32_t* __restrict__ status) {
    // unit u: row tile nrt - 1 - u / F (longest first), f-th frozen head
    const int u = blockIdx.x;
    const int rt = nrt - 1 - u / F;
    const int f = u - (u / F) * F;
    int h = 0;
    for (int c = -1; h < H; ++h)
        if (head_frozen(mask, h) && ++c == f) break;
    if (h >= H) return;
    const float* a = a_all + (size_t)h * ld;
    const float* r = r_all + (size_t)h * ld;
    __shared__ __align__(16) float ea_s[2][kLnChunk];
    __shared__ float er_s[2][kLnBandPad];
    __shared__ float part[kLnRuns][kLnRows];
    const float A = amax[h], R = amax[H + h];
    const int I0 = rt * kLnRows;
    const int imax = min(I0 + kLnRows, T) - 1;
    const int nch = imax / kLnChunk + 1;   // chunks of keys 0 .. imax
    // er_s[b][pad(x)] = er at offset base(c) + x, base(c) = I0 - j0 - kLnChunk + 1 (0 outside [0, T));
    // ea_s[b][t] = ea of key j0 + t (keys past imax meet only zero er: their value is not used)
    auto stage = [&](int c, int b) {
        const int j0 = c * kLnChunk;
        const int base = I0 - j0 - kLnChunk + 1;
        if (kPre) {
            const float* eah = eap + (size_t)h * Tp;
            const float* erh = erp + (size_t)h * (Tp + 256) + 127;   // erh[d], d in [-127, Tp + 129)
            for (int q = threadIdx.x; q < kLnChunk / 4; q += kLnThreads) {
                if (j0 + 4 * q < Tp)
                    cp_async16(&ea_s[b][4 * q], eah + j0 + 4 * q);
                else
                    *reinterpret_cast<float4*>(&ea_s[b][4 * q]) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (int t = threadIdx.x; t < kLnBand; t += kLnThreads) {
                const int dl = base + t;
                if (dl >= -127 && dl < Tp + 129)
                    cp_async4(&er_s[b][lz_pad(t)], erh + dl);
                else
                    er_s[b][lz_pad(t)] = 0.f;
            }
        } else {
            for (int t = threadIdx.x; t < kLnBand; t += kLnThreads) {
                if (t < kLnChunk) ea_s[b][t] = (j0 + t <= imax) ? expf(a[j0 + t] - A) : 0.f;
                const int dl = base + t;
                er_s[b][lz_pad(t)] = (dl >= 0 && dl < T) ? expf(r[dl] - R) : 0.f;
            }
        }
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int run = 2 * warp + (lane >> 4);
    const int i0 = I0 + 8 * (lane & 15);   // my 8 rows
    float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    stage(0, 0);
    cp_async_commit();
    for (int c = 0; c < nch; ++c) {
        const int b = c & 1;
        if (c + 1 < nch) stage(c + 1, b ^ 1);
        cp_async_commit();       // (an empty group on the last chunk keeps the count)
        cp_async_wait_prev();    // chunk c has landed
        __syncthreads();
        const int j0 = c * kLnChunk;
        const int base = I0 - j0 - kLnChunk + 1;
        const float* eb = ea_s[b];
        const float* rb = er_s[b];
        const int js = j0 + run * kLnRun;   // my key run js .. js + kLnRun - 1
        if (js <= i0 + 7 && js <= imax) {
            // step at key j: W[t] = er[i0 - j - 7 + t], t = 0..14; row r, key j + m uses W[r - m + 7]
            const int x0 = i0 - js - 7 - base;   // staging index of W[0] at the first step
            float W[15];
#pragma unroll
            for (int t = 0; t < 15; ++t) W[t] = rb[lz_pad(x0 + t)];
            const int nsteps = (min(kLnRun, i0 + 8 - js) + 7) >> 3;
            for (int st = 0; st < nsteps; ++st) {
                const int jj = js - j0 + 8 * st;
                const float4 e0 = *reinterpret_cast<const float4*>(eb + jj);
                const float4 e1 = *reinterpret_cast<const float4*>(eb + jj + 4);
                const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) z[rr] = fmaf(ev[m], W[rr - m + 7], z[rr]);
                // slide the window 8 keys on: W[8..14] = W[0..6], W[0..7] = the next 8 offsets down
#pragma unroll
                for (int t = 14; t >= 8; --t) W[t] = W[t - 8];
                const int xn = x0 - 8 * (st + 1);
#pragma unroll
                for (int t = 0; t < 8; ++t) W[t] = (xn + t >= 0) ? rb[lz_pad(xn + t)] : 0.f;
            }
        }
        __syncthreads();         // buffer b is free for chunk c + 2
    }
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) part[run][8 * (lane & 15) + rr] = z[rr];
    __syncthreads();
    if (threadIdx.x >= kLnRows) return;
    const int i = I0 + threadIdx.x;
    if (i >= T) return;
    float zs = 0.f;
#pragma unroll
    for (int w = 0; w < kLnRuns; ++w) zs += part[w][threadIdx.x];
    float out;
    if (zs >= 1e-28f) {
        out = logf(zs) + A + R;
    } else {
        float m = -INFINITY, sacc = 0.f;
        for (int j = 0; j <= i; ++j) {
            const float x = a[j] + r[i - j];
            if (x > m) {
                sacc = sacc * expf(m - x) + 1.f;
                m = x;
            } else {
                sacc += expf(x - m);
            }
        }
        out = m + logf(sacc);
        atomicOr(hflag + h, 1u);
        atomicOr(status, kStatusRange);
    }
    lz[(size_t)h * T + i] = out;
}

// Per frozen head, the slices that the tensor-core kernels read with aligned
// bulk copies, in two forms of Eq. 3:
//  exact form (log2 domain, -inf padded):
//    a2p[j] = a[j] log2(e) (j < T),   r2p[u] = r[u - 127] log2(e) (0 <= u - 127 < T)
//  factorised form, W(i, k) = er[i - k] ea[k] / Z'(i) with A = max a, R = max r:
//    eap[j] = exp(a[j] - A) (j < T, else 0),  erp[u] = exp(r[u - 127] - R) (else 0),
//    invz[i] = 1 / Z'(i) = exp(A + R - log Z(i)) (i < T, else 0).
// The factorised form is exact up to rounding while every row keeps a term
// within the normal fp32 range; a head with some log Z(i) - A - R < -64
// (Z' < 1.6e-28) is flagged (hflag bit 1) and the kernels use the exact form.
// log Z comes from lz_src (row stride lz_stride): the lognorm output in the
// forward pass, the frozen rows of lse (batch entry 0) in the backward pass.
// A and R come from frozen_max_kernel. Grid (ceil((Tp + 256) / 512), H), 512
// threads, one entry each; padded lengths Tp (a, invz) and Tp + 256 (r).
// kParts: kPrepPad writes a2p, r2p, eap, erp (needs A, R only); kPrepInvz
// writes invz and the hflag bit (needs log Z).
constexpr int kPrepPad = 1, kPrepInvz = 2;
template <int kParts>
__global__ void __launch_bounds__(512)
frozen_prep_kernel(const float* __restrict__ a_all, const float* __restrict__ r_all, int ld, HeadMask mask, int T,
                   int Tp, const float* __restrict__ lz_src, long long lz_stride, float* __restrict__ a2p,
                   float* __restrict__ r2p, float* __restrict__ eap, float* __restrict__ erp,
                   float* __restrict__ invz, uint32_t* __restrict__ hflag, const float* __restrict__ amax, int H) {
    const int h = blockIdx.y;
    if (!head_frozen(mask, h)) return;
    const float* a = a_all + (size_t)h * ld;
    const float* r = r_all + (size_t)h * ld;
    const float* lz = lz_src + (size_t)h * lz_stride;
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    const float A = amax[h], R = amax[H + h];
    const size_t ra = (size_t)h * Tp, rr = (size_t)h * (Tp + 256);
    for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < Tp + 256; u += gridDim.x * blockDim.x) {
        const int dl = u - 127;
        const bool in = dl >= 0 && dl < T;
        if (kParts & kPrepPad) {
            r2p[rr + u] = in ? r[dl] * kLog2e : -INFINITY;
            erp[rr + u] = in ? expf(r[dl] - R) : 0.f;
        }
        if (u < Tp && (kParts & kPrepPad)) {
            a2p[ra + u] = u < T ? a[u] * kLog2e : -INFINITY;
            eap[ra + u] = u < T ? expf(a[u] - A) : 0.f;
        }
        if (u < Tp && (kParts & kPrepInvz)) {
            float iz = 0.f;
            if (u < T) {
                const float sh = lz[u] - A - R;   // log Z'(u)
                if (!(sh >= -64.f)) bad = 1;
                iz = expf(fminf(-sh, 80.f));
            }
            invz[ra + u] = iz;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && bad) atomicOr(hflag + h, 2u);
}

// D_i = sum_c dO_ic * O_ic, one warp per row (d = 64: two elements per lane).
template <typename E>
__global__ void __launch_bounds__(256)
bwd_delta_kernel(const E* __restrict__ o, const E* __restrict__ dO, float* __restrict__ delta, long long rows) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const E* po = o + row * kHeadDim;
    const E* pd = dO + row * kHeadDim;
    float x = 0.f;
    for (int c = lane; c < kHeadDim; c += 32) x = fmaf(to_f(po[c]), to_f(pd[c]), x);
    for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
    if (lane == 0) delta[row] = x;
}

// Per-tile row vectors of the tensor-core backward: for slice bh and query
// block qb, rowvec[(bh * nqb + qb) * 256 + u] holds lse * log2(e) of query
// qb*128 + u (u < 128; +inf past T) and, at u + 128, D of that query (0 past
// T; frozen heads skip the dot product). Four threads per padded row, each
// reading 32 contiguous bytes of O and dO (a warp reads 1 KB of each);
// grid (nqb * 128 / 64, B*H), 256 threads.
__global__ void __launch_bounds__(256)
bwd_rowvec_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
                  const float* __restrict__ lse, HeadMask mask, int H, int T, int nqb, float* __restrict__ rowvec) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * 64 + (threadIdx.x >> 2);
    const int part = threadIdx.x & 3;
    const bool frozen = head_frozen(mask, bh % H);
    float d = 0.f;
    if (i < T && !frozen) {
        const size_t row = (size_t)bh * T + i;
        const uint4* po = reinterpret_cast<const uint4*>(o + row * kHeadDim) + 2 * part;
        const uint4* pd = reinterpret_cast<const uint4*>(dO + row * kHeadDim) + 2 * part;
        const uint4 x0 = __ldg(po), x1 = __ldg(po + 1), y0 = __ldg(pd), y1 = __ldg(pd + 1);
        const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t ys[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            d = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), d);
            d = fmaf(__uint_as_float(xs[e] & 0xffff0000u), __uint_as_float(ys[e] & 0xffff0000u), d);
        }
    }
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    if (part == 0 && i < nqb * 128) {
        float* v = rowvec + ((size_t)bh * nqb + (i >> 7)) * 256;
        v[i & 127] = i < T ? lse[(size_t)bh * T + i] * kLog2e : INFINITY;
        v[128 + (i & 127)] = d;
    }
}

}  // namespace

cudaError_t launch_frozen_max(const LayerArgs& p, cudaStream_t s) {
    frozen_max_kernel<<<p.H, 1024, 0, s>>>(p.a, p.r, p.ld_prior, p.mask, p.T, p.H, p.amax);
    return cudaGetLastError();
}

cudaError_t launch_lognorm(const LayerArgs& p, bool pre, cudaStream_t s) {
    int F = 0;
    for (int h = 0; h < p.H; ++h) F += head_frozen(p.mask, h) ? 1 : 0;
    if (F == 0) return cudaSuccess;
    const int Tp = (p.T + 127) / 128 * 128;
    const int nrt = (p.T + kLnRows - 1) / kLnRows;
    note_launch();
    if (pre)
        lognorm_kernel<true><<<(unsigned)(nrt * F), kLnThreads, 0, s>>>(
            p.a, p.r, p.ld_prior, p.mask, p.T, p.H, F, nrt, Tp, p.eap, p.erp, p.amax, p.lz, p.hflag, p.status);
    else
        lognorm_kernel<false><<<(unsigned)(nrt * F), kLnThreads, 0, s>>>(
            p.a, p.r, p.ld_prior, p.mask, p.T, p.H, F, nrt, Tp, nullptr, nullptr, p.amax, p.lz, p.hflag, p.status);
    return cudaGetLastError();
}

cudaError_t launch_frozen_pad(const LayerArgs& p, cudaStream_t s) {
    const int Tp = (p.T + 127) / 128 * 128;
    note_launch();
    const dim3 grid((unsigned)((Tp + 256 + 511) / 512), (unsigned)p.H);
    frozen_prep_kernel<kPrepPad><<<grid, 512, 0, s>>>(p.a, p.r, p.ld_prior, p.mask, p.T, Tp, nullptr, 0, p.a2p, p.r2p,
                                                       p.eap, p.erp, p.invz, p.hflag, p.amax, p.H);
    return cudaGetLastError();
}

cudaError_t launch_pattern_prep(const LayerArgs& p, const float* lz_src, long long lz_stride, bool pad,
                                cudaStream_t s) {
    const int Tp = (p.T + 127) / 128 * 128;
    before_launch(SAF_KERNEL_PATTERN_PREP, s);
    const dim3 grid((unsigned)((Tp + 256 + 511) / 512), (unsigned)p.H);
    if (pad)
        frozen_prep_kernel<kPrepPad | kPrepInvz><<<grid, 512, 0, s>>>(p.a, p.r, p.ld_prior, p.mask, p.T, Tp, lz_src,
                                                                      lz_stride, p.a2p, p.r2p, p.eap, p.erp, p.invz,
                                                                      p.hflag, p.amax, p.H);
    else
        frozen_prep_kernel<kPrepInvz><<<grid, 512, 0, s>>>(p.a, p.r, p.ld_prior, p.mask, p.T, Tp, lz_src, lz_stride,
                                                           p.a2p, p.r2p, p.eap, p.erp, p.invz, p.hflag, p.amax, p.H);
    after_launch(SAF_KERNEL_PATTERN_PREP, s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_delta(const LayerArgs& p, bool bf16, cudaStream_t s) {
    const long long rows = (long long)p.B * p.H * p.T;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    before_launch(SAF_KERNEL_BWD_DELTA, s);
    if (bf16)
        bwd_delta_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            (const __nv_bfloat16*)p.o, (const __nv_bfloat16*)p.dO, p.delta, rows);
    else
        bwd_delta_kernel<float><<<blocks, 256, 0, s>>>((const float*)p.o, (const float*)p.dO, p.delta, rows);
    after_launch(SAF_KERNEL_BWD_DELTA, s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_rowvec(const LayerArgs& p, cudaStream_t s) {
    const int nqb = (p.T + 127) / 128;
    dim3 grid((unsigned)(nqb * 128 / 64), p.B * p.H);
    before_launch(SAF_KERNEL_BWD_DELTA, s);
    bwd_rowvec_kernel<<<grid, 256, 0, s>>>((const __nv_bfloat16*)p.o, (const __nv_bfloat16*)p.dO, p.lse, p.mask, p.H,
                                           p.T, nqb, p.rowvec);
    after_launch(SAF_KERNEL_BWD_DELTA, s);
    return cudaGetLastError();
}

}  // namespace saf
