// Per-call preparation kernels of the hybrid attention layer.
//
//  * call_init: clears the call's status words and flags; per frozen head,
//    max a and max r, and the padded a, r slices in the exact (log2) and the
//    factorised form of Eq. 3, so that every tile of the tensor-core kernels
//    reads its slice with one aligned bulk copy.
//  * lognorm: the row normalisers log Z(i) of every frozen head
//    ("When Can Attention Heads Be Statically Defined?", §3.2 Eq. 3; §3.3
//    "precomputed normalisers"). They do not depend on the batch.
//  * bwd_prep / bwd_delta: D_i = sum_c dO_ic O_ic for the ordinary-head
//    backward (the softmax Jacobian term of Eqs. 5-7 differentiated; App. D.2);
//    bwd_prep also lays out lse * log2(e) per tile, zeroes the dQ accumulator
//    and forms 1 / Z' for the tensor-core backward.
#include <math.h>

#include "saf_internal.h"

namespace saf {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// max over the block of x and of y (red: 64 floats of shared memory)
__device__ float2 block_max2(float x, float y, float* red) {
    for (int o = 16; o > 0; o >>= 1) {
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, o));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[warp] = x;
        red[32 + warp] = y;
    }
    __syncthreads();
    const bool in = lane < (int)(blockDim.x >> 5);
    x = in ? red[lane] : -INFINITY;
    y = in ? red[32 + lane] : -INFINITY;
    for (int o = 16; o > 0; o >>= 1) {
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, o));
    }
    return make_float2(x, y);
}

// Per frozen head, the slices that the tensor-core kernels read with aligned
// bulk copies, in two forms of Eq. 3 (A = max a, R = max r):
//  exact form (log2 domain, -inf padded):
//    a2p[j] = a[j] log2(e) (j < T),   r2p[u] = r[u - 127] log2(e) (0 <= u - 127 < T)
//  factorised form, W(i, k) = er[i - k] ea[k] / Z'(i):
//    eap[j] = exp(a[j] - A) (j < T, else 0),  erp[u] = exp(r[u - 127] - R) (else 0),
//    invz[i] = 1 / Z'(i) = exp(A + R - log Z(i)) (i < T, else 0).
// The factorised form is exact up to rounding while every row keeps a term
// within the normal fp32 range; a head with some log Z(i) - A - R < -64
// (Z' < 1.6e-28) is flagged (hflag bit 1) and the kernels use the exact form.

// call_init_kernel: the first kernel of every call. Block (0, 0) clears the
// status words, block (0, h) the flags of head h (later kernels of the call
// raise them). For a frozen head every block finds max a and max r (the same
// exact values in every block), block (0, h) stores them, and with pad each
// block writes its 1024 entries of the padded slices above.
// Grid (npart, H), 1024 threads; npart = ceil((Tp + 256) / 1024) with pad, else 1.
__global__ void __launch_bounds__(1024)
call_init_kernel(const float* __restrict__ a_all, const float* __restrict__ r_all, int ld, HeadMask mask, int T,
                 int H, int Tp, float* __restrict__ amax, uint32_t* __restrict__ status,
                 uint32_t* __restrict__ hflag, float* __restrict__ a2p, float* __restrict__ r2p,
                 float* __restrict__ eap, float* __restrict__ erp) {
    grid_dep_wait();
    grid_dep_launch();
    const int h = blockIdx.y;
    if (blockIdx.x == 0) {
        if (h == 0 && threadIdx.x < kStatusBytes / sizeof(uint32_t)) status[threadIdx.x] = 0;
        if (threadIdx.x == 0) hflag[h] = 0;
    }
    if (!head_frozen(mask, h)) return;
    const float* a = a_all + (size_t)h * ld;
    const float* r = r_all + (size_t)h * ld;
    __shared__ float red[64];
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
    const float2 m = block_max2(ma, mr, red);
    const float A = m.x, R = m.y;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        amax[h] = A;
        amax[H + h] = R;
    }
    if (!eap) return;
    const int u = blockIdx.x * 1024 + threadIdx.x;
    if (u >= Tp + 256) return;
    const size_t ra = (size_t)h * Tp, rr = (size_t)h * (Tp + 256);
    const int dl = u - 127;
    const bool in = dl >= 0 && dl < T;
    r2p[rr + u] = in ? r[dl] * kLog2e : -INFINITY;
    erp[rr + u] = in ? expf(r[dl] - R) : 0.f;
    if (u < Tp) {
        a2p[ra + u] = u < T ? a[u] * kLog2e : -INFINITY;
        eap[ra + u] = u < T ? expf(a[u] - A) : 0.f;
    }
}

// Thread-block cluster primitives (PTX): rank of this CTA in its cluster, a
// barrier over the cluster's CTAs (release / acquire: shared-memory writes
// before it are visible to every CTA of the cluster after it), and a load
// from another CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(const float* p, uint32_t rank) {
    uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p)), remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Eq. 3 factorises: exp(a[j] + r[i-j]) = e^{A+R} * ea[j] * er[i-j] with
// ea = exp(a - A), er = exp(r - R), A = max a, R = max r. So
//     Z(i) = e^{A+R} * sum_{j<=i} ea[j] er[i-j],
// a causal convolution that needs no exp per term. Every factor lies in
// (0, 1]. If the shifted sum falls below 1e-28, terms that matter may have
// left the normal fp32 range; that row is recomputed exactly by a running
// log-sum-exp and the head is flagged (kStatusRange, informational).
//
// lognorm_kernel: one cluster of kLnSplit CTAs per (frozen head, 128-row
// tile), numbered so that the tiles with the most keys come first. A tile's
// keys 0 .. I0 + 127 form units of 128; CTA s of the cluster takes an even,
// contiguous share of the units (so the CTAs of a cluster finish together),
// in chunks of up to 16 units. The partial sums meet in CTA 0 through
// distributed shared memory and are added in rank order, so the result does
// not depend on scheduling. 256 threads: thread (warp w, lane l) sums rows
// i0 = 128 t + 8 (l % 16) .. +7 over key run 2 w + l / 16 of each chunk (16
// runs of 8 keys per unit in the chunk), eight keys per step. A step's 8 x 8
// products need 15 er values: the 8 of the step's own aligned group and 7 of
// the group the previous step loaded, so each step loads one group of 8 er and
// 8 ea (four 16-byte shared loads) for 64 FMAs, and the two register groups
// swap roles from step to step. The er staging puts four padding words after
// every group of 8: the 16-byte loads of the 8 lanes of a quarter-warp (rows 8
// apart, so groups 1 apart, 12 words) then cover all 32 banks once.
// kPre (tensor-core path): ea and er come from the padded eap, erp slices of
// call_init_kernel, copied into shared memory asynchronously (the next chunk
// while the current one is summed), and CTA 0 also writes 1 / Z' and the
// exact-form flag. Otherwise every chunk stages exp(a - A), exp(r - R) itself.
constexpr int kLnRows = 128, kLnThreads = 256, kLnRuns = 16, kLnUnit = 128, kLnChunkUnits = 16;
constexpr int kLnChunk = kLnChunkUnits * kLnUnit;   // keys per chunk at most (runs of up to 128)
constexpr int kLnBand = kLnChunk + kLnRows;         // er offsets a chunk needs at most (272 groups of 8)
constexpr int kLnBandPad = kLnBand / 8 * 12;
constexpr int kLnSplit = 4;
__device__ __forceinline__ int lz_pad(int x) { return x + 4 * (x >> 3); }

__device__ __forceinline__ uint32_t shared_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(shared_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// z[rr] += sum_m ev[m] * er[i0 + rr - (j + m)]: W[t] = er of staging index x + t,
// lo = W[0..7], hi = W[8..15] (W[15] unused), row rr and key j + m use W[rr - m + 7]
__device__ __forceinline__ void ln_step(float (&z)[8], const float* ep, const float4& l0, const float4& l1,
                                        const float4& h0, const float4& h1) {
    const float4 e0 = *reinterpret_cast<const float4*>(ep);
    const float4 e1 = *reinterpret_cast<const float4*>(ep + 4);
    const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
    const float W[16] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w,
                         h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) z[rr] = fmaf(ev[m], W[rr - m + 7], z[rr]);
}

template <bool kPre>
__global__ void __launch_bounds__(kLnThreads)
lognorm_kernel(const float* __restrict__ a_all, const float* __restrict__ r_all, int ld, HeadMask mask, int T, int H,
               int F, int nrt, int Tp, const float* __restrict__ eap, const float* __restrict__ erp,
               const float* __restrict__ amax, float* __restrict__ lz, float* __restrict__ invz,
               uint32_t* __restrict__ hflag, uint32_t* __restrict__ status) {
    grid_dep_wait();
    grid_dep_launch();
    // cluster u: row tile nrt - 1 - u / F (longest first), f-th frozen head
    const int S = (int)(gridDim.x / (unsigned)(nrt * F));
    const int rank = (int)cluster_rank();
    const int u = blockIdx.x / S;
    const int rt = nrt - 1 - u / F;
    const int f = u - (u / F) * F;
    int h = 0;
    for (int c = -1; h < H; ++h)
        if (head_frozen(mask, h) && ++c == f) break;
    const bool valid = h < H;   // always, for a mask with F frozen heads
    const float* a = a_all + (size_t)(valid ? h : 0) * ld;
    const float* r = r_all + (size_t)(valid ? h : 0) * ld;
    __shared__ __align__(16) float ea_s[2][kLnChunk];
    __shared__ __align__(16) float er_s[2][kLnBandPad];
    __shared__ float tot[kLnRows];
    // the runs' partial sums reuse the first ea buffer once every chunk is summed
    static_assert(kLnRuns * kLnRows <= kLnChunk, "partial sums must fit an ea buffer");
    float(*part)[kLnRows] = reinterpret_cast<float(*)[kLnRows]>(&ea_s[0][0]);
    const float A = valid ? amax[h] : 0.f, R = valid ? amax[H + h] : 0.f;
    const int I0 = rt * kLnRows;
    const int imax = min(I0 + kLnRows, T) - 1;
    // the tile's keys 0 .. I0 + 127 in units of kLnUnit keys; this CTA takes units
    // [ub0, ub1), an even share, in chunks of up to kLnChunk / kLnUnit units
    const int nu = valid ? rt + 1 : 0;
    const int ub0 = rank * nu / S, ub1 = (rank + 1) * nu / S;
    const int nck = (ub1 - ub0 + kLnChunkUnits - 1) / kLnChunkUnits;
    // chunk k: keys j0 .. j0 + L - 1, L = 128 nuc; runs of 8 nuc keys; er offsets
    // base .. base + L + 127, base = I0 - j0 - L + 1, at staging index x = offset - base
    // er_s[b][pad(x)] = er (0 outside [0, T)); ea_s[b][t] = ea of key j0 + t (keys past
    // imax meet only zero er: their value does not matter)
    auto stage = [&](int k, int b) {
        const int ub = ub0 + k * kLnChunkUnits;
        const int nuc = min(kLnChunkUnits, ub1 - ub);
        const int j0 = ub * kLnUnit, L = nuc * kLnUnit;
        const int base = I0 - j0 - L + 1;
        if (kPre) {
            const float* eah = eap + (size_t)h * Tp;
            // erh[d] = er at offset d for d in [-127, Tp + 129); base + 4 q + 127 is a
            // multiple of 4, so every 4-entry group is 16-byte aligned and lies wholly
            // inside or wholly outside the padded row (keys j0 + 4 q < I0 + 128 <= Tp)
            const float* erh = erp + (size_t)h * (Tp + 256) + 127;
            for (int q = threadIdx.x; q < L / 4; q += kLnThreads) cp_async16(&ea_s[b][4 * q], eah + j0 + 4 * q);
            for (int q = threadIdx.x; q < (L + kLnRows) / 4; q += kLnThreads) {
                const int dl = base + 4 * q;
                float* dst = &er_s[b][lz_pad(4 * q)];
                if (dl >= -127 && dl < Tp + 129)
                    cp_async16(dst, erh + dl);
                else
                    *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        } else {
            for (int t = threadIdx.x; t < L + kLnRows; t += kLnThreads) {
                if (t < L) ea_s[b][t] = (j0 + t <= imax) ? expf(a[j0 + t] - A) : 0.f;
                const int dl = base + t;
                er_s[b][lz_pad(t)] = (dl >= 0 && dl < T) ? expf(r[dl] - R) : 0.f;
            }
        }
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int run = 2 * warp + (lane >> 4);
    const int i0 = I0 + 8 * (lane & 15);   // my 8 rows
    float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (nck > 0) stage(0, 0);
    cp_async_commit();
    for (int k = 0, b = 0; k < nck; ++k, b ^= 1) {
        if (k + 1 < nck) stage(k + 1, b ^ 1);
        cp_async_commit();       // (an empty group on the last chunk keeps the count)
        cp_async_wait_prev();    // chunk k has landed
        __syncthreads();
        const int ub = ub0 + k * kLnChunkUnits;
        const int nuc = min(kLnChunkUnits, ub1 - ub);
        const int j0 = ub * kLnUnit, L = nuc * kLnUnit, rl = 8 * nuc;   // rl: keys per run
        const int base = I0 - j0 - L + 1;
        const float* eb = ea_s[b];
        const float* rb = er_s[b];
        const int js = j0 + run * rl;   // my key run js .. js + rl - 1
        if (js <= i0 + 7 && js <= imax) {
            // step st covers keys js + 8 st .. +7; its window starts at staging index
            // x0 - 8 st, x0 = i0 - js - 7 - base = 8 (l % 16) + rl (16 - run) - 8 (a
            // multiple of 8, >= 8 st for every step taken; x0 + 15 < L + 128)
            const int g0 = (i0 - js - 7 - base) >> 3;
            const int nsteps = (min(rl, i0 + 8 - js) + 7) >> 3;
            const float* ep = eb + run * rl;
            auto group = [&](int g, float4& v0, float4& v1) {
                const float* q = rb + 12 * g;
                v0 = *reinterpret_cast<const float4*>(q);
                v1 = *reinterpret_cast<const float4*>(q + 4);
            };
            float4 l0, l1, h0, h1;
            group(g0, l0, l1);
            group(g0 + 1, h0, h1);
            for (int st = 0;;) {
                ln_step(z, ep + 8 * st, l0, l1, h0, h1);
                if (++st >= nsteps) break;
                group(g0 - st, h0, h1);
                ln_step(z, ep + 8 * st, h0, h1, l0, l1);
                if (++st >= nsteps) break;
                group(g0 - st, l0, l1);
            }
        }
        __syncthreads();         // buffer b is free for chunk k + 2
    }
    // (every copy has landed: the last group committed in the loop is empty)
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) part[run][8 * (lane & 15) + rr] = z[rr];
    __syncthreads();
    if (threadIdx.x < kLnRows) {
        float zs = 0.f;
#pragma unroll
        for (int w = 0; w < kLnRuns; ++w) zs += part[w][threadIdx.x];
        tot[threadIdx.x] = zs;
    }
    cluster_barrier();   // every CTA's tot is written
    const int i = I0 + threadIdx.x;
    if (rank == 0 && valid && threadIdx.x < kLnRows && i < Tp) {
        float out = 0.f;
        if (i < T) {
            float zs = 0.f;
            for (int q = 0; q < S; ++q) zs += ld_cluster_f32(&tot[threadIdx.x], (uint32_t)q);
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
        if (kPre) {
            float iz = 0.f;
            if (i < T) {
                const float sh = out - A - R;   // log Z'(i)
                if (!(sh >= -64.f)) atomicOr(hflag + h, 2u);
                iz = expf(fminf(-sh, 80.f));
            }
            invz[(size_t)h * Tp + i] = iz;
        }
    }
    cluster_barrier();   // CTA 0 has read every tot: the other CTAs may exit
}

// D_i = sum_c dO_ic * O_ic, one warp per row (head dimension d: d / 32 elements per lane).
template <typename E>
__global__ void __launch_bounds__(256)
bwd_delta_kernel(const E* __restrict__ o, const E* __restrict__ dO, float* __restrict__ delta, long long rows,
                 int d) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const E* po = o + row * d;
    const E* pd = dO + row * d;
    float x = 0.f;
    for (int c = lane; c < d; c += 32) x = fmaf(to_f(po[c]), to_f(pd[c]), x);
    for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
    if (lane == 0) delta[row] = x;
}

// bwd_prep_kernel: the per-call preparation of the tensor-core backward, one
// launch (after call_init_kernel, which wrote max a, max r and the padded
// slices of the frozen heads).
//  * Blocks [0, BH * 2 nqb): 64 query rows of slice bh each. For query block qb,
//    rowvec[(bh * nqb + qb) * 256 + u] holds lse * log2(e) of query qb*128 + u
//    (u < 128; +inf past T) and, at u + 128, D of that query (0 past T; frozen
//    heads skip the dot product). Four threads per padded row, each reading 32
//    contiguous bytes of O and dO (a warp reads 1 KB of each). For an ordinary
//    head the block also zeroes the block's rows of the fp32 dQ accumulator
//    that the backward reduce-adds into.
//  * Then ceil(Tp / 256) blocks per frozen head: 1 / Z'(i) from log Z(i), read
//    back from the frozen rows of lse (batch entry 0; identical for every
//    batch entry), and the exact-form flag (hflag bit 1).
// 256 threads.
__global__ void __launch_bounds__(256)
bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
                const float* __restrict__ lse, HeadMask mask, int H, int T, int nqb, int BH,
                float* __restrict__ rowvec, float* __restrict__ dq_acc, int Tp, const float* __restrict__ amax,
                float* __restrict__ invz, uint32_t* __restrict__ hflag) {
    grid_dep_wait();
    grid_dep_launch();
    const int per_bh = 2 * nqb;
    const long long nrv = (long long)BH * per_bh;
    if ((long long)blockIdx.x < nrv) {
        const int bh = (int)(blockIdx.x / (unsigned)per_bh);
        const int bx = (int)(blockIdx.x - (unsigned)(bh * per_bh));
        const int i = bx * 64 + (threadIdx.x >> 2);
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
        if (!frozen) {
            const int rows = min(64, T - bx * 64);
            float4* acc = reinterpret_cast<float4*>(dq_acc + ((size_t)bh * T + (size_t)bx * 64) * kHeadDim);
            for (int q = threadIdx.x; q < rows * (kHeadDim / 4); q += 256) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const int nzb = (Tp + 255) / 256;
    const int v = (int)((long long)blockIdx.x - nrv);
    const int f = v / nzb;
    int h = 0;
    for (int c = -1; h < H; ++h)
        if (head_frozen(mask, h) && ++c == f) break;
    const int u = (v - f * nzb) * 256 + threadIdx.x;
    if (h >= H || u >= Tp) return;
    float iz = 0.f;
    if (u < T) {
        const float sh = lse[(size_t)h * T + u] - amax[h] - amax[H + h];   // log Z'(u)
        if (!(sh >= -64.f)) atomicOr(hflag + h, 2u);
        iz = expf(fminf(-sh, 80.f));
    }
    invz[(size_t)h * Tp + u] = iz;
}

}  // namespace

static int count_frozen(const LayerArgs& p) {
    int F = 0;
    for (int h = 0; h < p.H; ++h) F += head_frozen(p.mask, h) ? 1 : 0;
    return F;
}

cudaError_t launch_call_init(const LayerArgs& p, bool pad, bool pdl, cudaStream_t s) {
    const int Tp = (p.T + 127) / 128 * 128;
    const int npart = (pad && count_frozen(p) > 0) ? (Tp + 256 + 1023) / 1024 : 1;
    note_launch();
    return launch_ex(call_init_kernel, dim3((unsigned)npart, (unsigned)p.H), dim3(1024), 0, s, pdl, 1, p.a, p.r,
                     p.ld_prior, p.mask, p.T, p.H, Tp, p.amax, p.status, p.hflag, pad ? p.a2p : nullptr,
                     pad ? p.r2p : nullptr, pad ? p.eap : nullptr, pad ? p.erp : nullptr);
}

cudaError_t launch_lognorm(const LayerArgs& p, bool pre, bool pdl, cudaStream_t s) {
    const int F = count_frozen(p);
    if (F == 0) return cudaSuccess;
    const int Tp = (p.T + 127) / 128 * 128;
    const int nrt = (p.T + kLnRows - 1) / kLnRows;
    const int S = kLnSplit;
    const dim3 grid((unsigned)(nrt * F * S));
    note_launch();
    if (pre)
        return launch_ex(lognorm_kernel<true>, grid, dim3(kLnThreads), 0, s, pdl, S, p.a, p.r, p.ld_prior, p.mask,
                         p.T, p.H, F, nrt, Tp, (const float*)p.eap, (const float*)p.erp, (const float*)p.amax,
                         p.lz, p.invz, p.hflag, p.status);
    return launch_ex(lognorm_kernel<false>, grid, dim3(kLnThreads), 0, s, pdl, S, p.a, p.r, p.ld_prior, p.mask, p.T,
                     p.H, F, nrt, Tp, (const float*)nullptr, (const float*)nullptr, (const float*)p.amax, p.lz,
                     (float*)nullptr, p.hflag, p.status);
}

cudaError_t launch_bwd_delta(const LayerArgs& p, bool bf16, cudaStream_t s) {
    const long long rows = (long long)p.B * p.H * p.T;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    before_launch(SAF_KERNEL_BWD_DELTA, s);
    if (bf16)
        bwd_delta_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            (const __nv_bfloat16*)p.o, (const __nv_bfloat16*)p.dO, p.delta, rows, p.d);
    else
        bwd_delta_kernel<float><<<blocks, 256, 0, s>>>((const float*)p.o, (const float*)p.dO, p.delta, rows, p.d);
    after_launch(SAF_KERNEL_BWD_DELTA, s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const LayerArgs& p, cudaStream_t s, bool frozen_part) {
    const int nqb = (p.T + 127) / 128;
    const int Tp = nqb * 128;
    const int BH = p.B * p.H;
    const long long blocks =
        (long long)BH * 2 * nqb + (frozen_part ? (long long)count_frozen(p) * ((Tp + 255) / 256) : 0);
    before_launch(SAF_KERNEL_BWD_DELTA, s);
    const cudaError_t e = launch_ex(bwd_prep_kernel, dim3((unsigned)blocks), dim3(256), 0, s, true, 1,
                                    (const __nv_bfloat16*)p.o, (const __nv_bfloat16*)p.dO, p.lse, p.mask, p.H, p.T,
                                    nqb, BH, p.rowvec, p.dq_acc, Tp, (const float*)p.amax, p.invz, p.hflag);
    after_launch(SAF_KERNEL_BWD_DELTA, s);
    return e;
}

}  // namespace saf
