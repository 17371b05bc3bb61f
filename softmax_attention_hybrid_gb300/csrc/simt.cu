// fp32-arithmetic kernels of the hybrid attention layer (CUDA cores).
//
// These serve fp32 inputs, where the layer is computed in fp32 throughout
// (tensor cores have no fp32-input mode of full precision). They follow the
// same plan as the tensor-core path:
//   forward  : one launch; each program = (batch, head, 64-row query block);
//              the head's frozen flag picks ordinary online-softmax attention
//              (App. A.1 Eqs. 5-7, FlashAttention-2 tiling) or the frozen
//              pattern rebuilt from a, r and the precomputed log Z (§3.2 Eq. 3,
//              §3.3 "Fused computation"). Causal key blocks only.
//   backward : a key-block pass (dV for every head, dK for ordinary heads)
//              and a query-block pass (dQ for ordinary heads), as App. D.2
//              describes; frozen heads get dV = W^T dO and exact-zero dQ, dK.
//
// Tile: 64 query rows x 64 keys, head dimension D = 64, 96 or 128, 256
// threads. Thread (ty, tx), ty = tid / 16, tx = tid % 16, owns rows
// 4*ty .. 4*ty+3 and the columns tx, tx+16, ... of the key axis (4 of them)
// or of the head-dimension axis (D / 16 of them).
#include <math.h>

#include "saf_internal.h"

namespace saf {
namespace {

constexpr int kB = 64;          // rows per tile (queries and keys)
constexpr int kLd = kB + 1;     // padded fp32 row stride of a (key x query) tile
constexpr int kThreads = 256;
// floats per tile slot: every tile, (rows x D) or (key x query), fits one slot
template <int D>
__host__ __device__ constexpr int tile_floats() { return kB * ((D > kB ? D : kB) + 1); }

// rows r0 .. r0 + 63 of a [T, D] slice into shared memory, row stride D + 1
template <int D, typename E>
__device__ __forceinline__ void load_tile(float* s, const E* g, int r0, int T) {
    for (int e = threadIdx.x; e < kB * D; e += kThreads) {
        const int rr = e / D, c = e - rr * D;
        const int row = r0 + rr;
        s[rr * (D + 1) + c] = row < T ? to_f(g[(size_t)row * D + c]) : 0.f;
    }
}

__device__ __forceinline__ float quad16_max(float x) {
    for (int o = 1; o < 16; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float quad16_sum(float x) {
    for (int o = 1; o < 16; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---------------------------------------------------------------------------
// Forward. Grid (ceil(T/64), B*H).
// ---------------------------------------------------------------------------
template <typename E, int D>
__global__ void __launch_bounds__(kThreads) fwd_kernel(LayerArgs p) {
    extern __shared__ float sm[];
    float* Qs = sm;
    constexpr int LdD = D + 1, NC = D / 16, kT = tile_floats<D>();
    float* Ks = Qs + kT;
    float* Vs = Ks + kT;
    float* Ps = Vs + kT;

    const int T = p.T;
    const int qb = blockIdx.x, bh = blockIdx.y, h = bh % p.H;
    const bool frozen = head_frozen(p.mask, h);
    const size_t base = (size_t)bh * T * D;
    // key/value slice of this query head (grouped-query layout: head h reads h / (H / Hkv))
    const size_t kvbase = ((size_t)(bh / p.H) * p.Hkv + h / (p.H / p.Hkv)) * T * D;
    const E* q = (const E*)p.q + base;
    const E* k = (const E*)p.k + kvbase;
    const E* v = (const E*)p.v + kvbase;
    const float* a = p.a + (size_t)h * p.ld_prior;
    const float* r = p.r + (size_t)h * p.ld_prior;
    const int q0 = qb * kB;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const float scale = 1.f / sqrtf((float)D);

    if (!frozen) load_tile<D>(Qs, q, q0, T);
    float m[4], l[4], lzr[4], acc[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = q0 + ty * 4 + i;
        m[i] = -INFINITY;
        l[i] = 0.f;
        lzr[i] = (frozen && row < T) ? p.lz[(size_t)h * T + row] : 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[i][c] = 0.f;
    }

    for (int kb = 0; kb <= qb; ++kb) {
        __syncthreads();
        if (!frozen) load_tile<D>(Ks, k, kb * kB, T);
        load_tile<D>(Vs, v, kb * kB, T);
        __syncthreads();
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = q0 + ty * 4 + i;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int key = kb * kB + tx + 16 * c;
                if (frozen) {
                    // W(i, j) = exp(a[j] + r[i-j] - log Z(i)), causal (Eq. 3)
                    const bool ok = key <= row && row < T;
                    s[i][c] = ok ? expf(a[key] + r[row - key] - lzr[i]) : 0.f;
                } else {
                    float dot = 0.f;
                    const float* qr = Qs + (ty * 4 + i) * LdD;
                    const float* kr = Ks + (tx + 16 * c) * LdD;
#pragma unroll 16
                    for (int e = 0; e < D; ++e) dot = fmaf(qr[e], kr[e], dot);
                    s[i][c] = (key <= row && key < T) ? dot * scale : -INFINITY;
                }
            }
        }
        if (!frozen) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float mx = fmaxf(fmaxf(s[i][0], s[i][1]), fmaxf(s[i][2], s[i][3]));
                const float mnew = fmaxf(m[i], quad16_max(mx));
                const float corr = expf(m[i] - mnew);
                float ls = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    s[i][c] = expf(s[i][c] - mnew);
                    ls += s[i][c];
                }
                l[i] = l[i] * corr + quad16_sum(ls);
                m[i] = mnew;
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[i][c] *= corr;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) Ps[(ty * 4 + i) * kLd + tx + 16 * c] = s[i][c];
        __syncthreads();
#pragma unroll 4
        for (int j = 0; j < kB; ++j) {
            float vv[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) vv[c] = Vs[j * LdD + tx + 16 * c];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float pij = Ps[(ty * 4 + i) * kLd + j];
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[i][c] = fmaf(pij, vv[c], acc[i][c]);
            }
        }
    }

    E* o = (E*)p.out + base;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = q0 + ty * 4 + i;
        if (row >= T) continue;
        const float inv = frozen ? 1.f : 1.f / l[i];
#pragma unroll
        for (int c = 0; c < NC; ++c) from_f(o + (size_t)row * D + tx + 16 * c, acc[i][c] * inv);
        if (tx == 0) p.lse_out[(size_t)bh * T + row] = frozen ? lzr[i] : m[i] + logf(l[i]);
    }
}

// ---------------------------------------------------------------------------
// Backward, key-block pass. Grid (ceil(T/64), B*Hkv). Program owns keys
// k0..k0+63 of one key/value slice; loops over the query heads that share it
// (grouped-query layout; one head in the multi-head layer) and, for each, over
// query blocks qb >= kb, so that the slice's dV and dK are group sums formed
// without atomics. Thread rows = keys.
// ---------------------------------------------------------------------------
template <typename E, int D>
__global__ void __launch_bounds__(kThreads) bwd_kv_kernel(LayerArgs p) {
    extern __shared__ float sm[];
    constexpr int LdD = D + 1, NC = D / 16, kT = tile_floats<D>();
    float* Ks = sm;
    float* Vs = Ks + kT;
    float* Qs = Vs + kT;
    float* dOs = Qs + kT;
    float* Pt = dOs + kT;    // P^T  [key][query]
    float* dSt = Pt + kT;    // dS^T [key][query]
    __shared__ float rowstat[kB];  // lse (ordinary) or log Z (frozen) per query
    __shared__ float rowD[kB];

    const int T = p.T;
    const int G = p.H / p.Hkv;
    const int kb = blockIdx.x, bkv = blockIdx.y, b = bkv / p.Hkv, hk = bkv % p.Hkv;
    const size_t kvbase = (size_t)bkv * T * D;
    const E* k = (const E*)p.k + kvbase;
    const E* v = (const E*)p.v + kvbase;
    const int k0 = kb * kB;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const float scale = 1.f / sqrtf((float)D);
    bool any_ordinary = false;
    for (int gi = 0; gi < G; ++gi) any_ordinary |= !head_frozen(p.mask, hk * G + gi);

    if (any_ordinary) load_tile<D>(Ks, k, k0, T);
    load_tile<D>(Vs, v, k0, T);
    float dv[4][NC], dk[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < NC; ++c) dv[i][c] = dk[i][c] = 0.f;

    const int nqb = (T + kB - 1) / kB;
    for (int gi = 0; gi < G; ++gi) {
    const int h = hk * G + gi, bh = b * p.H + h;
    const bool frozen = head_frozen(p.mask, h);
    const size_t base = (size_t)bh * T * D;
    const E* q = (const E*)p.q + base;
    const E* dO = (const E*)p.dO + base;
    const float* a = p.a + (size_t)h * p.ld_prior;
    const float* r = p.r + (size_t)h * p.ld_prior;
    for (int qb = kb; qb < nqb; ++qb) {
        const int q0 = qb * kB;
        __syncthreads();
        if (!frozen) load_tile<D>(Qs, q, q0, T);
        load_tile<D>(dOs, dO, q0, T);
        if (tid < kB) {
            const int qi = q0 + tid;
            if (frozen) {
                rowstat[tid] = qi < T ? p.lz[(size_t)h * T + qi] : 0.f;
            } else {
                rowstat[tid] = qi < T ? p.lse[(size_t)bh * T + qi] : 0.f;
                rowD[tid] = qi < T ? p.delta[(size_t)bh * T + qi] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int key = k0 + ty * 4 + i;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int qq = tx + 16 * c;
                const int qi = q0 + qq;
                const bool ok = key <= qi && qi < T;
                float pt, dst = 0.f;
                if (frozen) {
                    pt = ok ? expf(a[key] + r[qi - key] - rowstat[qq]) : 0.f;
                } else {
                    float dot = 0.f, dpt = 0.f;
                    const float* kr = Ks + (ty * 4 + i) * LdD;
                    const float* qr = Qs + qq * LdD;
                    const float* vr = Vs + (ty * 4 + i) * LdD;
                    const float* gr = dOs + qq * LdD;
#pragma unroll 16
                    for (int e = 0; e < D; ++e) {
                        dot = fmaf(kr[e], qr[e], dot);
                        dpt = fmaf(vr[e], gr[e], dpt);
                    }
                    pt = ok ? expf(dot * scale - rowstat[qq]) : 0.f;
                    dst = pt * (dpt - rowD[qq]);
                }
                Pt[(ty * 4 + i) * kLd + qq] = pt;
                dSt[(ty * 4 + i) * kLd + qq] = dst;
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int qq = 0; qq < kB; ++qq) {
            float g[NC], x[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                g[c] = dOs[qq * LdD + tx + 16 * c];
                x[c] = frozen ? 0.f : Qs[qq * LdD + tx + 16 * c];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float pt = Pt[(ty * 4 + i) * kLd + qq];
                const float ds = dSt[(ty * 4 + i) * kLd + qq];
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    dv[i][c] = fmaf(pt, g[c], dv[i][c]);
                    dk[i][c] = fmaf(ds, x[c], dk[i][c]);
                }
            }
        }
    }
    }

    E* dvp = (E*)p.dv + kvbase;
    E* dkp = (E*)p.dk + kvbase;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int key = k0 + ty * 4 + i;
        if (key >= T) continue;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            from_f(dvp + (size_t)key * D + tx + 16 * c, dv[i][c]);
            from_f(dkp + (size_t)key * D + tx + 16 * c, any_ordinary ? dk[i][c] * scale : 0.f);
        }
    }
}

// ---------------------------------------------------------------------------
// Backward, query-block pass (dQ). Grid (ceil(T/64), B*H). Frozen heads
// write zeros.
// ---------------------------------------------------------------------------
template <typename E, int D>
__global__ void __launch_bounds__(kThreads) bwd_q_kernel(LayerArgs p) {
    extern __shared__ float sm[];
    constexpr int LdD = D + 1, NC = D / 16, kT = tile_floats<D>();
    float* Qs = sm;
    float* dOs = Qs + kT;
    float* Ks = dOs + kT;
    float* Vs = Ks + kT;
    float* dSs = Vs + kT;

    const int T = p.T;
    const int qb = blockIdx.x, bh = blockIdx.y, h = bh % p.H;
    const bool frozen = head_frozen(p.mask, h);
    const size_t base = (size_t)bh * T * D;
    E* dq = (E*)p.dq + base;
    const int q0 = qb * kB;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    if (frozen) {
        for (int e = tid; e < kB * D; e += kThreads) {
            const int row = q0 + e / D;
            if (row < T) from_f(dq + (size_t)row * D + e % D, 0.f);
        }
        return;
    }
    const size_t kvbase = ((size_t)(bh / p.H) * p.Hkv + h / (p.H / p.Hkv)) * T * D;
    const E* q = (const E*)p.q + base;
    const E* k = (const E*)p.k + kvbase;
    const E* v = (const E*)p.v + kvbase;
    const E* dO = (const E*)p.dO + base;
    const float scale = 1.f / sqrtf((float)D);

    load_tile<D>(Qs, q, q0, T);
    load_tile<D>(dOs, dO, q0, T);
    float lse[4], Dr[4], acc[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = q0 + ty * 4 + i;
        lse[i] = row < T ? p.lse[(size_t)bh * T + row] : 0.f;
        Dr[i] = row < T ? p.delta[(size_t)bh * T + row] : 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[i][c] = 0.f;
    }
    for (int kb = 0; kb <= qb; ++kb) {
        __syncthreads();
        load_tile<D>(Ks, k, kb * kB, T);
        load_tile<D>(Vs, v, kb * kB, T);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = q0 + ty * 4 + i;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int key = kb * kB + tx + 16 * c;
                float dot = 0.f, dp = 0.f;
                const float* qr = Qs + (ty * 4 + i) * LdD;
                const float* kr = Ks + (tx + 16 * c) * LdD;
                const float* gr = dOs + (ty * 4 + i) * LdD;
                const float* vr = Vs + (tx + 16 * c) * LdD;
#pragma unroll 16
                for (int e = 0; e < D; ++e) {
                    dot = fmaf(qr[e], kr[e], dot);
                    dp = fmaf(gr[e], vr[e], dp);
                }
                const bool ok = key <= row && row < T;
                const float pij = ok ? expf(dot * scale - lse[i]) : 0.f;
                dSs[(ty * 4 + i) * kLd + tx + 16 * c] = pij * (dp - Dr[i]);
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int j = 0; j < kB; ++j) {
            float kk[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) kk[c] = Ks[j * LdD + tx + 16 * c];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float ds = dSs[(ty * 4 + i) * kLd + j];
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[i][c] = fmaf(ds, kk[c], acc[i][c]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = q0 + ty * 4 + i;
        if (row >= T) continue;
#pragma unroll
        for (int c = 0; c < NC; ++c) from_f(dq + (size_t)row * D + tx + 16 * c, acc[i][c] * scale);
    }
}

template <int D, typename K>
cudaError_t launch(K kernel, int id, int tiles, const LayerArgs& p, cudaStream_t s, int slices) {
    const int smem = tiles * tile_floats<D>() * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.T + kB - 1) / kB, slices);
    before_launch(id, s);
    kernel<<<grid, kThreads, smem, s>>>(p);
    after_launch(id, s);
    return cudaGetLastError();
}

template <typename E, int D>
cudaError_t fwd_d(const LayerArgs& p, cudaStream_t s) {
    return launch<D>(fwd_kernel<E, D>, SAF_KERNEL_FWD, 4, p, s, p.B * p.H);
}

template <typename E, int D>
cudaError_t bwd_d(const LayerArgs& p, cudaStream_t s) {
    cudaError_t e = launch<D>(bwd_kv_kernel<E, D>, SAF_KERNEL_BWD_KV, 6, p, s, p.B * p.Hkv);
    if (e != cudaSuccess) return e;
    return launch<D>(bwd_q_kernel<E, D>, SAF_KERNEL_BWD_Q, 5, p, s, p.B * p.H);
}

}  // namespace

cudaError_t launch_simt_fwd(const LayerArgs& p, bool bf16, cudaStream_t s) {
    if (bf16) return fwd_d<__nv_bfloat16, 64>(p, s);
    switch (p.d) {
        case 96: return fwd_d<float, 96>(p, s);
        case 128: return fwd_d<float, 128>(p, s);
        default: return fwd_d<float, 64>(p, s);
    }
}

cudaError_t launch_simt_bwd(const LayerArgs& p, bool bf16, cudaStream_t s) {
    if (bf16) return bwd_d<__nv_bfloat16, 64>(p, s);
    switch (p.d) {
        case 96: return bwd_d<float, 96>(p, s);
        case 128: return bwd_d<float, 128>(p, s);
        default: return bwd_d<float, 64>(p, s);
    }
}

}  // namespace saf
