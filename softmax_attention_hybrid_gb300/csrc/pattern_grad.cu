// Gradients of the frozen patterns' parameters, for the trainable-pattern
// variant ("When Can Attention Heads Be Statically Defined?", App. C.3.2: the
// trainable variant "computes pattern gradients" and refreshes the normalisers
// after each update).
//
// Eq. 3 is a row softmax of the logits L(i, j) = a(j) + r(i - j). With
// G(i, j) = dO_i . V_j (the gradient with respect to W(i, j)) and
// D_i = sum_j W(i, j) G(i, j) = dO_i . O_i, the logit gradient is
//     dL(i, j) = W(i, j) (G(i, j) - D_i),
// and a(j) collects key column j, r(d) the diagonal i - j = d, both summed over
// the batch (one pattern per head, §3.2):
//     da(j) = sum_b sum_{i >= j} dL(i, j),   dr(d) = sum_b sum_{i >= d} dL(i, i - d).
//
// CUDA-core kernel, fp32 arithmetic: one CTA per (64-query, 64-key) causal
// tile of one (batch entry, frozen head). It forms G with a 4 x 4 register
// block per thread over shared-memory tiles, weights it with W rebuilt from
// a, r and log Z (the frozen rows of lse), and adds the tile's column sums and
// its 127 diagonal sums into da, dr with atomic adds (so the order of the
// fp32 additions, and the last bits of the result, vary from run to run).
#include <math.h>
#include <string.h>

#include "saf_internal.h"

namespace saf {
namespace {

constexpr int kPgTile = 64;

template <typename E>
__global__ void __launch_bounds__(256)
pattern_grad_kernel(const E* __restrict__ v, const E* __restrict__ dO, const E* __restrict__ o,
                    const float* __restrict__ lse, const float* __restrict__ a_all, const float* __restrict__ r_all,
                    int ld, HeadMask mask, int H, int T, int d, int F, int ntq, float* __restrict__ da,
                    float* __restrict__ dr) {
    // tile (qt, kt), kt <= qt, numbered row by row: x = qt (qt + 1) / 2 + kt
    const int x = blockIdx.x;
    int qt = (int)((sqrtf(8.f * (float)x + 1.f) - 1.f) * 0.5f);
    while ((qt + 1) * (qt + 2) / 2 <= x) ++qt;
    while (qt * (qt + 1) / 2 > x) --qt;
    const int kt = x - qt * (qt + 1) / 2;
    const int f = blockIdx.y, b = blockIdx.z;
    int h = 0;
    for (int c = -1; h < H; ++h)
        if (head_frozen(mask, h) && ++c == f) break;
    if (h >= H || qt >= ntq) return;
    const int i0 = qt * kPgTile, j0 = kt * kPgTile;
    const size_t slice = ((size_t)b * H + h) * T;
    const float* a = a_all + (size_t)h * ld;
    const float* r = r_all + (size_t)h * ld;

    __shared__ float sA[kPgTile][kPgTile + 1];   // dO rows i0 ..
    __shared__ float sB[kPgTile][kPgTile + 1];   // O rows i0 .., then V rows j0 ..
    __shared__ float sD[kPgTile];
    __shared__ float sCol[16][kPgTile];
    __shared__ float sDiag[2 * kPgTile - 1];
    const int tid = threadIdx.x;
    if (tid < 2 * kPgTile - 1) sDiag[tid] = 0.f;
    if (tid < kPgTile) sD[tid] = 0.f;
    // G block: rows 4 ty .. +3, keys 4 tx .. +3; D and G summed over the head
    // dimension in chunks of 64 columns (zeros past d)
    const int ty = tid >> 4, tx = tid & 15;
    float g[4][4] = {};
    for (int c0 = 0; c0 < d; c0 += kPgTile) {
        for (int e = tid; e < kPgTile * kPgTile; e += 256) {
            const int rr = e / kPgTile, cc = e % kPgTile;
            const int i = i0 + rr;
            const bool in = i < T && c0 + cc < d;
            sA[rr][cc] = in ? to_f(dO[(slice + i) * d + c0 + cc]) : 0.f;
            sB[rr][cc] = in ? to_f(o[(slice + i) * d + c0 + cc]) : 0.f;
        }
        __syncthreads();
        if (tid < kPgTile) {
            float s = 0.f;
            for (int c = 0; c < kPgTile; ++c) s = fmaf(sA[tid][c], sB[tid][c], s);
            sD[tid] += s;   // D_i = dO_i . O_i
        }
        __syncthreads();
        for (int e = tid; e < kPgTile * kPgTile; e += 256) {
            const int rr = e / kPgTile, cc = e % kPgTile;
            const int j = j0 + rr;
            sB[rr][cc] = (j < T && c0 + cc < d) ? to_f(v[(slice + j) * d + c0 + cc]) : 0.f;
        }
        __syncthreads();
        for (int c = 0; c < kPgTile; ++c) {
            float av[4], bv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                av[u] = sA[4 * ty + u][c];
                bv[u] = sB[4 * tx + u][c];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int w = 0; w < 4; ++w) g[u][w] = fmaf(av[u], bv[w], g[u][w]);
        }
        __syncthreads();   // sA, sB are loaded again for the next chunk
    }
    float col[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int rr = 4 * ty + u, i = i0 + rr;
        const float lz = i < T ? lse[slice + i] : 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int cc = 4 * tx + w, j = j0 + cc;
            if (i < T && j <= i) {
                const float wij = expf(a[j] + r[i - j] - lz);   // Eq. 3
                const float dl = wij * (g[u][w] - sD[rr]);
                col[w] += dl;
                atomicAdd(&sDiag[rr - cc + kPgTile - 1], dl);
            }
        }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) sCol[ty][4 * tx + w] = col[w];
    __syncthreads();
    float* dah = da + (size_t)h * T;
    float* drh = dr + (size_t)h * T;
    if (tid < kPgTile) {
        float s = 0.f;
        for (int t = 0; t < 16; ++t) s += sCol[t][tid];
        if (j0 + tid < T && s != 0.f) atomicAdd(dah + j0 + tid, s);
    }
    if (tid < 2 * kPgTile - 1) {
        const int dlt = i0 - j0 + tid - (kPgTile - 1);   // i - j of this diagonal
        if (dlt >= 0 && dlt < T && sDiag[tid] != 0.f) atomicAdd(drh + dlt, sDiag[tid]);
    }
}

}  // namespace
}  // namespace saf

using namespace saf;

extern "C" int saf_pattern_grad(const void* v, const void* dO, const void* o, const float* lse, const float* a,
                                const float* r, int ld_prior, const uint8_t* frozen, int B, int H, int T, int d,
                                saf_dtype_t dt, float* da, float* dr, void* stream) {
    if (B < 0 || H <= 0 || H > SAF_MAX_HEADS || T < 0) return SAF_EINVAL;
    if (dt != SAF_BF16 && dt != SAF_FP32) return SAF_EINVAL;
    if (d != 64 && d != 96 && d != 128) return SAF_EUNSUPPORTED;
    if (!da || !dr) return SAF_EINVAL;
    if (((uintptr_t)da & 3u) || ((uintptr_t)dr & 3u)) return SAF_EALIGN;
    HeadMask mask;
    memset(&mask, 0, sizeof(mask));
    int F = 0;
    for (int h = 0; h < H; ++h)
        if (frozen && frozen[h]) {
            mask.w[h >> 6] |= 1ull << (h & 63);
            ++F;
        }
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) return SAF_OK;
    // every argument and the device are checked before the first work is enqueued
    const bool work = B > 0 && F > 0;
    if (work) {
        if (!v || !dO || !o || !lse || !a || !r || ld_prior < T) return SAF_EINVAL;
        if (((uintptr_t)v | (uintptr_t)dO | (uintptr_t)o | (uintptr_t)lse) & 15u) return SAF_EALIGN;
        if (((uintptr_t)a | (uintptr_t)r) & 3u) return SAF_EALIGN;
    }
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        return SAF_ECUDA;
    }
    if (!(prop.major == 10 && prop.minor == 3)) return SAF_EUNSUPPORTED;
    if (cudaMemsetAsync(da, 0, (size_t)H * T * sizeof(float), s) != cudaSuccess ||
        cudaMemsetAsync(dr, 0, (size_t)H * T * sizeof(float), s) != cudaSuccess) {
        cudaGetLastError();
        return SAF_ELAUNCH;
    }
    if (!work) return SAF_OK;
    const int ntq = (T + kPgTile - 1) / kPgTile;
    const dim3 grid((unsigned)(ntq * (ntq + 1) / 2), (unsigned)F, (unsigned)B);
    note_launch();
    if (dt == SAF_BF16)
        pattern_grad_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            (const __nv_bfloat16*)v, (const __nv_bfloat16*)dO, (const __nv_bfloat16*)o, lse, a, r, ld_prior, mask, H,
            T, d, F, ntq, da, dr);
    else
        pattern_grad_kernel<float><<<grid, 256, 0, s>>>((const float*)v, (const float*)dO, (const float*)o, lse, a, r,
                                                         ld_prior, mask, H, T, d, F, ntq, da, dr);
    if (cudaGetLastError() != cudaSuccess) return SAF_ELAUNCH;
    return SAF_OK;
}
