// The layer in bf16 on the tensor cores at head dimensions 96 and 128 (the
// paper's 1B model uses d_h = 96, App. C.5; App. D.2 tests d_h in {64, 96, 128}).
//
// A [128 rows x d] tile is held in shared memory as two 128-byte-swizzled atoms of
// 64 columns, the layout of the d = 64 kernels twice over. At d = 96 the second
// atom's TMA box reaches past the row end, and TMA fills columns 96..127 with
// zeros: they add nothing to Q K^T, and the outputs' columns 96..127 are never
// stored. So one code path serves both head dimensions, padded to 128.
//
// Launches (all with programmatic dependent launch after the layer's call_init
// and, in the forward, lognorm kernels):
//   forward     dh_fwd_kernel        one CTA per (query block, slice): online
//                                    softmax (ordinary) or Eq. 3 in its exact
//                                    form (frozen), O in tensor memory
//   backward    dh_rowvec_kernel     lse * log2(e) and D = dO . O per query block
//               dh_bwd_kv_kernel     one CTA per (key block, slice): dV, dK
//               dh_bwd_q_kernel      one CTA per (query block, slice): dQ
// Each CTA: warps 0-3 own one tile row per thread (the TMEM lanes), warp 4 loads
// with TMA, warp 5 owns tensor memory and issues the MMAs from one thread.
// Every wait is bounded (mbar_wait): on expiry the CTA records the timeout in the
// call's status word, every role gives up, and tensor memory is freed.
#include <math.h>
#include <string.h>

#include "saf_internal.h"
#include "tc_common.cuh"

namespace saf {
namespace {

using namespace tc;

constexpr int kAtom = 128 * 64 * 2;    // 128 rows x 64 bf16, 128-byte swizzle
constexpr int kTile = 2 * kAtom;       // 128 rows x 128 (d padded to 128)
constexpr int kThreads = 192;      // forward: 4 row warps, a TMA warp, an MMA warp
constexpr int kThreadsBwd = 320;   // backward: 8 row warps (a row's columns in two halves), TMA, MMA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Descriptor of k-step k (16 columns of d) of a K-major [128 x 128] tile.
__device__ __forceinline__ uint64_t kmaj(uint32_t tile, int k) {
    return sdesc_sw128(tile + (uint32_t)(k >> 2) * kAtom + (uint32_t)(k & 3) * 32, 16, 1024);
}
// Descriptor of k-step k (16 rows) of a tile read MN-major (d as the N dimension):
// the leading-dimension offset steps from the first 64 columns of d (atom 0) to the
// next (atom 1), so one N = 128 MMA covers the whole padded head dimension.
__device__ __forceinline__ uint64_t mnmaj(uint32_t tile, int k) {
    return sdesc_sw128(tile + (uint32_t)k * 2048, kAtom, 1024);
}

// Load a [128 x 128] tile (two atoms) of tensor map `map` at row y of slice z.
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int y, int z) {
    tma_load_3d(dst, map, bar, 0, y, z);
    tma_load_3d(dst + kAtom, map, bar, 64, y, z);
}

// Columns c0 .. c0 + n - 1 (n a multiple of 32, at most 128, the same in every lane) of a
// warp's 32 bf16 output rows of d elements: lane l holds row row0 + l as n fp32 values, which
// are scaled and rounded; rows l < nrows only. Whole 32-byte sectors per store instruction.
__device__ __forceinline__ void store_rows_cols(__nv_bfloat16* row0, int d, int nrows, int c0, int n,
                                                const uint32_t* v, float scale) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (32 * q < n) {
            uint4 x[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t* w = v + 32 * q + 8 * c;
                x[c] = make_uint4(pack_bf16(__uint_as_float(w[0]) * scale, __uint_as_float(w[1]) * scale),
                                  pack_bf16(__uint_as_float(w[2]) * scale, __uint_as_float(w[3]) * scale),
                                  pack_bf16(__uint_as_float(w[4]) * scale, __uint_as_float(w[5]) * scale),
                                  pack_bf16(__uint_as_float(w[6]) * scale, __uint_as_float(w[7]) * scale));
            }
            store_rows64(reinterpret_cast<uint8_t*>(row0 + c0 + 32 * q), 2 * (size_t)d, nrows, x);
        }
    }
}

// Head kinds of a key-block item, as a compile-time tag so that each kind gets its own
// tile loop: 0 every query head ordinary, 1 every one frozen, 2 mixed.
template <int M>
struct HeadKinds {
    static constexpr int value = M;
};

struct DhParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    __nv_bfloat16* o;
    float* lse;
    __nv_bfloat16 *dq, *dk, *dv;
    const __nv_bfloat16* o_in;
    const __nv_bfloat16* dO;
    const float* lse_in;
    const float* lz;       // [H, T]: log Z of frozen heads
    const float* a2p;      // [H, Tp]: a * log2(e), -inf padded
    const float* r2p;      // [H, Tp + 256]: r * log2(e) shifted by 127, -inf padded
    float* rowvec;         // [B, H, nqb, 256]: lse * log2(e) | D per query block
    uint32_t* status;
    int B, H, T, d, Tp, nqb;
    int Hkv, G;            // key/value heads; query head h reads key/value head h / G
    float scale_log2;      // log2(e) / sqrt(d)
    float scale;           // 1 / sqrt(d)
    HeadMask mask;
};

// ---------------------------------------------------------------------------
// Forward. Two CTAs share an SM (about 99 KB of shared memory and 256 TMEM
// columns each), so that one CTA's MMAs run while the other's rows are in the
// softmax. K and V have a buffer each: K(j + 1) loads while the rows work on
// S(j), V(j + 1) while they work on S(j + 1).
// TMEM: S [0, 128) fp32, P written over S[0, 64) as bf16 pairs | O [128, 256).
// ---------------------------------------------------------------------------
struct FwdSmem {
    static constexpr int q = 0;
    static constexpr int k = kTile;
    static constexpr int v = 2 * kTile;
    static constexpr int vec = 3 * kTile;   // frozen: a2 slice [128] | r2 band [256]
    static constexpr int total = vec + 2048;
};

struct FwdBars {
    uint64_t q_full, k_full, k_empty, v_full, v_empty, s_full, p_ready, o_done, mma_idle;
};

__global__ void __launch_bounds__(kThreads, 2) dh_fwd_kernel(const __grid_constant__ DhParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ FwdBars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qb = p.nqb - 1 - (int)blockIdx.x;   // the longest blocks first
    const int bh = blockIdx.y;
    const int h = bh % p.H;
    const int bkv = (bh / p.H) * p.Hkv + h / p.G;   // key/value slice
    const bool frz = head_frozen(p.mask, h);
    const int nblk = qb + 1;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.k_full, 1);
        mbar_init(&bars.k_empty, 1);
        mbar_init(&bars.v_full, 1);
        mbar_init(&bars.v_empty, 1);
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.p_ready, 4);
        mbar_init(&bars.o_done, 1);
        mbar_init(&bars.mma_idle, 1);
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&tmem_base_sh, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abort = &abort_flag;
    uint32_t* status = p.status;

    if (warp == 4) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            if (!frz) {
                mbar_expect_tx(&bars.q_full, kTile);
                load_tile(sm + FwdSmem::q, &p.tm_q, &bars.q_full, qb * 128, bh);
            }
            float* vec = reinterpret_cast<float*>(sm + FwdSmem::vec);
            for (int j = 0; j < nblk; ++j) {
                // the K buffer is free once S(j - 1) has been computed, the V buffer
                // (and the frozen rows' vectors) once P(j - 1) V has
                if (!frz) {
                    if (!mbar_wait(&bars.k_empty, (j & 1) ^ 1u, abort, status, kStatusTimeout)) break;
                    mbar_expect_tx(&bars.k_full, kTile);
                    load_tile(sm + FwdSmem::k, &p.tm_k, &bars.k_full, j * 128, bkv);
                }
                if (!mbar_wait(&bars.v_empty, (j & 1) ^ 1u, abort, status, kStatusTimeout)) break;
                mbar_expect_tx(&bars.v_full, frz ? kTile + 512 + 1024 : kTile);
                load_tile(sm + FwdSmem::v, &p.tm_v, &bars.v_full, j * 128, bkv);
                if (frz) {
                    bulk_load(vec, p.a2p + (size_t)h * p.Tp + (size_t)j * 128, 512, &bars.v_full);
                    bulk_load(vec + 128, p.r2p + (size_t)h * (p.Tp + 256) + (size_t)(qb - j) * 128, 1024,
                              &bars.v_full);
                }
            }
        }
    } else if (warp == 5) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S = Q K^T
            const uint32_t id_o = idesc_bf16(128, 128, 0, 1);   // O += P V, V MN-major
            const uint32_t d_s = tmem, d_o = tmem + 128;
            const uint32_t sq = smem_u32(sm + FwdSmem::q), sk = smem_u32(sm + FwdSmem::k);
            const uint32_t sv = smem_u32(sm + FwdSmem::v);
            bool ok = true;
            auto issue_s = [&](int j) -> bool {
                if (!mbar_wait(&bars.k_full, j & 1, abort, status, kStatusTimeout)) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) mma_ss(d_s, kmaj(sq, k), kmaj(sk, k), id_s, k > 0);
                mma_commit(&bars.s_full);
                mma_commit(&bars.k_empty);
                return true;
            };
            if (!frz) ok = mbar_wait(&bars.q_full, 0, abort, status, kStatusTimeout) && issue_s(0);
            for (int j = 0; j < nblk && ok; ++j) {
                if (!(ok = mbar_wait(&bars.v_full, j & 1, abort, status, kStatusTimeout))) break;
                if (!(ok = mbar_wait(&bars.p_ready, j & 1, abort, status, kStatusTimeout))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) mma_ts(d_o, d_s + 8 * k, mnmaj(sv, k), id_o, (j > 0 || k > 0) ? 1u : 0u);
                mma_commit(&bars.o_done);
                mma_commit(&bars.v_empty);
                // S(j + 1) overwrites the columns P(j) is read from; MMAs run in issue order
                if (!frz && j + 1 < nblk) ok = issue_s(j + 1);
            }
            mma_commit(&bars.mma_idle);
            mbar_wait_bounded(&bars.mma_idle, 0, kWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------------- softmax / pattern rows
        const int t = threadIdx.x;   // row of the tile = TMEM lane
        const int row = qb * 128 + t;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float m = -INFINITY, l = 0.f;
        const float lz2 = (frz && row < p.T) ? p.lz[(size_t)h * p.T + row] * kLog2e : INFINITY;
        const float* vec = reinterpret_cast<const float*>(sm + FwdSmem::vec);
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            uint32_t pk[64];
            if (!frz) {
                if (!(ok = mbar_wait(&bars.s_full, j & 1, abort, status, kStatusTimeout))) break;
                tc_fence_after();
                float sv[128];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t u[32];
                    tmem_ld32(lane_base + 32 * c4, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) sv[32 * c4 + e] = __uint_as_float(u[e]) * p.scale_log2;
                }
                if (j == qb) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c > t) sv[c] = -INFINITY;
                }
                float mx = m;
#pragma unroll
                for (int c = 0; c < 128; ++c) mx = fmaxf(mx, sv[c]);
                float sum = 0.f;
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    const float e0 = fast_exp2(sv[c] - mx), e1 = fast_exp2(sv[c + 1] - mx);
                    sum += e0 + e1;
                    pk[c >> 1] = pack_bf16(e0, e1);
                }
                const float corr = fast_exp2(m - mx);   // 0 on the first block (m = -inf)
                l = l * corr + sum;
                // P(j - 1) V has been added before O is rescaled (S(j) was computed after it,
                // so its columns are free for P(j) already)
                if (j > 0) {
                    if (!(ok = mbar_wait(&bars.o_done, (j - 1) & 1, abort, status, kStatusTimeout))) break;
                    tc_fence_after();
                    // tcgen05.ld/st are warp-collective: when any row of the warp has a new
                    // maximum, every lane rescales (by exactly 1 where its maximum held)
                    if (__any_sync(0xffffffffu, mx > m)) {
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            uint32_t u[32];
                            tmem_ld32(lane_base + 128 + 32 * c4, u);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * corr);
                            tmem_st32(lane_base + 128 + 32 * c4, u);
                        }
                    }
                }
                m = mx;
            } else {
                if (!(ok = mbar_wait(&bars.v_full, j & 1, abort, status, kStatusTimeout))) break;
                if (j > 0 && !(ok = mbar_wait(&bars.o_done, (j - 1) & 1, abort, status, kStatusTimeout))) break;
                tc_fence_after();
                // W(row, key) = exp2(a2[key] + r2[row - key] - log2 Z(row)) (Eq. 3); the band
                // holds r at distance (qb - j) 128 + t - c at entry 127 + t - c
                const float* band = vec + 128 + 127 + t;
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    const float w0 = fast_exp2(vec[c] + band[-c] - lz2);
                    const float w1 = fast_exp2(vec[c + 1] + band[-c - 1] - lz2);
                    pk[c >> 1] = pack_bf16(w0, w1);
                }
            }
            tmem_st32(lane_base, pk);
            tmem_st32(lane_base + 32, pk + 32);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.p_ready);
        }
        if (ok && mbar_wait_warp(&bars.o_done, (nblk - 1) & 1, abort, status, kStatusTimeout)) {
            tc_fence_after();
            const float inv = frz ? 1.f : 1.f / l;
            uint32_t ov[128];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(lane_base + 128 + 32 * c4, ov + 32 * c4);
            tmem_ld_wait();
            const int row0 = row - lane;
            store_rows_cols(p.o + ((size_t)bh * p.T + row0) * p.d, p.d, p.T - row0, 0, p.d, ov, inv);
            if (row < p.T) p.lse[(size_t)bh * p.T + row] = frz ? lz2 * kLn2 : (m + log2f(l)) * kLn2;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ---------------------------------------------------------------------------
// Backward prep: rowvec[bh, qb, 0..127] = lse * log2(e) (+inf past T),
// rowvec[bh, qb, 128..255] = D = sum_c dO_c O_c (0 past T, and for frozen heads,
// which do not use it). One thread per row, grid (Tp / 128, B H).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) dh_rowvec_kernel(const __grid_constant__ DhParams p) {
    grid_dep_wait();
    grid_dep_launch();
    const int bh = blockIdx.y, qb = blockIdx.x;
    const int i = qb * 128 + threadIdx.x;
    float l2 = INFINITY, dd = 0.f;
    if (i < p.T) {
        const size_t row = (size_t)bh * p.T + i;
        l2 = p.lse_in[row] * kLog2e;
        if (!head_frozen(p.mask, bh % p.H)) {
            const uint4* po = reinterpret_cast<const uint4*>(p.o_in + row * p.d);
            const uint4* pd = reinterpret_cast<const uint4*>(p.dO + row * p.d);
            for (int c = 0; c < p.d / 8; ++c) {
                const uint4 x = __ldg(po + c), y = __ldg(pd + c);
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dd = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), dd);
                    dd = fmaf(__uint_as_float(xs[e] & 0xffff0000u), __uint_as_float(ys[e] & 0xffff0000u), dd);
                }
            }
        }
    }
    float* v = p.rowvec + ((size_t)bh * p.nqb + qb) * 256;
    v[threadIdx.x] = l2;
    v[128 + threadIdx.x] = dd;
}

// TMEM column of k-step k (16 rows of the contraction) of an operand written in
// chunks of 32 rows: chunk c holds its 16 packed pairs at [32 c, 32 c + 16) and the
// second operand's at [32 c + 16, 32 c + 32).
__device__ __forceinline__ uint32_t chunk_col(int k, int second) {
    return 32u * (uint32_t)(k >> 1) + 16u * (uint32_t)second + 8u * (uint32_t)(k & 1);
}

// ---------------------------------------------------------------------------
// Backward, key-block pass: dV, dK of key block kb of key/value slice bkv. The
// tiles run over the G query heads that share the slice (one head in the
// multi-head layer) and, for each, the query blocks kb .. nqb - 1; dV sums every
// head's share, dK the ordinary heads' (zeros when the group has none). Q, dO and
// the row vectors of the next query tile load while this one runs (two stages).
// TMEM: S^T [0, 128) fp32, overwritten chunk by chunk with P^T and dS^T as bf16
//       pairs (chunk c: P^T at [32 c, +16), dS^T at [32 c + 16, +16)) |
//       dP^T [128, 256) | dV [256, 384) | dK [384, 512).
// ---------------------------------------------------------------------------
struct KvSmem {
    static constexpr int k = 0, v = kTile;
    static constexpr int st = 2 * kTile;                  // 2 stages: Q | dO | lse2 [128] | D [128] | r2 band [256]
    static constexpr int st_q = 0, st_do = kTile, st_vec = 2 * kTile;
    static constexpr int st_bytes = 2 * kTile + 2048;
    static constexpr int total = st + 2 * st_bytes;
};

struct KvBars {
    uint64_t kv_full, st_full[2], st_empty[2], sdp_full, pds_ready, tile_done, mma_idle;
};

__global__ void __launch_bounds__(kThreadsBwd, 1) dh_bwd_kv_kernel(const __grid_constant__ DhParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ KvBars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kb = (int)blockIdx.x;
    const int bkv = blockIdx.y;                        // key/value slice
    const int b = bkv / p.Hkv, h0 = (bkv - b * p.Hkv) * p.G;   // its query heads: h0 .. h0 + G - 1
    const int nq = p.nqb - kb;                         // query tiles per query head
    const int ntiles = p.G * nq;
    bool any_ord = false, any_frz = false;
    for (int gi = 0; gi < p.G; ++gi) (head_frozen(p.mask, h0 + gi) ? any_frz : any_ord) = true;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars.kv_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.st_full[i], 1);
            mbar_init(&bars.st_empty[i], 1);
        }
        mbar_init(&bars.sdp_full, 1);
        mbar_init(&bars.pds_ready, 8);
        mbar_init(&bars.tile_done, 1);
        mbar_init(&bars.mma_idle, 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abort = &abort_flag;
    uint32_t* status = p.status;

    if (warp == 8) {
        if (lane == 0) {
            mbar_expect_tx(&bars.kv_full, any_ord ? 2 * kTile : kTile);
            if (any_ord) load_tile(sm + KvSmem::k, &p.tm_k, &bars.kv_full, kb * 128, bkv);
            load_tile(sm + KvSmem::v, &p.tm_v, &bars.kv_full, kb * 128, bkv);
            for (int i = 0, gi = 0, qi = 0; i < ntiles; ++i) {   // tile i: query head h0 + gi, block kb + qi
                const int qb = kb + qi, s = i & 1;
                const int h = h0 + gi, bh = b * p.H + h;
                const bool frz = head_frozen(p.mask, h);
                if (++qi == nq) {
                    qi = 0;
                    ++gi;
                }
                if (!mbar_wait(&bars.st_empty[s], ((i >> 1) & 1) ^ 1u, abort, status, kStatusTimeout)) break;
                uint8_t* st = sm + KvSmem::st + s * KvSmem::st_bytes;
                float* vec = reinterpret_cast<float*>(st + KvSmem::st_vec);
                mbar_expect_tx(&bars.st_full[s], (frz ? kTile : 2 * kTile) + 1024 + (frz ? 1024 : 0));
                if (!frz) load_tile(st + KvSmem::st_q, &p.tm_q, &bars.st_full[s], qb * 128, bh);
                load_tile(st + KvSmem::st_do, &p.tm_do, &bars.st_full[s], qb * 128, bh);
                bulk_load(vec, p.rowvec + ((size_t)bh * p.nqb + qb) * 256, 1024, &bars.st_full[s]);
                if (frz)
                    bulk_load(vec + 256, p.r2p + (size_t)h * (p.Tp + 256) + (size_t)(qb - kb) * 128, 1024,
                              &bars.st_full[s]);
            }
        }
    } else if (warp == 9) {
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S^T = K Q^T, dP^T = V dO^T
            const uint32_t id_n = idesc_bf16(128, 128, 0, 1);   // dV += P^T dO, dK += dS^T Q (B MN-major)
            const uint32_t sk = smem_u32(sm + KvSmem::k), sv = smem_u32(sm + KvSmem::v);
            bool ok = mbar_wait(&bars.kv_full, 0, abort, status, kStatusTimeout);
            auto tiles = [&](auto kinds) {
                constexpr int M = decltype(kinds)::value;
                int nord = 0;   // ordinary tiles so far (the first one starts dK)
                for (int i = 0, gi = 0, qi = 0; i < ntiles && ok; ++i) {
                    const int s = i & 1;
                    const bool frz = M == 0 ? false : M == 1 ? true : head_frozen(p.mask, h0 + gi);
                    if (++qi == nq) {
                        qi = 0;
                        ++gi;
                    }
                    if (!(ok = mbar_wait(&bars.st_full[s], (i >> 1) & 1, abort, status, kStatusTimeout))) break;
                    tc_fence_after();
                    const uint32_t st = smem_u32(sm + KvSmem::st + s * KvSmem::st_bytes);
                    const uint32_t sq = st + KvSmem::st_q, sdo = st + KvSmem::st_do;
                    if (!frz) {
                        // after the previous tile's dV and dK MMAs, which read columns [0, 128)
    #pragma unroll
                        for (int k = 0; k < 8; ++k) mma_ss(tmem, kmaj(sk, k), kmaj(sq, k), id_s, k > 0);
    #pragma unroll
                        for (int k = 0; k < 8; ++k) mma_ss(tmem + 128, kmaj(sv, k), kmaj(sdo, k), id_s, k > 0);
                        mma_commit(&bars.sdp_full);
                    }
                    if (!(ok = mbar_wait(&bars.pds_ready, i & 1, abort, status, kStatusTimeout))) break;
                    tc_fence_after();
    #pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_ts(tmem + 256, tmem + chunk_col(k, 0), mnmaj(sdo, k), id_n, (i > 0 || k > 0) ? 1u : 0u);
                    if (!frz) {
    #pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mma_ts(tmem + 384, tmem + chunk_col(k, 1), mnmaj(sq, k), id_n,
                                   (nord > 0 || k > 0) ? 1u : 0u);
                        ++nord;
                    }
                    mma_commit(&bars.st_empty[s]);
                    mma_commit(&bars.tile_done);
                }
            };
            if (!any_frz)
                tiles(HeadKinds<0>{});
            else if (!any_ord)
                tiles(HeadKinds<1>{});
            else
                tiles(HeadKinds<2>{});
            mma_commit(&bars.mma_idle);
            mbar_wait_bounded(&bars.mma_idle, 0, kWaitLimitNs);
        }
    } else {
        // warp w: key rows 32 (w % 4) .. + 31 (its TMEM lanes), query columns 64 (w / 4) .. + 63
        const int quarter = warp & 3, half = warp >> 2;
        const int t = quarter * 32 + lane;   // key row of the block = TMEM lane
        const int key = kb * 128 + t;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        bool ok = true;
        auto tiles = [&](auto kinds) {
            constexpr int M = decltype(kinds)::value;
            int nord = 0;     // ordinary tiles so far: phases of sdp_full
            float a2k = 0.f;  // a * log2(e) of my key for the current query head (frozen heads)
            for (int i = 0, gi = 0, qi = 0; i < ntiles; ++i) {
                const bool diag = qi == 0;   // the query head's first tile: query block kb
                const int h = h0 + gi;
                const bool frz = M == 0 ? false : M == 1 ? true : head_frozen(p.mask, h);
                if (frz && diag) a2k = p.a2p[(size_t)h * p.Tp + key];   // in flight during the wait below
                if (++qi == nq) {
                    qi = 0;
                    ++gi;
                }
                const int s = i & 1;
                if (!(ok = mbar_wait(&bars.st_full[s], (i >> 1) & 1, abort, status, kStatusTimeout))) break;
                const float* vec =
                    reinterpret_cast<const float*>(sm + KvSmem::st + s * KvSmem::st_bytes + KvSmem::st_vec);
                if (!frz) {
                    // S^T, dP^T of this tile; their commit also means the previous tile's MMAs are done
                    if (!(ok = mbar_wait(&bars.sdp_full, nord & 1, abort, status, kStatusTimeout))) break;
                    ++nord;
                    tc_fence_after();
    #pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c4 = 2 * half + cc;   // chunk of 32 queries
                        uint32_t su[32], du[32], pk[16], dk[16];
                        tmem_ld32(lane_base + 32 * c4, su);
                        tmem_ld32(lane_base + 128 + 32 * c4, du);
                        tmem_ld_wait();
    #pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const int q0 = 32 * c4 + e;
                            float p0 = fast_exp2(__uint_as_float(su[e]) * p.scale_log2 - vec[q0]);
                            float p1 = fast_exp2(__uint_as_float(su[e + 1]) * p.scale_log2 - vec[q0 + 1]);
                            if (diag && q0 < t) p0 = 0.f;
                            if (diag && q0 + 1 < t) p1 = 0.f;
                            const float d0 = p0 * (__uint_as_float(du[e]) - vec[128 + q0]);
                            const float d1 = p1 * (__uint_as_float(du[e + 1]) - vec[128 + q0 + 1]);
                            pk[e >> 1] = pack_bf16(p0, p1);
                            dk[e >> 1] = pack_bf16(d0, d1);
                        }
                        // chunk c4's own columns, already read
                        tmem_st16(lane_base + 32 * c4, pk);
                        tmem_st16(lane_base + 32 * c4 + 16, dk);
                    }
                } else {
                    // W^T(key, q) = exp2(a2[key] + r2[q - key] - log2 Z(q)); the band holds r at
                    // distance i 128 + c - t at entry 127 + c - t. The previous tile's dV MMA has
                    // read its W^T before this one is written.
                    if (i > 0 && !(ok = mbar_wait(&bars.tile_done, (i - 1) & 1, abort, status, kStatusTimeout))) break;
                    tc_fence_after();
                    const float* band = vec + 256 + 127 - t;
    #pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c4 = 2 * half + cc;
                        uint32_t pk[16];
    #pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const int c = 32 * c4 + e;
                            pk[e >> 1] = pack_bf16(fast_exp2(a2k + band[c] - vec[c]),
                                                   fast_exp2(a2k + band[c + 1] - vec[c + 1]));
                        }
                        tmem_st16(lane_base + 32 * c4, pk);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.pds_ready);
            }
        };
        if (!any_frz)
            tiles(HeadKinds<0>{});
        else if (!any_ord)
            tiles(HeadKinds<1>{});
        else
            tiles(HeadKinds<2>{});
        // tcgen05.ld is warp-collective: every lane loads, only rows inside T are stored;
        // each half of the warps writes its 64 columns of dV and dK (those inside d)
        if (ok && mbar_wait_warp(&bars.tile_done, (ntiles - 1) & 1, abort, status, kStatusTimeout)) {
            tc_fence_after();
            const int c0 = 64 * half, n = min(64, p.d - c0);
            const int key0 = key - lane;
            uint32_t v[64];
            tmem_ld32(lane_base + 256 + c0, v);
            tmem_ld32(lane_base + 256 + c0 + 32, v + 32);
            tmem_ld_wait();
            store_rows_cols(p.dv + ((size_t)bkv * p.T + key0) * p.d, p.d, p.T - key0, c0, n, v, 1.f);
            if (any_ord) {
                tmem_ld32(lane_base + 384 + c0, v);
                tmem_ld32(lane_base + 384 + c0 + 32, v + 32);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) v[c] = 0u;
            }
            store_rows_cols(p.dk + ((size_t)bkv * p.T + key0) * p.d, p.d, p.T - key0, c0, n, v, p.scale);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// Backward, query-block pass: dQ of query block qb of an ordinary slice (zeros
// for frozen slices). K and V of the next key block load while this one runs.
// TMEM: S [0, 128) fp32, overwritten chunk by chunk with dS as bf16 pairs
//       (chunk c at [32 c, 32 c + 16)) | dP [128, 256) | dQ [256, 384).
// ---------------------------------------------------------------------------
struct QSmem {
    static constexpr int q = 0, dO = kTile;
    static constexpr int st = 2 * kTile;                  // 2 stages: K | V
    static constexpr int st_k = 0, st_v = kTile;
    static constexpr int st_bytes = 2 * kTile;
    static constexpr int total = st + 2 * st_bytes;
};

struct QBars {
    uint64_t q_full, st_full[2], st_empty[2], sdp_full, ds_ready, tile_done, mma_idle;
};

__global__ void __launch_bounds__(kThreadsBwd, 1) dh_bwd_q_kernel(const __grid_constant__ DhParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ QBars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qb = p.nqb - 1 - (int)blockIdx.x;
    const int bh = blockIdx.y;
    const int h = bh % p.H;
    const int bkv = (bh / p.H) * p.Hkv + h / p.G;   // key/value slice
    if (head_frozen(p.mask, h)) {
        // dQ of a frozen head is exactly zero
        if (threadIdx.x < 128) {
            const int row = qb * 128 + threadIdx.x;
            if (row < p.T) {
                uint4* dst = reinterpret_cast<uint4*>(p.dq + ((size_t)bh * p.T + row) * p.d);
                for (int c = 0; c < p.d / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        return;
    }
    const int nblk = qb + 1;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars.q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.st_full[i], 1);
            mbar_init(&bars.st_empty[i], 1);
        }
        mbar_init(&bars.sdp_full, 1);
        mbar_init(&bars.ds_ready, 8);
        mbar_init(&bars.tile_done, 1);
        mbar_init(&bars.mma_idle, 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abort = &abort_flag;
    uint32_t* status = p.status;

    if (warp == 8) {
        if (lane == 0) {
            mbar_expect_tx(&bars.q_full, 2 * kTile);
            load_tile(sm + QSmem::q, &p.tm_q, &bars.q_full, qb * 128, bh);
            load_tile(sm + QSmem::dO, &p.tm_do, &bars.q_full, qb * 128, bh);
            for (int j = 0; j < nblk; ++j) {
                const int s = j & 1;
                if (!mbar_wait(&bars.st_empty[s], ((j >> 1) & 1) ^ 1u, abort, status, kStatusTimeout)) break;
                uint8_t* st = sm + QSmem::st + s * QSmem::st_bytes;
                mbar_expect_tx(&bars.st_full[s], 2 * kTile);
                load_tile(st + QSmem::st_k, &p.tm_k, &bars.st_full[s], j * 128, bkv);
                load_tile(st + QSmem::st_v, &p.tm_v, &bars.st_full[s], j * 128, bkv);
            }
        }
    } else if (warp == 9) {
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S = Q K^T, dP = dO V^T
            const uint32_t id_n = idesc_bf16(128, 128, 0, 1);   // dQ += dS K (K MN-major)
            const uint32_t sq = smem_u32(sm + QSmem::q), sdo = smem_u32(sm + QSmem::dO);
            bool ok = mbar_wait(&bars.q_full, 0, abort, status, kStatusTimeout);
            for (int j = 0; j < nblk && ok; ++j) {
                const int s = j & 1;
                if (!(ok = mbar_wait(&bars.st_full[s], (j >> 1) & 1, abort, status, kStatusTimeout))) break;
                tc_fence_after();
                const uint32_t st = smem_u32(sm + QSmem::st + s * QSmem::st_bytes);
                const uint32_t sk = st + QSmem::st_k, sv = st + QSmem::st_v;
                // after the previous block's dQ MMAs, which read dS from columns [0, 128)
#pragma unroll
                for (int k = 0; k < 8; ++k) mma_ss(tmem, kmaj(sq, k), kmaj(sk, k), id_s, k > 0);
#pragma unroll
                for (int k = 0; k < 8; ++k) mma_ss(tmem + 128, kmaj(sdo, k), kmaj(sv, k), id_s, k > 0);
                mma_commit(&bars.sdp_full);
                if (!(ok = mbar_wait(&bars.ds_ready, j & 1, abort, status, kStatusTimeout))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ts(tmem + 256, tmem + chunk_col(k, 0), mnmaj(sk, k), id_n, (j > 0 || k > 0) ? 1u : 0u);
                mma_commit(&bars.st_empty[s]);
                mma_commit(&bars.tile_done);
            }
            mma_commit(&bars.mma_idle);
            mbar_wait_bounded(&bars.mma_idle, 0, kWaitLimitNs);
        }
    } else {
        // warp w: query rows 32 (w % 4) .. + 31 (its TMEM lanes), key columns 64 (w / 4) .. + 63
        const int quarter = warp & 3, half = warp >> 2;
        const int t = quarter * 32 + lane;   // query row of the block = TMEM lane
        const int row = qb * 128 + t;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const float* rv = p.rowvec + ((size_t)bh * p.nqb + qb) * 256;
        const float l2 = rv[t], dd = rv[128 + t];
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            if (!(ok = mbar_wait(&bars.sdp_full, j & 1, abort, status, kStatusTimeout))) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c4 = 2 * half + cc;   // chunk of 32 keys
                uint32_t su[32], du[32], dk[16];
                tmem_ld32(lane_base + 32 * c4, su);
                tmem_ld32(lane_base + 128 + 32 * c4, du);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int k0 = 32 * c4 + e;
                    float p0 = fast_exp2(__uint_as_float(su[e]) * p.scale_log2 - l2);
                    float p1 = fast_exp2(__uint_as_float(su[e + 1]) * p.scale_log2 - l2);
                    if (j == qb && k0 > t) p0 = 0.f;
                    if (j == qb && k0 + 1 > t) p1 = 0.f;
                    dk[e >> 1] = pack_bf16(p0 * (__uint_as_float(du[e]) - dd), p1 * (__uint_as_float(du[e + 1]) - dd));
                }
                tmem_st16(lane_base + 32 * c4, dk);   // chunk c4's own columns, already read
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.ds_ready);
        }
        if (ok && mbar_wait_warp(&bars.tile_done, (nblk - 1) & 1, abort, status, kStatusTimeout)) {
            tc_fence_after();
            const int c0 = 64 * half, n = min(64, p.d - c0);
            const int row0 = row - lane;
            uint32_t v[64];
            tmem_ld32(lane_base + 256 + c0, v);
            tmem_ld32(lane_base + 256 + c0 + 32, v + 32);
            tmem_ld_wait();
            store_rows_cols(p.dq + ((size_t)bh * p.T + row0) * p.d, p.d, p.T - row0, c0, n, v, p.scale);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

DhParams make_params(const LayerArgs& a) {
    DhParams p;
    memset(&p, 0, sizeof(p));
    p.B = a.B;
    p.H = a.H;
    p.T = a.T;
    p.d = a.d;
    p.nqb = (a.T + 127) / 128;
    p.Tp = p.nqb * 128;
    p.scale = 1.f / sqrtf((float)a.d);
    p.scale_log2 = kLog2e * p.scale;
    p.mask = a.mask;
    p.status = a.status;
    p.lz = a.lz;
    p.a2p = a.a2p;
    p.r2p = a.r2p;
    p.rowvec = a.rowvec;
    p.Hkv = a.Hkv > 0 ? a.Hkv : a.H;
    p.G = a.H / p.Hkv;
    return p;
}

bool make_maps(DhParams& p, const LayerArgs& a, bool backward) {
    const int BH = a.B * a.H, BHkv = a.B * p.Hkv;
    bool ok = make_tmap_bf16_3d(&p.tm_v, a.v, a.d, a.T, BHkv, 64, 128);
    if (a.q) ok = ok && make_tmap_bf16_3d(&p.tm_q, a.q, a.d, a.T, BH, 64, 128);
    if (a.k) ok = ok && make_tmap_bf16_3d(&p.tm_k, a.k, a.d, a.T, BHkv, 64, 128);
    if (backward) ok = ok && make_tmap_bf16_3d(&p.tm_do, a.dO, a.d, a.T, BH, 64, 128);
    return ok;
}

}  // namespace

cudaError_t launch_dh_fwd(const LayerArgs& a, cudaStream_t s) {
    DhParams p = make_params(a);
    if (!make_maps(p, a, false)) return cudaErrorInvalidValue;
    p.o = (__nv_bfloat16*)a.out;
    p.lse = a.lse_out;
    const int smem = FwdSmem::total + 1024;
    cudaError_t e = cudaFuncSetAttribute(dh_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    before_launch(SAF_KERNEL_FWD, s);
    e = launch_ex(dh_fwd_kernel, dim3((unsigned)p.nqb, (unsigned)(a.B * a.H)), dim3(kThreads), (size_t)smem, s,
                  true, 1, p);
    after_launch(SAF_KERNEL_FWD, s);
    return e;
}

cudaError_t launch_dh_bwd(const LayerArgs& a, cudaStream_t s) {
    DhParams p = make_params(a);
    if (!make_maps(p, a, true)) return cudaErrorInvalidValue;
    p.o_in = (const __nv_bfloat16*)a.o;
    p.dO = (const __nv_bfloat16*)a.dO;
    p.lse_in = a.lse;
    p.dq = (__nv_bfloat16*)a.dq;
    p.dk = (__nv_bfloat16*)a.dk;
    p.dv = (__nv_bfloat16*)a.dv;
    const dim3 grid((unsigned)p.nqb, (unsigned)(a.B * a.H));
    before_launch(SAF_KERNEL_BWD_DELTA, s);
    cudaError_t e = launch_ex(dh_rowvec_kernel, grid, dim3(128), 0, s, true, 1, p);
    after_launch(SAF_KERNEL_BWD_DELTA, s);
    if (e != cudaSuccess) return e;
    const int smem_kv = KvSmem::total + 1024, smem_q = QSmem::total + 1024;
    e = cudaFuncSetAttribute(dh_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(dh_bwd_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q);
    if (e != cudaSuccess) return e;
    before_launch(SAF_KERNEL_BWD_KV, s);
    e = launch_ex(dh_bwd_kv_kernel, dim3((unsigned)p.nqb, (unsigned)(a.B * p.Hkv)), dim3(kThreadsBwd),
                  (size_t)smem_kv, s, true, 1, p);
    after_launch(SAF_KERNEL_BWD_KV, s);
    if (e != cudaSuccess) return e;
    before_launch(SAF_KERNEL_BWD_Q, s);
    e = launch_ex(dh_bwd_q_kernel, grid, dim3(kThreadsBwd), (size_t)smem_q, s, true, 1, p);
    after_launch(SAF_KERNEL_BWD_Q, s);
    return e;
}

}  // namespace saf
