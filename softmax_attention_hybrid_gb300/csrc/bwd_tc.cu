// Fused hybrid backward on the 5th-generation tensor cores (bf16, d = 64).
//
// "When Can Attention Heads Be Statically Defined?", App. D.2: key-block
// programs accumulate value gradients for every head and key gradients for
// ordinary heads. Here one persistent launch runs every key-block program of
// both kinds of head; the query gradients of ordinary heads are produced in
// the same programs (dQ = dS K per tile pair, added into an fp32 accumulator
// in the workspace) instead of by a separate query-block pass that would
// recompute S and dP. Frozen heads compute only dV = W^T dO (§3.3), with W
// rebuilt from a, r and log Z; their dK rows are written as zeros here and
// their dQ rows by the finishing kernel.
//
// Work item: (batch b, head h, key block kb) = key rows [128 kb, 128 kb + 128);
// it loops over query blocks qb = kb .. nqb-1 (causal). Items: all ordinary
// ones by ascending kb (longest first), then all frozen ones, dealt to the
// persistent CTAs in snake order.
//
// Per (kb, qb) tile of an ordinary head (thread j = key row j of the block):
//   S^T  = K Q^T          (tcgen05, TMEM)      P^T = exp(S^T / sqrt(d) - lse)
//   dP^T = V dO^T         (tcgen05, TMEM)      dS  = P o (dP - D)
//   dV  += P^T dO         (A = P^T from TMEM)
//   dK  += dS^T Q         (A = dS in shared memory, K-major view)
//   dQ   = dS K           (A = dS in shared memory, MN-major view) -> red.add
//
// Warp roles (320 threads, one CTA per SM):
//   warps 0-3 : pattern group, thread j = key row j (P^T, dS, or W^T)
//   warps 4-7 : epilogue group: dQ rows to the accumulator; dV, dK rows out
//   warp 8    : TMA producer (K, V per item; Q, dO and row vectors per tile)
//   warp 9    : tensor-memory owner and single-thread MMA issuer
// Tensor memory (512 columns): S^T [0,128) | dP^T [128,256) | P^T bf16
// [256,320) | dV [320,384) | dK [384,448) | dQ [448,512).
#include <string.h>

#include "saf_internal.h"
#include "tc_common.cuh"

namespace saf {
namespace {

using namespace tc;

constexpr int kTileBytes = 128 * 64 * 2;
constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;
constexpr float kScale = 0.125f;

constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDV = 320, kColDK = 384, kColDQ = 448;

struct BwdParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tm_do;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    float* dq_acc;
    const float* lse;
    const float* delta;
    const float* a;
    const float* r;
    const float* lz;
    uint32_t* status;
    int B, H, T, ld;
    int nqb, n_items, n_ord_items;
    int n_ord, n_frz;
    uint8_t ord_heads[SAF_MAX_HEADS];
    uint8_t frz_heads[SAF_MAX_HEADS];
};

struct Smem {
    static constexpr int kv = 0;                        // 2 buffers x (K, V)
    static constexpr int kv_bytes = 2 * kTileBytes;
    static constexpr int st = kv + 2 * kv_bytes;        // 2 stages x (Q, dO)
    static constexpr int st_bytes = 2 * kTileBytes;
    static constexpr int ds = st + 2 * st_bytes;        // 2 buffers x dS (128 x 128 bf16)
    static constexpr int ds_bytes = 2 * kTileBytes;
    static constexpr int vec = ds + 2 * ds_bytes;       // 2 stages x 384 fp32
    static constexpr int vec_floats = 384;
    static constexpr int total = vec + 2 * vec_floats * 4;
};

struct Item {
    int b, h, kb;
    bool frozen;
};

__device__ __forceinline__ Item decode_item(const BwdParams& p, int idx) {
    Item it;
    if (idx < p.n_ord_items) {
        const int per = p.B * p.n_ord;
        it.kb = idx / per;
        const int rem = idx - it.kb * per;
        it.b = rem / p.n_ord;
        it.h = p.ord_heads[rem - it.b * p.n_ord];
        it.frozen = false;
    } else {
        const int f = idx - p.n_ord_items;
        const int per = p.B * p.n_frz;
        it.kb = f / per;
        const int rem = f - it.kb * per;
        it.b = rem / p.n_frz;
        it.h = p.frz_heads[rem - it.b * p.n_frz];
        it.frozen = true;
    }
    return it;
}

__device__ __forceinline__ int item_index(int round, int cta, int grid) {
    return round * grid + ((round & 1) ? (grid - 1 - cta) : cta);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

struct Barriers {
    uint64_t kv_full[2], kv_empty[2];
    uint64_t st_full[2], st_empty[2];
    uint64_t s_full;          // S^T and dP^T of the current tile are in TMEM
    uint64_t p_ready;         // P^T in TMEM and dS in shared memory (128 arrivals)
    uint64_t p_free;          // the dV MMA has read P^T
    uint64_t ds_free[2];      // dK and dQ MMAs have read dS buffer b
    uint64_t dq_full, dq_free;
    uint64_t dkv_full, dkv_free;
};

__global__ void __launch_bounds__(kThreads, 1) bwd_tc_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Barriers bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.kv_full[i], 1);
            mbar_init(&bars.kv_empty[i], 1);
            mbar_init(&bars.st_full[i], 1 + 32);   // TMA transaction arrive + 32 producer lanes
            mbar_init(&bars.st_empty[i], 1);
            mbar_init(&bars.ds_free[i], 1);
        }
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.p_ready, 128);
        mbar_init(&bars.p_free, 1);
        mbar_init(&bars.dq_full, 1);
        mbar_init(&bars.dq_free, 128);
        mbar_init(&bars.dkv_full, 1);
        mbar_init(&bars.dkv_free, 128);
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
    const int grid = gridDim.x, cta = blockIdx.x;
    const int nqb = p.nqb;

    if (warp == 8) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_do);
        }
        uint32_t kv_empty_bits = 3u, st_empty_bits = 3u;
        int kvbuf = 0, stage = 0;
        bool ok = true;
        for (int round = 0; ok; ++round) {
            const int idx = item_index(round, cta, grid);
            if (idx >= p.n_items) break;
            const Item it = decode_item(p, idx);
            const int bh = it.b * p.H + it.h;
            if (!it.frozen) {
                if (lane == 0) {
                    ok = mbar_wait(&bars.kv_empty[kvbuf], (kv_empty_bits >> kvbuf) & 1u, abort, status,
                                   kStatusTimeout);
                    if (ok) {
                        uint8_t* kv = sm + Smem::kv + kvbuf * Smem::kv_bytes;
                        mbar_expect_tx(&bars.kv_full[kvbuf], 2 * kTileBytes);
                        tma_load_3d(kv, &p.tm_k, &bars.kv_full[kvbuf], 0, it.kb * 128, bh);
                        tma_load_3d(kv + kTileBytes, &p.tm_v, &bars.kv_full[kvbuf], 0, it.kb * 128, bh);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                kv_empty_bits ^= 1u << kvbuf;
                kvbuf ^= 1;
            }
            const float* lse_row = p.lse + (size_t)bh * p.T;
            const float* dl_row = p.delta + (size_t)bh * p.T;
            const float* lz_row = p.lz + (size_t)it.h * p.T;
            const float* r_row = p.r + (size_t)it.h * p.ld;
            for (int qb = it.kb; qb < nqb; ++qb) {
                ok = mbar_wait(&bars.st_empty[stage], (st_empty_bits >> stage) & 1u, abort, status, kStatusTimeout);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                st_empty_bits ^= 1u << stage;
                uint8_t* st = sm + Smem::st + stage * Smem::st_bytes;
                if (lane == 0) {
                    mbar_expect_tx(&bars.st_full[stage], (it.frozen ? 1 : 2) * kTileBytes);
                    if (!it.frozen) tma_load_3d(st, &p.tm_q, &bars.st_full[stage], 0, qb * 128, bh);
                    tma_load_3d(st + kTileBytes, &p.tm_do, &bars.st_full[stage], 0, qb * 128, bh);
                }
                float* vec = reinterpret_cast<float*>(sm + Smem::vec + stage * Smem::vec_floats * 4);
                if (!it.frozen) {
                    // vec[0..128): lse * log2(e) (+inf past T), vec[128..256): D (0 past T)
                    for (int u = lane; u < 128; u += 32) {
                        const int q = qb * 128 + u;
                        vec[u] = q < p.T ? lse_row[q] * kLog2e : INFINITY;
                        vec[128 + u] = q < p.T ? dl_row[q] : 0.f;
                    }
                } else {
                    // vec[0..128): log Z * log2(e) (+inf past T); vec[128..383): r * log2(e) over the
                    // offsets (qb - kb) * 128 - 127 + u (-inf outside [0, T))
                    const int d0 = (qb - it.kb) * 128 - 127;
                    for (int u = lane; u < 128; u += 32) {
                        const int q = qb * 128 + u;
                        vec[u] = q < p.T ? lz_row[q] * kLog2e : INFINITY;
                    }
                    for (int u = lane; u < 255; u += 32) {
                        const int dl = d0 + u;
                        vec[128 + u] = (dl >= 0 && dl < p.T) ? r_row[dl] * kLog2e : -INFINITY;
                    }
                }
                mbar_arrive(&bars.st_full[stage]);
                stage ^= 1;
            }
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S^T = K Q^T, dP^T = V dO^T
            const uint32_t id_dv = idesc_bf16(128, 64, 0, 1);   // dV += P^T dO (dO MN-major)
            const uint32_t id_dk = idesc_bf16(128, 64, 0, 1);   // dK += dS^T Q (A K-major view, Q MN-major)
            const uint32_t id_dq = idesc_bf16(128, 64, 1, 1);   // dQ = dS K (A MN-major, K MN-major)
            uint32_t kv_full_bits = 0, st_full_bits = 0;
            uint32_t p_ready_ph = 0, dq_free_ph = 1, dkv_free_ph = 1;
            int kvbuf = 0, stage = 0, dsbuf = 0;
            bool ok = true;
            for (int round = 0; ok; ++round) {
                const int idx = item_index(round, cta, grid);
                if (idx >= p.n_items) break;
                const Item it = decode_item(p, idx);
                const int n = nqb - it.kb;
                const uint32_t skv = smem_u32(sm + Smem::kv + kvbuf * Smem::kv_bytes);
                if (!it.frozen) {
                    if (!(ok = mbar_wait(&bars.kv_full[kvbuf], (kv_full_bits >> kvbuf) & 1u, abort, status,
                                         kStatusTimeout)))
                        break;
                    kv_full_bits ^= 1u << kvbuf;
                }
                auto st_addr = [&](int s) { return smem_u32(sm + Smem::st + s * Smem::st_bytes); };
                auto wait_st = [&](int s) -> bool {
                    if (!mbar_wait(&bars.st_full[s], (st_full_bits >> s) & 1u, abort, status, kStatusTimeout))
                        return false;
                    st_full_bits ^= 1u << s;
                    tc_fence_after();
                    return true;
                };
                auto issue_s_dp = [&](int s) {
                    const uint32_t sq = st_addr(s), sdo = sq + kTileBytes;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss(tmem + kColS, sdesc_sw128(skv + 32 * k, 16, 1024), sdesc_sw128(sq + 32 * k, 16, 1024),
                               id_s, k > 0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss(tmem + kColDP, sdesc_sw128(skv + kTileBytes + 32 * k, 16, 1024),
                               sdesc_sw128(sdo + 32 * k, 16, 1024), id_s, k > 0);
                    mma_commit(&bars.s_full);
                };
                // The first dV / dK MMA of this item overwrites the accumulators: wait until
                // the epilogue group has read the previous item's dV and dK.
                if (!(ok = mbar_wait(&bars.dkv_free, dkv_free_ph, abort, status, kStatusTimeout))) break;
                dkv_free_ph ^= 1;
                tc_fence_after();
                if (!(ok = wait_st(stage))) break;
                if (!it.frozen) issue_s_dp(stage);
                for (int i = 0; i < n && ok; ++i) {
                    const int s = stage;
                    const int s_next = stage ^ 1;
                    if (!(ok = mbar_wait(&bars.p_ready, p_ready_ph, abort, status, kStatusTimeout))) break;
                    p_ready_ph ^= 1;
                    tc_fence_after();
                    if (i + 1 < n) {
                        if (!(ok = wait_st(s_next))) break;
                        if (!it.frozen) issue_s_dp(s_next);
                    }
                    const uint32_t sq = st_addr(s), sdo = sq + kTileBytes;
                    const uint32_t sds = smem_u32(sm + Smem::ds + dsbuf * Smem::ds_bytes);
                    // dV += P^T dO
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_ts(tmem + kColDV, tmem + kColP + 8 * k, sdesc_sw128(sdo + 2048 * k, 16384, 1024), id_dv,
                               (i > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&bars.p_free);
                    if (!it.frozen) {
                        // dK += dS^T Q: dS buffer viewed K-major (keys x queries, two 64-query halves)
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mma_ss(tmem + kColDK, sdesc_sw128(sds + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                                   sdesc_sw128(sq + 2048 * k, 16384, 1024), id_dk, (i > 0 || k > 0) ? 1u : 0u);
                        if (!(ok = mbar_wait(&bars.dq_free, dq_free_ph, abort, status, kStatusTimeout))) break;
                        dq_free_ph ^= 1;
                        tc_fence_after();
                        // dQ = dS K: dS buffer viewed MN-major (queries x keys)
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mma_ss(tmem + kColDQ, sdesc_sw128(sds + 2048 * k, 16384, 1024),
                                   sdesc_sw128(skv + 2048 * k, 16384, 1024), id_dq, k > 0);
                        mma_commit(&bars.dq_full);
                        mma_commit(&bars.ds_free[dsbuf]);
                    }
                    mma_commit(&bars.st_empty[s]);
                    stage = s_next;
                    dsbuf ^= 1;
                }
                if (!ok) break;
                mma_commit(&bars.dkv_full);
                if (!it.frozen) {
                    mma_commit(&bars.kv_empty[kvbuf]);
                    kvbuf ^= 1;
                }
            }
        }
    } else if (warp < 4) {
        // ---------------------------------------------------------------- pattern group
        const int j = threadIdx.x;   // key row within the block = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t s_full_ph = 0, st_full_bits = 0, p_free_ph = 1, ds_free_bits = 3u;
        int stage = 0, dsbuf = 0;
        bool ok = true;
        for (int round = 0; ok; ++round) {
            const int idx = item_index(round, cta, grid);
            if (idx >= p.n_items) break;
            const Item it = decode_item(p, idx);
            const int key = it.kb * 128 + j;
            float a2j = -INFINITY;
            if (it.frozen && key < p.T) a2j = p.a[(size_t)it.h * p.ld + key] * kLog2e;
            for (int qb = it.kb; qb < nqb && ok; ++qb) {
                const bool diag = qb == it.kb;
                // the row vectors of this tile (written by the producer lanes)
                if (!(ok = mbar_wait(&bars.st_full[stage], (st_full_bits >> stage) & 1u, abort, status,
                                     kStatusTimeout)))
                    break;
                st_full_bits ^= 1u << stage;
                const float* vec = reinterpret_cast<const float*>(sm + Smem::vec + stage * Smem::vec_floats * 4);
                if (!it.frozen) {
                    if (!(ok = mbar_wait(&bars.s_full, s_full_ph, abort, status, kStatusTimeout))) break;
                    s_full_ph ^= 1;
                    tc_fence_after();
                }
                // P^T may be overwritten once the previous tile's dV MMA has read it
                if (!(ok = mbar_wait(&bars.p_free, p_free_ph, abort, status, kStatusTimeout))) break;
                p_free_ph ^= 1;
                if (!it.frozen) {
                    if (!(ok = mbar_wait(&bars.ds_free[dsbuf], (ds_free_bits >> dsbuf) & 1u, abort, status,
                                         kStatusTimeout)))
                        break;
                    ds_free_bits ^= 1u << dsbuf;
                }
                tc_fence_after();
                uint8_t* dsp = sm + Smem::ds + dsbuf * Smem::ds_bytes;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
                    if (!it.frozen) {
                        uint32_t sv[32], dp[32];
                        tmem_ld32(lane_base + kColS + 32 * c, sv);
                        tmem_ld32(lane_base + kColDP + 32 * c, dp);
                        tmem_ld_wait();
                        uint32_t dk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const int q0 = 32 * c + e;
                            float p0 = fast_exp2(__uint_as_float(sv[e]) * kScaleLog2 - vec[q0]);
                            float p1 = fast_exp2(__uint_as_float(sv[e + 1]) * kScaleLog2 - vec[q0 + 1]);
                            if (diag && j > q0) p0 = 0.f;
                            if (diag && j > q0 + 1) p1 = 0.f;
                            const float d0 = p0 * (__uint_as_float(dp[e]) - vec[128 + q0]);
                            const float d1 = p1 * (__uint_as_float(dp[e + 1]) - vec[128 + q0 + 1]);
                            pk[e >> 1] = pack_bf16(p0, p1);
                            dk[e >> 1] = pack_bf16(d0, d1);
                        }
                        // dS row j, queries 32c..32c+31: MN-major tile, K-row j, 64-query half c/2
                        uint8_t* rowp = dsp + (c >> 1) * 16384;
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const uint32_t off = sw128_offset(j, ((c & 1) * 4 + t) * 16);
                            *reinterpret_cast<uint4*>(rowp + off) =
                                make_uint4(dk[4 * t], dk[4 * t + 1], dk[4 * t + 2], dk[4 * t + 3]);
                        }
                    } else {
                        // W^T(j, q) = W(q, j) = exp(a[j] + r[q - j] - log Z(q)) (Eq. 3)
                        const float* band = vec + 128 + 127 - j;   // band[q] = r2 at offset q - j
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const int q0 = 32 * c + e;
                            const float w0 = fast_exp2(a2j + band[q0] - vec[q0]);
                            const float w1 = fast_exp2(a2j + band[q0 + 1] - vec[q0 + 1]);
                            pk[e >> 1] = pack_bf16(w0, w1);
                        }
                    }
                    tmem_st16(lane_base + kColP + 16 * c, pk);
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars.p_ready);
                stage ^= 1;
                dsbuf ^= 1;
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue group
        const int t = threadIdx.x - 128;   // TMEM lane: query row (dQ) or key row (dV, dK)
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        uint32_t dq_full_ph = 0, dkv_full_ph = 0;
        bool ok = true;
        for (int round = 0; ok; ++round) {
            const int idx = item_index(round, cta, grid);
            if (idx >= p.n_items) break;
            const Item it = decode_item(p, idx);
            const int bh = it.b * p.H + it.h;
            if (!it.frozen) {
                for (int qb = it.kb; qb < nqb; ++qb) {
                    if (!(ok = mbar_wait(&bars.dq_full, dq_full_ph, abort, status, kStatusTimeout))) break;
                    dq_full_ph ^= 1;
                    tc_fence_after();
                    uint32_t v[64];
                    tmem_ld32(lane_base + kColDQ, v);
                    tmem_ld32(lane_base + kColDQ + 32, v + 32);
                    tmem_ld_wait();
                    tc_fence_before();
                    mbar_arrive(&bars.dq_free);
                    const int q = qb * 128 + t;
                    if (q < p.T) {
                        float* dst = p.dq_acc + ((size_t)bh * p.T + q) * 64;
#pragma unroll
                        for (int c = 0; c < 64; c += 4)
                            red_add_v4(dst + c, __uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                                       __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
                    }
                }
                if (!ok) break;
            }
            if (!(ok = mbar_wait(&bars.dkv_full, dkv_full_ph, abort, status, kStatusTimeout))) break;
            dkv_full_ph ^= 1;
            tc_fence_after();
            uint32_t dv[64], dk[64];
            tmem_ld32(lane_base + kColDV, dv);
            tmem_ld32(lane_base + kColDV + 32, dv + 32);
            if (!it.frozen) {
                tmem_ld32(lane_base + kColDK, dk);
                tmem_ld32(lane_base + kColDK + 32, dk + 32);
            }
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bars.dkv_free);
            const int key = it.kb * 128 + t;
            if (key < p.T) {
                uint4* pv = reinterpret_cast<uint4*>(p.dv + ((size_t)bh * p.T + key) * 64);
                uint4* pk = reinterpret_cast<uint4*>(p.dk + ((size_t)bh * p.T + key) * 64);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t* x = dv + 8 * c;
                    pv[c] = make_uint4(pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                       pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                       pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                       pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
                }
                if (it.frozen) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) pk[c] = make_uint4(0, 0, 0, 0);
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t* x = dk + 8 * c;
                        pk[c] = make_uint4(pack_bf16(__uint_as_float(x[0]) * kScale, __uint_as_float(x[1]) * kScale),
                                           pack_bf16(__uint_as_float(x[2]) * kScale, __uint_as_float(x[3]) * kScale),
                                           pack_bf16(__uint_as_float(x[4]) * kScale, __uint_as_float(x[5]) * kScale),
                                           pack_bf16(__uint_as_float(x[6]) * kScale, __uint_as_float(x[7]) * kScale));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// dq = dq_acc / sqrt(d) for ordinary heads, exact zeros for frozen heads.
__global__ void __launch_bounds__(256) dq_finish_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                        HeadMask mask, int H, long long rows_per_head_T) {
    // one thread per 8 elements
    const long long i8 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total8 = (long long)gridDim.y * rows_per_head_T * 8;
    (void)total8;
    const int bh = blockIdx.y;
    const long long per_bh8 = rows_per_head_T * 8;   // T rows x 64 elements / 8
    if (i8 >= per_bh8) return;
    const int h = bh % H;
    const size_t off = ((size_t)bh * per_bh8 + i8) * 8;
    uint4 out;
    if (head_frozen(mask, h)) {
        out = make_uint4(0, 0, 0, 0);
    } else {
        const float4 x0 = *reinterpret_cast<const float4*>(acc + off);
        const float4 x1 = *reinterpret_cast<const float4*>(acc + off + 4);
        out = make_uint4(pack_bf16(x0.x * kScale, x0.y * kScale), pack_bf16(x0.z * kScale, x0.w * kScale),
                         pack_bf16(x1.x * kScale, x1.y * kScale), pack_bf16(x1.z * kScale, x1.w * kScale));
    }
    *reinterpret_cast<uint4*>(dq + off) = out;
}

}  // namespace

cudaError_t launch_tc_bwd(const LayerArgs& a, cudaStream_t s) {
    BwdParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    const void* vbase = a.v;
    const void* qbase = a.q ? a.q : vbase;
    const void* kbase = a.k ? a.k : vbase;
    if (!make_tmap_bf16_3d(&p.tm_q, qbase, 64, a.T, BH, 64, 128) ||
        !make_tmap_bf16_3d(&p.tm_k, kbase, 64, a.T, BH, 64, 128) ||
        !make_tmap_bf16_3d(&p.tm_v, vbase, 64, a.T, BH, 64, 128) ||
        !make_tmap_bf16_3d(&p.tm_do, a.dO, 64, a.T, BH, 64, 128))
        return cudaErrorInvalidValue;
    p.dk = (__nv_bfloat16*)a.dk;
    p.dv = (__nv_bfloat16*)a.dv;
    p.dq_acc = a.dq_acc;
    p.lse = a.lse;
    p.delta = a.delta;
    p.a = a.a;
    p.r = a.r;
    p.lz = a.lz;
    p.status = a.status;
    p.B = a.B;
    p.H = a.H;
    p.T = a.T;
    p.ld = a.ld_prior;
    p.nqb = (a.T + 127) / 128;
    for (int h = 0; h < a.H; ++h) {
        if (head_frozen(a.mask, h))
            p.frz_heads[p.n_frz++] = (uint8_t)h;
        else
            p.ord_heads[p.n_ord++] = (uint8_t)h;
    }
    p.n_ord_items = a.B * p.n_ord * p.nqb;
    p.n_items = a.B * a.H * p.nqb;

    cudaError_t e;
    if (p.n_ord > 0) {
        e = cudaMemsetAsync(a.dq_acc, 0, (size_t)BH * a.T * 64 * sizeof(float), s);
        if (e != cudaSuccess) return e;
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = Smem::total + 1024;
    e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int grid = p.n_items < sms ? p.n_items : sms;
    before_launch(SAF_KERNEL_BWD, s);
    bwd_tc_kernel<<<grid, kThreads, smem, s>>>(p);
    after_launch(SAF_KERNEL_BWD, s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long per_bh8 = (long long)a.T * 8;
    dim3 g2((unsigned)((per_bh8 + 255) / 256), BH);
    before_launch(SAF_KERNEL_DQ_FINISH, s);
    dq_finish_kernel<<<g2, 256, 0, s>>>(a.dq_acc, (__nv_bfloat16*)a.dq, a.mask, a.H, a.T);
    after_launch(SAF_KERNEL_DQ_FINISH, s);
    return cudaGetLastError();
}

}  // namespace saf
