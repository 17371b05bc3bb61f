// Fused hybrid backward on the 5th-generation tensor cores (bf16, d = 64).
//
// "When Can Attention Heads Be Statically Defined?", App. D.2: key-block
// programs accumulate value gradients for every head and key gradients for
// ordinary heads. Here one persistent launch runs every key-block program of
// both kinds of head; the query gradients of ordinary heads are produced in
// the same programs (dQ = dS K per tile, added into an fp32 accumulator
// in the workspace) instead of by a separate query-block pass that would
// recompute S and dP. Frozen heads compute only dV = W^T dO (§3.3), with W
// rebuilt from a, r and log Z; their dK rows are written as zeros here and
// their dQ rows by the finishing kernel.
//
// Key and value heads may be shared (grouped-query layout, §3.3 and App. C.6:
// query head h reads key/value head h / G, G = H / Hkv; with G = 1 this is the
// multi-head layer). The gradient of a shared head is the sum over its group,
// so one work item covers a whole group: (batch b, key/value head hk, key
// block kb) = key rows [128 kb, 128 kb + 128); it loops over the group's query
// heads, ordinary ones first, and for each over query blocks qb = kb .. nqb-1
// (causal), accumulating dV (every head) and dK (ordinary heads) in tensor
// memory without atomics. Items are taken from a global counter, in this
// order: items of key/value heads that have an ordinary query head, in groups
// of kSliceGroup (batch, key/value head) slices, each group by ascending kb
// (longest first, and the group's dQ accumulator rows stay in L2), then the
// items whose query heads are all frozen, by ascending kb.
//
// Per (kb, qb) tile of an ordinary head (key row j of the block):
//   S^T  = K Q^T          (tcgen05, TMEM)      P^T = exp(S^T / sqrt(d) - lse)
//   dP^T = V dO^T         (tcgen05, TMEM)      dS  = P o (dP - D)
//   dV  += P^T dO         (A = P^T from TMEM)
//   dK  += dS^T Q         (A = dS in shared memory, K-major view)
//   dQ   = dS K           (A = dS in shared memory, MN-major view), then added
//                         into the fp32 accumulator by a bulk tensor reduce-add
//
// Warp roles (320 threads, one CTA per SM):
//   warps 0-7 : pattern warps; warp w handles key rows 32(w%4)..+31 and query
//               columns 64(w/4)..+63 of each tile (P^T, dS or W^T), then drains
//               dQ rows 32(w%4)..+31, d-columns 32(w/4)..+31 through shared
//               memory into the accumulator, and at the end of an item writes
//               its half of the dV, dK rows
//   warp 8    : producer: takes items from the counter and publishes them,
//               TMA of K, V per item and of Q, dO and the row vectors per tile
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
constexpr int kStages = 3;
constexpr int kRing = 4;
constexpr int kSliceGroup = 8;
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;
constexpr float kScale = 0.125f;

constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDV = 320, kColDK = 384, kColDQ = 448;

struct BwdParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tm_do;
    CUtensorMap tm_dq;     // fp32 dQ accumulator [BH, T, 64], box {32, 128}
    __nv_bfloat16* dk;     // [B, Hkv, T, 64]
    __nv_bfloat16* dv;     // [B, Hkv, T, 64]
    float* dq_acc;
    const float* rowvec;   // [BH, nqb, 256]: lse * log2(e) | D
    const float* a2p;      // [H, Tp]: a * log2(e)                (exact form)
    const float* r2p;      // [H, Tp + 256]: r * log2(e), + 127   (exact form)
    const float* eap;      // [H, Tp]: exp(a - max a)             (factorised form)
    const float* erp;      // [H, Tp + 256]: exp(r - max r), + 127
    const float* invz;     // [H, Tp]: 1 / Z'
    const uint32_t* hflag; // per head: bit 1 = use the exact form
    uint32_t* status;
    int B, H, Hkv, G, T, Tp;
    int nqb, n_items, n_act_items;
    int n_act, n_pas;                  // key/value heads with / without an ordinary query head
    uint8_t act_kv[SAF_MAX_HEADS];     // the former
    uint8_t pas_kv[SAF_MAX_HEADS];     // the latter
    uint8_t gheads[SAF_MAX_HEADS];     // query heads of key/value head hk at [hk G, hk G + G), ordinary first
    uint8_t gord[SAF_MAX_HEADS];       // ordinary query heads of key/value head hk
};

struct Smem {
    static constexpr int kv = 0;                      // K, V of the current item
    static constexpr int kv_bytes = 2 * kTileBytes;
    static constexpr int st = kv + kv_bytes;          // kStages x (Q, dO, row vectors)
    static constexpr int st_vec = 2 * kTileBytes;     // offset of the 512 fp32 row vectors in a stage
    static constexpr int st_bytes = 2 * kTileBytes + 3 * 1024;   // 1024-aligned
    // Two 32 KB buffers R[0], R[1]: ordinary tile t writes its dS (128 x 128 bf16) into
    // R[t & 1]; once the tile's MMAs are done the same buffer stages its dQ for the bulk
    // reduce (2 halves x 128 x 32 fp32), and tile t + 2's dS goes there after that reduce
    // has read it. So dS can be stored before the previous tile's MMAs have finished.
    static constexpr int ds = st + kStages * st_bytes;
    static constexpr int ds_bytes = 2 * kTileBytes;
    static constexpr int total = ds + 2 * ds_bytes;
};

struct Item {
    int b, hk, kb;
    int nord;   // ordinary query heads of the group (their tiles come first); 0: no K, V, dK
};

__device__ __forceinline__ Item decode_item(const BwdParams& p, int idx) {
    Item it;
    if (idx < p.n_act_items) {
        const int n_slices = p.B * p.n_act;
        const int per_group = kSliceGroup * p.nqb;
        const int g = idx / per_group;
        const int gsize = min(kSliceGroup, n_slices - g * kSliceGroup);
        const int within = idx - g * per_group;
        it.kb = within / gsize;
        const int slice = g * kSliceGroup + (within - it.kb * gsize);
        it.b = slice / p.n_act;
        it.hk = p.act_kv[slice - it.b * p.n_act];
    } else {
        const int f = idx - p.n_act_items;
        const int per = p.B * p.n_pas;
        it.kb = f / per;
        const int rem = f - it.kb * per;
        it.b = rem / p.n_pas;
        it.hk = p.pas_kv[rem - it.b * p.n_pas];
    }
    it.nord = p.gord[it.hk];
    return it;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

struct Barriers {
    uint64_t item_full[kRing], item_empty[kRing];
    uint64_t kv_full, kv_empty;
    uint64_t st_full[kStages], st_empty[kStages];
    uint64_t sdp_full;      // S^T and dP^T of the current tile are in TMEM (one commit after both)
    uint64_t s_consumed;    // pattern warps have read S^T (8 arrivals)
    uint64_t dp_consumed;   // pattern warps have read dP^T (8 arrivals)
    uint64_t p_ready;       // P^T in TMEM and dS in shared memory (8 warp arrivals)
    // (a tile's MMAs have all completed when the st_empty commit of its stage arrives: the
    // pattern warps wait on that barrier too)
    uint64_t dq_free;       // dQ of the previous tile has been read out (8 arrivals)
    uint64_t dkv_free;      // dV, dK of the previous item have been read out (8 arrivals)
    uint64_t mma_idle;      // every MMA this CTA issued has completed (commit before TMEM is freed)
};

// kGrouped = false compiles the multi-head layer (one query head per key/value
// head) with the group size fixed at 1, so that its loops keep their simple form.
template <bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1) bwd_tc_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (swizzled tiles), derived from the shared array itself so that
    // every access through it stays a shared-memory access
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ Barriers bars;
    __shared__ int item_ring[kRing];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    // the preparation kernels before this one on the stream have completed
    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bars.item_full[i], 1);
            mbar_init(&bars.item_empty[i], 9);   // MMA warp + 8 pattern warps
        }
        mbar_init(&bars.kv_full, 1);
        mbar_init(&bars.kv_empty, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars.st_full[i], 1);
            mbar_init(&bars.st_empty[i], 1);
        }
        mbar_init(&bars.sdp_full, 1);
        mbar_init(&bars.s_consumed, 8);
        mbar_init(&bars.dp_consumed, 8);
        mbar_init(&bars.p_ready, 8);
        mbar_init(&bars.dq_free, 8);
        mbar_init(&bars.dkv_free, 8);
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
    const int nqb = p.nqb;
    const int G = kGrouped ? p.G : 1;   // query heads per key/value head

    if (warp == 8) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_do);
            uint32_t ring_empty_bits = (1u << kRing) - 1, kv_empty_ph = 1;
            uint32_t st_empty_bits = (1u << kStages) - 1;
            int slot = 0, stage = 0;
            bool ok = true;
            while (ok) {
                if (!(ok = mbar_wait(&bars.item_empty[slot], (ring_empty_bits >> slot) & 1u, abort, status,
                                     kStatusTimeout)))
                    break;
                ring_empty_bits ^= 1u << slot;
                int idx = (int)atomicAdd(status + kCounterBwd, 1u);
                if (idx >= p.n_items) idx = -1;
                item_ring[slot] = idx;
                mbar_arrive(&bars.item_full[slot]);
                slot = (slot + 1) % kRing;
                if (idx < 0) break;
                const Item it = decode_item(p, idx);
                if (it.nord > 0) {
                    if (!(ok = mbar_wait(&bars.kv_empty, kv_empty_ph, abort, status, kStatusTimeout))) break;
                    kv_empty_ph ^= 1;
                    uint8_t* kv = sm + Smem::kv;
                    const int bkv = it.b * p.Hkv + it.hk;
                    mbar_expect_tx(&bars.kv_full, 2 * kTileBytes);
                    tma_load_3d(kv, &p.tm_k, &bars.kv_full, 0, it.kb * 128, bkv);
                    tma_load_3d(kv + kTileBytes, &p.tm_v, &bars.kv_full, 0, it.kb * 128, bkv);
                }
                // the group's query heads, ordinary first, each over query blocks kb .. nqb-1
                for (int gi = 0; gi < G && ok; ++gi) {
                    const int h = p.gheads[it.hk * G + gi];
                    const int bh = it.b * p.H + h;
                    const bool frz = gi >= it.nord;
                    const bool exact = frz && (p.hflag[h] & 2u) != 0;
                    for (int qb = it.kb; qb < nqb; ++qb) {
                        if (!(ok = mbar_wait(&bars.st_empty[stage], (st_empty_bits >> stage) & 1u, abort, status,
                                             kStatusTimeout)))
                            break;
                        st_empty_bits ^= 1u << stage;
                        uint8_t* st = sm + Smem::st + stage * Smem::st_bytes;
                        float* vec = reinterpret_cast<float*>(st + Smem::st_vec);
                        const float* rv = p.rowvec + ((size_t)bh * nqb + qb) * 256;
                        if (!frz) {
                            mbar_expect_tx(&bars.st_full[stage], 2 * kTileBytes + 1024);
                            tma_load_3d(st, &p.tm_q, &bars.st_full[stage], 0, qb * 128, bh);
                            tma_load_3d(st + kTileBytes, &p.tm_do, &bars.st_full[stage], 0, qb * 128, bh);
                            bulk_load(vec, rv, 1024, &bars.st_full[stage]);
                        } else {
                            // exact form: vec[0..128) lse * log2(e) (= log2 Z), vec[256..512) r * log2(e);
                            // factorised form: vec[0..128) 1 / Z', vec[256..512) exp(r - R)
                            const float* band = (exact ? p.r2p : p.erp) + (size_t)h * (p.Tp + 256) +
                                                (size_t)(qb - it.kb) * 128;
                            mbar_expect_tx(&bars.st_full[stage], kTileBytes + 1024 + 512);
                            tma_load_3d(st + kTileBytes, &p.tm_do, &bars.st_full[stage], 0, qb * 128, bh);
                            if (exact)
                                bulk_load(vec, rv, 512, &bars.st_full[stage]);
                            else
                                bulk_load(vec, p.invz + (size_t)h * p.Tp + (size_t)qb * 128, 512,
                                          &bars.st_full[stage]);
                            bulk_load(vec + 256, band, 1024, &bars.st_full[stage]);
                        }
                        stage = (stage + 1) % kStages;
                    }
                }
            }
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S^T = K Q^T, dP^T = V dO^T
            const uint32_t id_dv = idesc_bf16(128, 64, 0, 1);   // dV += P^T dO (dO MN-major)
            const uint32_t id_dk = idesc_bf16(128, 64, 0, 1);   // dK += dS^T Q (A K-major view, Q MN-major)
            const uint32_t id_dq = idesc_bf16(128, 64, 1, 1);   // dQ = dS K (A MN-major, K MN-major)
            uint32_t ring_full_bits = 0, kv_full_ph = 0, st_full_bits = 0;
            uint32_t s_consumed_ph = 0, dp_consumed_ph = 0, p_ready_ph = 0, dq_free_ph = 1, dkv_free_ph = 1;
            int slot = 0, stage = 0;
            bool ok = true;
            int gto = 0;   // ordinary tiles so far: dS buffer gto & 1
            const uint32_t skv = smem_u32(sm + Smem::kv);
            // descriptors of the fixed operands; per-stage ones are formed once per tile and
            // every K step advances a descriptor by a constant
            const uint64_t d_k = sdesc_sw128(skv, 16, 1024);                  // K, K-major (S^T)
            const uint64_t d_v = sdesc_sw128(skv + kTileBytes, 16, 1024);     // V, K-major (dP^T)
            const uint64_t d_kmn = sdesc_sw128(skv, 16384, 1024);             // K, MN-major (dQ)

            auto st_addr = [&](int s) { return smem_u32(sm + Smem::st + s * Smem::st_bytes); };
            auto wait_st = [&](int s) -> bool {
                if (!mbar_wait(&bars.st_full[s], (st_full_bits >> s) & 1u, abort, status, kStatusTimeout))
                    return false;
                st_full_bits ^= 1u << s;
                tc_fence_after();
                return true;
            };
            auto issue_s = [&](int s) {   // S^T = K Q^T
                const uint64_t d_q = sdesc_sw128(st_addr(s), 16, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss(tmem + kColS, sdesc_advance(d_k, 32 * k), sdesc_advance(d_q, 32 * k), id_s, k > 0);
            };
            auto issue_dp = [&](int s) {  // dP^T = V dO^T
                const uint64_t d_do = sdesc_sw128(st_addr(s) + kTileBytes, 16, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss(tmem + kColDP, sdesc_advance(d_v, 32 * k), sdesc_advance(d_do, 32 * k), id_s, k > 0);
                mma_commit(&bars.sdp_full);   // S^T (issued just before) and dP^T
            };
            while (ok) {
                if (!(ok = mbar_wait(&bars.item_full[slot], (ring_full_bits >> slot) & 1u, abort, status,
                                     kStatusTimeout)))
                    break;
                ring_full_bits ^= 1u << slot;
                const int idx = item_ring[slot];
                mbar_arrive(&bars.item_empty[slot]);
                slot = (slot + 1) % kRing;
                if (idx < 0) break;
                const Item it = decode_item(p, idx);
                const int n = G * (nqb - it.kb);        // tiles of the item
                const int n_ord = it.nord * (nqb - it.kb);   // its ordinary tiles come first
                if (n_ord > 0) {
                    if (!(ok = mbar_wait(&bars.kv_full, kv_full_ph, abort, status, kStatusTimeout))) break;
                    kv_full_ph ^= 1;
                    if (!(ok = wait_st(stage))) break;
                    issue_s(stage);
                    issue_dp(stage);
                }
                for (int i = 0; i < n && ok; ++i) {
                    const int s = stage;
                    const int s_next = (stage + 1) % kStages;
                    const bool ord = i < n_ord;
                    if (ord) {
                        // S^T and dP^T of the next tile may overwrite TMEM once this tile's are read
                        if (!(ok = mbar_wait(&bars.s_consumed, s_consumed_ph, abort, status, kStatusTimeout))) break;
                        s_consumed_ph ^= 1;
                        tc_fence_after();
                        if (i + 1 < n_ord) {
                            if (!(ok = wait_st(s_next))) break;
                            issue_s(s_next);
                        }
                        if (!(ok = mbar_wait(&bars.dp_consumed, dp_consumed_ph, abort, status, kStatusTimeout))) break;
                        dp_consumed_ph ^= 1;
                        tc_fence_after();
                        if (i + 1 < n_ord) issue_dp(s_next);
                    } else {
                        if (!(ok = wait_st(s))) break;
                    }
                    if (!(ok = mbar_wait(&bars.p_ready, p_ready_ph, abort, status, kStatusTimeout))) break;
                    p_ready_ph ^= 1;
                    if (i == 0) {
                        // the first dV / dK MMA of this item overwrites the accumulators:
                        // the previous item's dV and dK must have been read out
                        if (!(ok = mbar_wait(&bars.dkv_free, dkv_free_ph, abort, status, kStatusTimeout))) break;
                        dkv_free_ph ^= 1;
                    }
                    tc_fence_after();
                    const uint32_t sq = st_addr(s);
                    const uint64_t d_qmn = sdesc_sw128(sq, 16384, 1024);                // Q, MN-major (dK)
                    const uint64_t d_domn = sdesc_sw128(sq + kTileBytes, 16384, 1024);  // dO, MN-major (dV)
                    // dV += P^T dO
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_ts(tmem + kColDV, tmem + kColP + 8 * k, sdesc_advance(d_domn, 2048 * k), id_dv,
                               (i > 0 || k > 0) ? 1u : 0u);
                    if (ord) {
                        const uint32_t sds = smem_u32(sm + Smem::ds + (gto++ & 1) * Smem::ds_bytes);
                        const uint64_t d_ds = sdesc_sw128(sds, 16, 1024);       // dS, K-major view (dK)
                        const uint64_t d_dsmn = sdesc_sw128(sds, 16384, 1024);  // dS, MN-major view (dQ)
                        // dK += dS^T Q: dS viewed K-major (keys x queries, two 64-query halves)
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mma_ss(tmem + kColDK, sdesc_advance(d_ds, (k >> 2) * 16384 + (k & 3) * 32),
                                   sdesc_advance(d_qmn, 2048 * k), id_dk, (i > 0 || k > 0) ? 1u : 0u);
                        // dQ may be overwritten once the previous tile's dQ has been read out
                        if (!(ok = mbar_wait(&bars.dq_free, dq_free_ph, abort, status, kStatusTimeout))) break;
                        dq_free_ph ^= 1;
                        tc_fence_after();
                        // dQ = dS K: dS viewed MN-major (queries x keys)
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mma_ss(tmem + kColDQ, sdesc_advance(d_dsmn, 2048 * k), sdesc_advance(d_kmn, 2048 * k), id_dq,
                                   k > 0);
                    }
                    mma_commit(&bars.st_empty[s]);
                    stage = s_next;
                }
                if (!ok) break;
                if (n_ord > 0) mma_commit(&bars.kv_empty);
            }
            // Tensor memory is freed below: every MMA issued here must have completed (on
            // the normal path the pattern warps have already seen it; after an abort the
            // last MMAs may still run), with a bounded wait of its own.
            mma_commit(&bars.mma_idle);
            mbar_wait_bounded(&bars.mma_idle, 0, kWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------------- pattern warps
        const int quarter = warp & 3, half = warp >> 2;
        const int j = quarter * 32 + lane;                   // key row of the block = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t ring_full_bits = 0, st_full_bits = 0;
        uint32_t sdp_full_ph = 0;
        uint32_t done_bits = 0;   // per stage: parity of the st_empty phase that ends its next tile
        int pending = -1;         // stage of the last tile handed over whose MMAs were not waited for
        int slot = 0, stage = 0;
        bool ok = true;
        int gto = 0;   // ordinary tiles so far: dS buffer gto & 1
        // my half of buffer b: 64 queries of dS (MN-major atom), or 32 columns of dQ staging
        auto dsbuf = [&](int b) { return sm + Smem::ds + b * Smem::ds_bytes + half * 16384; };
        const bool dq_issuer = quarter == 0 && lane == 0;     // issues the bulk reduce of this half

        // The previous tile's MMAs have all completed: P^T, dS may be overwritten
        // and its dQ (ordinary tiles) can be read out.
        auto wait_tile_done = [&]() -> bool {
            if (pending < 0) return true;
            if (!mbar_wait(&bars.st_empty[pending], (done_bits >> pending) & 1u, abort, status, kStatusTimeout))
                return false;
            done_bits ^= 1u << pending;
            pending = -1;
            tc_fence_after();
            return true;
        };
        // Drain dQ of tile (bh, qb) into the fp32 accumulator with a bulk tensor
        // reduce-add: rows 32*quarter + lane, d-columns 32*half .. +31.
        auto drain_dq = [&](int bh, int qb, uint8_t* dqs) {
            uint32_t v[32];
            tmem_ld32(lane_base + kColDQ + 32 * half, v);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.dq_free);
            if (dq_issuer) bulk_wait_read_all();   // the previous reduce has read the staging buffer
            named_bar_sync(1 + half, 128);
#pragma unroll
            for (int t = 0; t < 8; ++t)
                *reinterpret_cast<uint4*>(dqs + sw128_offset(j, 16 * t)) =
                    make_uint4(v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
            fence_proxy_async_smem();
            named_bar_sync(1 + half, 128);
            if (dq_issuer) {
                tma_reduce_add_3d(&p.tm_dq, dqs, 32 * half, qb * 128, bh);
                bulk_commit_group();
            }
        };

        while (ok) {
            if (!(ok = mbar_wait(&bars.item_full[slot], (ring_full_bits >> slot) & 1u, abort, status,
                                 kStatusTimeout)))
                break;
            ring_full_bits ^= 1u << slot;
            const int idx = item_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.item_empty[slot]);
            slot = (slot + 1) % kRing;
            if (idx < 0) break;
            const Item it = decode_item(p, idx);
            const int bkv = it.b * p.Hkv + it.hk;   // the key/value slice whose dK, dV this item writes
            const int key = it.kb * 128 + j;
            const int n = G * (nqb - it.kb);
            // tile i: query head gheads[hk G + gi] (ordinary for gi < nord), query block qb
            int gi = 0, qb = it.kb;
            const int n_ord = it.nord * (nqb - it.kb);   // the ordinary tiles come first
            // In the multi-head layer a frozen item's tiles all belong to one head: the factor
            // exp(a[j] - A) of its key rows stays out of W^T and is applied to dV at the end.
            // A group of query heads puts it into each W^T tile instead.
            const bool ea_at_end = !kGrouped && it.nord == 0;
            // exact-form flag of the current query head (read when the head changes)
            bool exact = it.nord == 0 && (p.hflag[p.gheads[it.hk * G]] & 2u) != 0;
            // the multi-head layer has one query head per item: its slice and kind are fixed
            const int h_item = p.gheads[it.hk * G];
            for (int i = 0; i < n && ok; ++i) {
                if (!kGrouped) qb = it.kb + i;
                const bool diag = qb == it.kb;
                const int h = kGrouped ? p.gheads[it.hk * G + gi] : h_item;
                const int bh = it.b * p.H + h;
                const bool frz = kGrouped ? gi >= it.nord : it.nord == 0;
                if (!(ok = mbar_wait(&bars.st_full[stage], (st_full_bits >> stage) & 1u, abort, status,
                                     kStatusTimeout)))
                    break;
                st_full_bits ^= 1u << stage;
                const float* vec =
                    reinterpret_cast<const float*>(sm + Smem::st + stage * Smem::st_bytes + Smem::st_vec);
                if (!frz) {
                    if (!(ok = mbar_wait(&bars.sdp_full, sdp_full_ph, abort, status, kStatusTimeout))) break;
                    sdp_full_ph ^= 1;
                    tc_fence_after();
                    // P^T first: S^T row (64 columns) -> P (bf16 pairs); then dP^T row -> dS.
                    uint32_t pk[32];
                    {
                        uint32_t sv[64];
                        tmem_ld32(lane_base + kColS + 64 * half, sv);
                        tmem_ld32(lane_base + kColS + 64 * half + 32, sv + 32);
                        tmem_ld_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars.s_consumed);   // S^T of the next tile may land
                        // lse * log2(e) of four query columns per (broadcast) shared-memory load
                        const float4* lse4 = reinterpret_cast<const float4*>(vec + 64 * half);
#pragma unroll
                        for (int e = 0; e < 64; e += 4) {
                            const float4 l4 = lse4[e >> 2];
#pragma unroll
                            for (int u = 0; u < 4; u += 2) {
                                const int q0 = 64 * half + e + u;
                                // x = S * log2(e) / sqrt(d) - lse * log2(e), two columns per instruction
                                const float2 x = ffma2(
                                    make_float2(__uint_as_float(sv[e + u]), __uint_as_float(sv[e + u + 1])),
                                    make_float2(kScaleLog2, kScaleLog2),
                                    u == 0 ? make_float2(-l4.x, -l4.y) : make_float2(-l4.z, -l4.w));
                                float p0 = fast_exp2(x.x);
                                float p1 = fast_exp2(x.y);
                                if (diag && j > q0) p0 = 0.f;
                                if (diag && j > q0 + 1) p1 = 0.f;
                                pk[(e + u) >> 1] = pack_bf16(p0, p1);
                            }
                        }
                    }
                    uint32_t dp[64];
                    tmem_ld32(lane_base + kColDP + 64 * half, dp);
                    tmem_ld32(lane_base + kColDP + 64 * half + 32, dp + 32);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.dp_consumed);   // dP^T of the next tile may land
                    // dS goes to buffer gto & 1 while the previous tile's MMAs may still run: that
                    // buffer last staged the dQ of tile gto - 2, whose reduce must have read it
                    uint8_t* dsp = dsbuf(gto & 1);
                    if (dq_issuer) bulk_wait_read_all();
                    named_bar_sync(1 + half, 128);
                    const float4* dvec4 = reinterpret_cast<const float4*>(vec + 128 + 64 * half);
#pragma unroll
                    for (int g2 = 0; g2 < 2; ++g2) {
                        uint32_t dk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const float4 d4 = dvec4[(32 * g2 + e) >> 2];   // D of four query columns
#pragma unroll
                            for (int u = 0; u < 4; u += 2) {
                                const int c = 32 * g2 + e + u;
                                // dS = P o (dP - D) with P as rounded to bf16 for the MMAs
                                const float2 pp = make_float2(__uint_as_float(pk[c >> 1] << 16),
                                                              __uint_as_float(pk[c >> 1] & 0xffff0000u));
                                const float2 dd = fmul2(
                                    pp, fsub2(make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])),
                                              u == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w)));
                                dk[(e + u) >> 1] = pack_bf16(dd.x, dd.y);
                            }
                        }
                        // dS row j, queries 64*half + 32*g2 .. +31: MN-major atom `half`, K-row j
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            *reinterpret_cast<uint4*>(dsp + sw128_offset(j, 16 * (4 * g2 + t))) =
                                make_uint4(dk[4 * t], dk[4 * t + 1], dk[4 * t + 2], dk[4 * t + 3]);
                    }
                    // the previous tile's MMAs are done: P^T of this tile overwrites the previous one
                    if (!(ok = wait_tile_done())) break;
                    tmem_st32(lane_base + kColP + 32 * half, pk);
                    ++gto;
                } else {
                    // W^T(j, q) = W(q, j) (Eq. 3); band[q] is r at offset q - j = (qb - kb) * 128 +
                    // q - j. Factorised: W(q, j) = exp(a[j] - A) exp(r[q-j] - R) / Z'(q), no exp per
                    // element (exp(a[j] - A) in the tile, or on dV at the end: ea_at_end). Exact:
                    // exp(a[j] + r[q-j] - log Z(q)).
                    uint32_t pk[32];
                    if (!exact) {
                        // W^T is Toeplitz up to the row factor exp(a[j] - A) and the column
                        // factor 1 / Z'(q). In the 16x128b shape a thread holds key rows
                        // 32 quarter + rho + 8 m (m = 0..3) at packed columns 4 jr + qq, queries
                        // q = 64 half + 8 jr + 2 qq + {0, 1} (jr = 0..7): the band value of
                        // (row, q) depends on jr - m alone, so 22 band loads serve the thread's
                        // 64 products.
                        const int rho = lane >> 2, qq = lane & 3;
                        const float* b1 = vec + 256 + 127 + 64 * half + 2 * qq - 32 * quarter - rho;
                        // exp(a - A) of my four key rows (1 when it is applied to dV at the end)
                        float ea4[4] = {1.f, 1.f, 1.f, 1.f};
                        if (kGrouped) {
                            const float* ea = p.eap + (size_t)h * p.Tp + it.kb * 128 + 32 * quarter + rho;
#pragma unroll
                            for (int m = 0; m < 4; ++m) ea4[m] = ea[8 * m];
                        }
                        float e0[11], e1[11];   // index jr - m + 3
#pragma unroll
                        for (int d = -3; d <= 7; ++d) {
                            e0[d + 3] = b1[8 * d];
                            e1[d + 3] = b1[8 * d + 1];
                        }
#pragma unroll
                        for (int jr = 0; jr < 8; ++jr) {
                            const float2 iz = *reinterpret_cast<const float2*>(vec + 64 * half + 8 * jr + 2 * qq);
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const float2 izm = kGrouped ? fmul2(iz, make_float2(ea4[m], ea4[m])) : iz;
                                const float2 w = fmul2(make_float2(e0[jr - m + 3], e1[jr - m + 3]), izm);
                                pk[16 * (m >> 1) + 2 * jr + (m & 1)] = pack_bf16(w.x, w.y);
                            }
                        }
                    } else {
                        const float a2j = p.a2p[(size_t)h * p.Tp + key];   // a * log2(e) of my key
                        const float* band = vec + 256 + 127 - j;
#pragma unroll
                        for (int e = 0; e < 64; e += 2) {
                            const int q0 = 64 * half + e;
                            const float w0 = fast_exp2(a2j + band[q0] - vec[q0]);
                            const float w1 = fast_exp2(a2j + band[q0 + 1] - vec[q0 + 1]);
                            pk[e >> 1] = pack_bf16(w0, w1);
                        }
                    }
                    if (!(ok = wait_tile_done())) break;
                    if (!exact) {
                        tmem_st_16x128b_x8(lane_base + kColP + 32 * half, pk);
                        tmem_st_16x128b_x8(lane_base + (16u << 16) + kColP + 32 * half, pk + 16);
                    } else {
                        tmem_st32(lane_base + kColP + 32 * half, pk);
                    }
                }
                // every thread's P^T stores are complete and its dS stores visible to the
                // tensor cores; the warp then hands the tile over with one arrival
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p_ready);
                // dQ of the previous tile if it was ordinary (its MMAs are done), staged in the
                // buffer that held its dS (gto has counted this tile if it is ordinary)
                if (!kGrouped) {
                    if (!frz && i > 0) drain_dq(bh, qb - 1, dsbuf(gto & 1));
                } else if (i > 0 && i - 1 < n_ord) {
                    const bool first = qb == it.kb;
                    const int bhp = it.b * p.H + p.gheads[it.hk * G + (first ? gi - 1 : gi)];
                    drain_dq(bhp, first ? nqb - 1 : qb - 1, dsbuf((frz ? gto - 1 : gto) & 1));
                }
                pending = stage;
                stage = (stage + 1) % kStages;
                if (kGrouped && ++qb == nqb) {   // next query head of the group
                    qb = it.kb;
                    if (++gi >= it.nord && gi < G) exact = (p.hflag[p.gheads[it.hk * G + gi]] & 2u) != 0;
                }
            }
            if (!ok) break;
            // all MMAs of this item done: the last dQ, then the dV and dK rows (my 32 d-columns)
            if (!(ok = wait_tile_done())) break;
            if (n > 0 && n - 1 < n_ord)   // the last tile was ordinary
                drain_dq(it.b * p.H + p.gheads[it.hk * G + G - 1], nqb - 1, dsbuf((gto - 1) & 1));
            uint32_t dv[32], dk[32];
            tmem_ld32(lane_base + kColDV + 32 * half, dv);
            if (it.nord > 0) tmem_ld32(lane_base + kColDK + 32 * half, dk);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.dkv_free);
            {
                // exp(a[j] - A) of my key, when the item left it out of W^T (factorised form)
                float fv = 1.f;
                if (ea_at_end && !exact) fv = p.eap[(size_t)p.gheads[it.hk * G] * p.Tp + key];
                const size_t off = ((size_t)bkv * p.T + it.kb * 128 + 32 * quarter) * 64 + 32 * half;
                const int nrows = p.T - it.kb * 128 - 32 * quarter;
                uint4 x[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t* v = dv + 8 * c;
                    x[c] = make_uint4(pack_bf16(__uint_as_float(v[0]) * fv, __uint_as_float(v[1]) * fv),
                                      pack_bf16(__uint_as_float(v[2]) * fv, __uint_as_float(v[3]) * fv),
                                      pack_bf16(__uint_as_float(v[4]) * fv, __uint_as_float(v[5]) * fv),
                                      pack_bf16(__uint_as_float(v[6]) * fv, __uint_as_float(v[7]) * fv));
                }
                store_rows64(reinterpret_cast<uint8_t*>(p.dv + off), 128, nrows, x);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t* v = dk + 8 * c;
                    x[c] = it.nord == 0 ? make_uint4(0, 0, 0, 0)
                                        : make_uint4(pack_bf16(__uint_as_float(v[0]) * kScale, __uint_as_float(v[1]) * kScale),
                                                     pack_bf16(__uint_as_float(v[2]) * kScale, __uint_as_float(v[3]) * kScale),
                                                     pack_bf16(__uint_as_float(v[4]) * kScale, __uint_as_float(v[5]) * kScale),
                                                     pack_bf16(__uint_as_float(v[6]) * kScale, __uint_as_float(v[7]) * kScale));
                }
                store_rows64(reinterpret_cast<uint8_t*>(p.dk + off), 128, nrows, x);
            }
        }
    }

    if (warp < 8 && (warp & 3) == 0 && lane == 0) bulk_wait_all();   // dQ reduces complete
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// dq = dq_acc / sqrt(d) for ordinary heads, exact zeros for frozen heads.
// Grid (ceil(T * 8 / 256), B*H); one thread per 8 elements of a slice.
__global__ void __launch_bounds__(256) dq_finish_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                        HeadMask mask, int H, int T) {
    grid_dep_wait();   // the backward kernel has completed
    grid_dep_launch();
    const long long per_bh8 = (long long)T * 8;
    const long long i8 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i8 >= per_bh8) return;
    const int bh = blockIdx.y;
    const size_t off = ((size_t)bh * per_bh8 + i8) * 8;
    uint4 out;
    if (head_frozen(mask, bh % H)) {
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
    const int Hkv = a.Hkv > 0 ? a.Hkv : a.H;
    const int BHkv = a.B * Hkv;
    const void* vbase = a.v;
    const void* kbase = a.k ? a.k : vbase;
    // q (and k) may be NULL when every head is frozen; the maps then point at v and are never used
    const void* qbase = a.q ? a.q : vbase;
    const int BHq = a.q ? BH : BHkv;
    if (!make_tmap_bf16_3d(&p.tm_q, qbase, 64, a.T, BHq, 64, 128) ||
        !make_tmap_bf16_3d(&p.tm_k, kbase, 64, a.T, BHkv, 64, 128) ||
        !make_tmap_bf16_3d(&p.tm_v, vbase, 64, a.T, BHkv, 64, 128) ||
        !make_tmap_bf16_3d(&p.tm_do, a.dO, 64, a.T, BH, 64, 128) ||
        !make_tmap_f32_3d(&p.tm_dq, a.dq_acc, 64, a.T, BH, 32, 128))
        return cudaErrorInvalidValue;
    p.dk = (__nv_bfloat16*)a.dk;
    p.dv = (__nv_bfloat16*)a.dv;
    p.dq_acc = a.dq_acc;
    p.rowvec = a.rowvec;
    p.a2p = a.a2p;
    p.r2p = a.r2p;
    p.eap = a.eap;
    p.erp = a.erp;
    p.invz = a.invz;
    p.hflag = a.hflag;
    p.status = a.status;
    p.B = a.B;
    p.H = a.H;
    p.Hkv = Hkv;
    p.G = a.H / Hkv;
    p.T = a.T;
    p.nqb = (a.T + 127) / 128;
    p.Tp = p.nqb * 128;
    // per key/value head: its query heads, ordinary first
    for (int hk = 0; hk < Hkv; ++hk) {
        int n = 0;
        for (int pass = 0; pass < 2; ++pass)
            for (int gi = 0; gi < p.G; ++gi) {
                const int h = hk * p.G + gi;
                if (head_frozen(a.mask, h) == (pass == 1)) p.gheads[hk * p.G + n++] = (uint8_t)h;
            }
        int nord = 0;
        for (int gi = 0; gi < p.G; ++gi) nord += head_frozen(a.mask, hk * p.G + gi) ? 0 : 1;
        p.gord[hk] = (uint8_t)nord;
        if (nord > 0)
            p.act_kv[p.n_act++] = (uint8_t)hk;
        else
            p.pas_kv[p.n_pas++] = (uint8_t)hk;
    }
    p.n_act_items = a.B * p.n_act * p.nqb;
    p.n_items = BHkv * p.nqb;

    // (the dQ accumulator of the ordinary heads was zeroed by bwd_prep_kernel)
    cudaError_t e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = Smem::total + 1024;
    void (*kernel)(BwdParams) = p.G > 1 ? bwd_tc_kernel<true> : bwd_tc_kernel<false>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int grid = p.n_items < sms ? p.n_items : sms;
    before_launch(SAF_KERNEL_BWD, s);
    e = launch_ex(kernel, dim3(grid), dim3(kThreads), smem, s, true, 1, p);
    after_launch(SAF_KERNEL_BWD, s);
    if (e != cudaSuccess) return e;
    dim3 g2((unsigned)(((long long)a.T * 8 + 255) / 256), BH);
    before_launch(SAF_KERNEL_DQ_FINISH, s);
    e = launch_ex(dq_finish_kernel, g2, dim3(256), 0, s, true, 1, (const float*)a.dq_acc, (__nv_bfloat16*)a.dq,
                  a.mask, a.H, a.T);
    after_launch(SAF_KERNEL_DQ_FINISH, s);
    return e;
}

}  // namespace saf
