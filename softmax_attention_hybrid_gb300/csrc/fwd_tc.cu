// Fused hybrid forward on the 5th-generation tensor cores (bf16, d = 64).
//
// "When Can Attention Heads Be Statically Defined?": ordinary heads run
// online-softmax attention with FlashAttention-2 tiling (App. A.1 Eqs. 5-7,
// §3.3); frozen heads rebuild causal tiles of the fixed pattern P-hat of
// Eq. 3 in registers from a, r and the precomputed normalisers and multiply
// them with value tiles (§3.3 "Fused computation", App. D.2). One persistent
// launch runs both kinds of head; a per-item head-state flag picks the path
// and outputs keep their head order.
//
// Work item: (batch b, head h, query-block pair p) = query rows
// [256p, 256p + 256) as two 128-row tiles that share every K/V tile load.
// Items are numbered in groups of (batch, head) slices (ordinary slices before
// frozen ones), longest first inside a group, so that a group's key and value
// tiles stay in L2 while its query pairs re-read them; the producer of each
// persistent CTA takes the next number from a global counter when its CTA is
// ready for more work and publishes it to the CTA's other warps through a small
// ring in shared memory.
//
// Warp roles (384 threads, one CTA per SM; warp 11 idles):
//   warps 0-3 / 4-7 : softmax group g = 0 / 1, thread = one query row of tile g
//   warp 8          : TMA producer (Q tiles, K/V stages)
//   warps 9 / 10    : MMA issuers of tile 0 / 1 (the whole warp runs the issue
//                     loop, one elected lane issues; two issuers keep the
//                     tensor core fed at N = 64); warp 9 owns tensor memory
// Tensor memory (512 columns), per tile g at column 256g:
//   [0, 128)   S = Q K^T (fp32); frozen items: W of odd key blocks (bf16 pairs)
//   [128, 192) P, or W of even key blocks (bf16 pairs), the A operand of P V
//   [192, 256) O accumulator (fp32)
// Frozen items have no S, so their W alternates between the two buffers and
// the next block's W is built while the current P V runs.
// Shared memory: two Q slots of 2 tiles (16 KB each; alternate ordinary items, so
// the next item's Q loads while this one runs) and kStages K/V stages (32 KB each); for
// frozen items the K slot of a stage holds the key block's slice of a and the
// band of r that the tiles' diagonals need.
#include <string.h>

#include "saf_internal.h"
#include "tc_common.cuh"

namespace saf {
namespace {

using namespace tc;

constexpr int kStages = 3;   // 4 and 5 measured slower (likely: a larger shared-memory carve-out leaves less L1)
constexpr int kRing = 4;   // work items published ahead by the producer
// Items run in groups of slices whose key/value tiles stay in L2 together
// (launch_tc_fwd picks the group size: all slices when their K and V fit in
// kL2GroupBytes, else kSliceGroup slices).
constexpr int kSliceGroup = 8;
constexpr size_t kL2GroupBytes = 64ull << 20;
constexpr int kTileBytes = 128 * 64 * 2;  // one 128 x 64 bf16 tile
constexpr int kThreads = 384;   // 3 warpgroups: 2 softmax, 1 producer / issuers / idle
// Register split (setmaxnreg): warpgroup 2 drops to kRegsOther registers per thread and
// the softmax warpgroups rise to kRegsSoftmax. The launch gives every thread
// kRegsLaunch (checked on the host); the split must not exceed that total:
// 2 x 128 x kRegsSoftmax + 128 x kRegsOther <= 384 x kRegsLaunch.
constexpr int kRegsLaunch = 168, kRegsSoftmax = 216, kRegsOther = 72;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= kThreads * kRegsLaunch, "register split too large");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;  // log2(e) / sqrt(64)
constexpr float kRescaleThreshold = 8.0f;                    // lazy rescale: factor 256

struct FwdParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    __nv_bfloat16* o;
    float* lse;
    const float* lz;
    const float* a2p;     // [H, Tp]: a * log2(e), -inf padded          (exact form)
    const float* r2p;     // [H, Tp + 256]: r * log2(e) at offset + 127  (exact form)
    const float* eap;     // [H, Tp]: exp(a - max a), 0 padded          (factorised form)
    const float* erp;     // [H, Tp + 256]: exp(r - max r) at offset + 127
    const float* invz;    // [H, Tp]: 1 / Z' of the factorised form
    const uint32_t* hflag;   // per head: bit 1 = use the exact form
    uint32_t* status;
    int B, H, T, ld, Tp;
    int Hkv, G;        // key/value heads; query heads per key/value head (query head h reads h / G)
    int nqb, npairs, n_items;
    int slice_group;   // (batch, head) slices per item group
    unsigned long long wait_ns;   // limit of every bounded wait (kWaitLimitNs unless a diagnostic call sets it)
    int withhold;      // diagnostic: the producer publishes no work item, so every waiter gives up
    int n_ord, n_frz;
    uint8_t ord_heads[SAF_MAX_HEADS];
    uint8_t frz_heads[SAF_MAX_HEADS];
};

// A stage holds K and V of one key block; for frozen items the K slot holds
// instead the block's slice of a (128 fp32 at byte 0) and the band of r both
// tiles need (384 fp32 at byte 1024), in the factorised form (exp(a - A),
// exp(r - R)) or, for flagged heads, in the exact form (log2 domain).
struct SmemLayout {
    static constexpr int q = 0;                                     // 2 slots x 2 tiles
    static constexpr int q_slot_bytes = 2 * kTileBytes;
    static constexpr int kv = q + 2 * q_slot_bytes;                 // kStages x (K, V)
    static constexpr int stage_bytes = 2 * kTileBytes;
    static constexpr int frz_band = 1024;
    static constexpr int total = kv + kStages * stage_bytes;
};

struct Item {
    int b, h, pair;
    bool frozen;
};

// Items are numbered group by group: the (batch, head) slices, ordinary before
// frozen, form groups of p.slice_group consecutive slices, and inside a group the
// query-block pairs go longest first, all slices of the group at one level before
// the next. A group's key and value tiles are re-read by each of its pairs, and
// they stay in L2 while the group runs. (With one group for all slices this is
// longest first over the whole launch.)
__device__ __forceinline__ Item decode_item(const FwdParams& p, int idx) {
    Item it;
    const int n_slices = p.B * p.H;
    const int G = p.slice_group;
    const int per_group = G * p.npairs;
    const int grp = idx / per_group;
    const int gsize = min(G, n_slices - grp * G);
    const int within = idx - grp * per_group;
    const int level = within / gsize;
    const int slice = grp * G + (within - level * gsize);
    it.pair = p.npairs - 1 - level;
    const int n_ord_items = p.B * p.n_ord;
    if (slice < n_ord_items) {
        it.b = slice / p.n_ord;
        it.h = p.ord_heads[slice - it.b * p.n_ord];
        it.frozen = false;
    } else {
        const int f = slice - n_ord_items;
        it.b = f / p.n_frz;
        it.h = p.frz_heads[f - it.b * p.n_frz];
        it.frozen = true;
    }
    return it;
}

// 2^x on the special-function unit (ex2.approx, flushes subnormal results to 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct Barriers {
    uint64_t q_full[2], q_empty[2];   // Q slot of alternate ordinary items
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2], s_empty[2], p_full[2], o_done[2];
    uint64_t w_full[2][2];   // frozen items: W buffer b of tile g is written (4 arrivals)
    uint64_t w_done[2][2];   // frozen items: P V of tile g that read W buffer b has completed
    uint64_t item_full[kRing], item_empty[kRing];   // work-item ring (10 consumer warps)
    uint64_t mma_idle[2];   // every MMA issuer g issued has completed (before TMEM is freed)
};

__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ FwdParams p) {
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.q_full[i], 1);
            mbar_init(&bars.q_empty[i], 2);   // one commit per issuer
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars.kv_full[s], 1);
            mbar_init(&bars.kv_empty[s], 2);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&bars.s_full[g], 1);
            mbar_init(&bars.s_empty[g], 4);
            mbar_init(&bars.p_full[g], 4);
            mbar_init(&bars.o_done[g], 1);
            mbar_init(&bars.w_done[g][0], 1);
            mbar_init(&bars.w_done[g][1], 1);
            mbar_init(&bars.w_full[g][0], 4);
            mbar_init(&bars.w_full[g][1], 4);
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bars.item_full[i], 1);
            mbar_init(&bars.item_empty[i], 10);   // 2 MMA issuers + 8 softmax warps
        }
        mbar_init(&bars.mma_idle[0], 1);
        mbar_init(&bars.mma_idle[1], 1);
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

    // warpgroup 2 (warps 8-11) gives up registers in one instruction for the whole
    // warpgroup; the softmax warpgroups take them
    if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            uint32_t q_empty_bits = 3;   // phase parity per Q slot
            int nord = 0;                // ordinary items so far: Q slot nord & 1
            uint32_t kv_empty_bits = (1u << kStages) - 1;   // phase parity per stage, bit s
            int stage = 0;
            bool ok = true;
            uint32_t ring_empty_bits = (1u << kRing) - 1;
            int slot = 0;
            // diagnostic call: publish nothing and leave; the other roles' first waits expire
            if (p.withhold) ok = false;
            while (ok) {
                // next item from the global counter (longest first), published to the ring
                if (!(ok = mbar_wait(&bars.item_empty[slot], (ring_empty_bits >> slot) & 1u, abort, status,
                                     kStatusTimeout, p.wait_ns)))
                    break;
                ring_empty_bits ^= 1u << slot;
                int idx = (int)atomicAdd(status + kCounterFwd, 1u);
                if (idx >= p.n_items) idx = -1;
                item_ring[slot] = idx;
                mbar_arrive(&bars.item_full[slot]);
                slot = (slot + 1) % kRing;
                if (idx < 0) break;
                const Item it = decode_item(p, idx);
                const int bh = it.b * p.H + it.h;
                const int bkv = it.b * p.Hkv + it.h / p.G;   // the key/value slice this head reads
                const int qb0 = 2 * it.pair, qb1 = qb0 + 1;
                const bool t1 = qb1 < p.nqb;
                const int nblk = t1 ? qb1 + 1 : qb0 + 1;
                const bool exact = it.frozen && (p.hflag[it.h] & 2u) != 0;
                if (!it.frozen) {
                    // the next item's Q goes to the other slot while this CTA may still work
                    // on the previous item
                    const int qs = nord++ & 1;
                    if (!(ok = mbar_wait(&bars.q_empty[qs], (q_empty_bits >> qs) & 1u, abort, status,
                                         kStatusTimeout, p.wait_ns)))
                        break;
                    q_empty_bits ^= 1u << qs;
                    uint8_t* sq = sm + SmemLayout::q + qs * SmemLayout::q_slot_bytes;
                    mbar_expect_tx(&bars.q_full[qs], (t1 ? 2 : 1) * kTileBytes);
                    tma_load_3d(sq, &p.tm_q, &bars.q_full[qs], 0, qb0 * 128, bh);
                    if (t1) tma_load_3d(sq + kTileBytes, &p.tm_q, &bars.q_full[qs], 0, qb1 * 128, bh);
                }
                for (int j = 0; j < nblk; ++j) {
                    if (!(ok = mbar_wait(&bars.kv_empty[stage], (kv_empty_bits >> stage) & 1u, abort, status,
                                         kStatusTimeout, p.wait_ns)))
                        break;
                    kv_empty_bits ^= 1u << stage;
                    uint8_t* st = sm + SmemLayout::kv + stage * SmemLayout::stage_bytes;
                    if (!it.frozen) {
                        mbar_expect_tx(&bars.kv_full[stage], 2 * kTileBytes);
                        tma_load_3d(st, &p.tm_k, &bars.kv_full[stage], 0, j * 128, bkv);
                    } else {
                        const float* as = exact ? p.a2p : p.eap;
                        const float* rs = exact ? p.r2p : p.erp;
                        mbar_expect_tx(&bars.kv_full[stage], kTileBytes + 512 + 1536);
                        bulk_load(st, as + (size_t)it.h * p.Tp + (size_t)j * 128, 512, &bars.kv_full[stage]);
                        bulk_load(st + SmemLayout::frz_band,
                                  rs + (size_t)it.h * (p.Tp + 256) + (size_t)(qb0 - j) * 128, 1536,
                                  &bars.kv_full[stage]);
                    }
                    tma_load_3d(st + kTileBytes, &p.tm_v, &bars.kv_full[stage], 0, j * 128, bkv);
                    stage = (stage + 1 == kStages) ? 0 : stage + 1;
                }
            }
        }
    } else if (warp == 9 || warp == 10) {
        // ------------------------------------------------------------ MMA issuer of tile g
        // The whole warp runs the issue loop (warp-uniform descriptors); one elected lane
        // issues each MMA and commit, lane 0 waits on barriers and arrives.
        {
            const int g = warp - 9;
            const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);  // S = Q K^T
            const uint32_t idesc_o = idesc_bf16(128, 64, 0, 1);   // O += P V, V MN-major
            uint32_t q_full_bits = 0;    // phase parity per Q slot
            int nord = 0;                // ordinary items so far: Q slot nord & 1
            uint32_t kv_full_bits = 0;   // phase parity per stage, bit s
            uint32_t s_empty_ph = 1, p_full_ph = 0, w_full_bits = 0;
            int stage = 0;
            bool ok = true;
            uint64_t d_q = 0;   // this tile's Q (slot of the current item), K-major
            int qs = 0;
            const uint32_t d_s = tmem + 256 * g, d_p = d_s + 128, d_o = d_s + 192;
            uint32_t ring_full_bits = 0;
            int slot = 0;
            while (ok) {
                if (!(ok = mbar_wait_warp(&bars.item_full[slot], (ring_full_bits >> slot) & 1u, abort, status,
                                     kStatusTimeout, p.wait_ns)))
                    break;
                ring_full_bits ^= 1u << slot;
                const int idx = item_ring[slot];
                if (lane == 0) mbar_arrive(&bars.item_empty[slot]);
                slot = (slot + 1) % kRing;
                if (idx < 0) break;
                const Item it = decode_item(p, idx);
                const int qb0 = 2 * it.pair, qb1 = qb0 + 1;
                const bool t1 = qb1 < p.nqb;
                const int ng = g == 0 ? qb0 + 1 : (t1 ? qb1 + 1 : 0);   // key blocks of my tile
                const int nblk = t1 ? qb1 + 1 : qb0 + 1;                 // key blocks of the item
                if (!it.frozen) {
                    qs = nord++ & 1;
                    if (!(ok = mbar_wait_warp(&bars.q_full[qs], (q_full_bits >> qs) & 1u, abort, status, kStatusTimeout, p.wait_ns)))
                        break;
                    q_full_bits ^= 1u << qs;
                    d_q = sdesc_sw128(smem_u32(sm + SmemLayout::q + qs * SmemLayout::q_slot_bytes) + g * kTileBytes, 16,
                                      1024);
                }
                // stage index of block j is (stage + j) mod kStages
                auto stage_of = [&](int j) { return (stage + j) % kStages; };
                auto issue_s = [&](int j) -> bool {
                    if (!mbar_wait_warp(&bars.s_empty[g], s_empty_ph, abort, status, kStatusTimeout, p.wait_ns)) return false;
                    s_empty_ph ^= 1;
                    tc_fence_after();
                    const uint64_t d_k =
                        sdesc_sw128(smem_u32(sm + SmemLayout::kv + stage_of(j) * SmemLayout::stage_bytes), 16, 1024);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss_warp(d_s, sdesc_advance(d_q, 32 * k), sdesc_advance(d_k, 32 * k), idesc_s, k > 0);
                    mma_commit_warp(&bars.s_full[g]);
                    return true;
                };
                // frozen items alternate W between the P columns and the (unused) S columns
                const bool frz = it.frozen;
                auto issue_pv = [&](int j) -> bool {
                    if (frz) {   // one barrier per W buffer: the softmax group may be a block ahead
                        const int b = j & 1;
                        if (!mbar_wait_warp(&bars.w_full[g][b], (w_full_bits >> b) & 1u, abort, status, kStatusTimeout, p.wait_ns))
                            return false;
                        w_full_bits ^= 1u << b;
                    } else {
                        if (!mbar_wait_warp(&bars.p_full[g], p_full_ph, abort, status, kStatusTimeout, p.wait_ns)) return false;
                        p_full_ph ^= 1;
                    }
                    tc_fence_after();
                    const uint64_t d_v = sdesc_sw128(
                        smem_u32(sm + SmemLayout::kv + stage_of(j) * SmemLayout::stage_bytes + kTileBytes), 16384, 1024);
                    const uint32_t a = (frz && (j & 1)) ? d_s : d_p;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_ts_warp(d_o, a + 8 * k, sdesc_advance(d_v, 2048 * k), idesc_o,
                               (j > 0 || k > 0) ? 1u : 0u);
                    mma_commit_warp(frz ? &bars.w_done[g][j & 1] : &bars.o_done[g]);
                    return true;
                };
                int kv_ready = 0;   // blocks of this item whose K/V stage has been waited for
                auto ensure_kv = [&](int j) -> bool {
                    while (kv_ready <= j) {
                        const int s = stage_of(kv_ready);
                        if (!mbar_wait_warp(&bars.kv_full[s], (kv_full_bits >> s) & 1u, abort, status, kStatusTimeout, p.wait_ns))
                            return false;
                        kv_full_bits ^= 1u << s;
                        ++kv_ready;
                    }
                    return true;
                };
                if (!it.frozen && ng > 0) ok = ensure_kv(0) && issue_s(0);
                // Per block j: the next block's S (as soon as the softmax group has read this
                // block's S, so that it runs under the softmax), then P V. Every issuer waits
                // for and releases every stage of the item, used or not.
                for (int j = 0; j < nblk && ok; ++j) {
                    if (!(ok = ensure_kv(j))) break;
                    if (!it.frozen && j + 1 < ng) ok = ensure_kv(j + 1) && issue_s(j + 1);
                    // A frozen item's W also sits in the S columns. The softmax group arrives on
                    // s_empty once the item's last P V is done, and the next S waits for that
                    // phase; its predecessor phase is taken here, before that last P V is issued,
                    // so that s_empty never runs two phases ahead of this thread.
                    if (ok && it.frozen && j + 1 == ng) {
                        ok = mbar_wait_warp(&bars.s_empty[g], s_empty_ph, abort, status, kStatusTimeout, p.wait_ns);
                        s_empty_ph ^= 1;
                    }
                    if (ok && j < ng) ok = issue_pv(j);
                    if (!ok) break;
                    mma_commit_warp(&bars.kv_empty[stage_of(j)]);
                }
                if (!ok) break;
                if (!it.frozen) mma_commit_warp(&bars.q_empty[qs]);
                stage = stage_of(nblk);
            }
            // Tensor memory is freed at the end: every MMA issued here must have completed
            // (after an abort the last ones may still run), with a bounded wait of its own.
            mma_commit_warp(&bars.mma_idle[g]);
            if (lane == 0) mbar_wait_bounded(&bars.mma_idle[g], 0, kWaitLimitNs);
            __syncwarp();
        }
    }   // warp 11: idle
    } else {
        // ------------------------------------------------------------ softmax groups
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        const int g = warp >> 2;               // 0 or 1
        const int r = threadIdx.x & 127;       // row within the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 256 * g;
        uint32_t s_full_ph = 0, o_done_ph = 0;
        uint32_t w_done_ph[2] = {0, 0};
        bool w_pend[2] = {false, false};   // a P V that read W buffer b may not have been waited for
        auto wait_w = [&](int b) -> bool {
            if (!w_pend[b]) return true;
            if (!mbar_wait(&bars.w_done[g][b], w_done_ph[b], abort, status, kStatusTimeout, p.wait_ns)) return false;
            w_done_ph[b] ^= 1;
            w_pend[b] = false;
            tc_fence_after();
            return true;
        };
        // epilogue of a row: O (tensor memory) times inv, rounded to bf16, and the row's lse
        auto store_o = [&](int bh, int row, float inv, float lse_row) {
            uint32_t ov[64];
            tmem_ld32(lane_base + 192, ov);
            tmem_ld32(lane_base + 224, ov + 32);
            tmem_ld_wait();
            tc_fence_before();
            if (row < p.T) {
                uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)bh * p.T + row) * 64);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(ov[8 * c + 0]) * inv, __uint_as_float(ov[8 * c + 1]) * inv);
                    w.y = pack_bf16(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv);
                    w.z = pack_bf16(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv);
                    w.w = pack_bf16(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv);
                    dst[c] = w;
                }
                p.lse[(size_t)bh * p.T + row] = lse_row;
            }
        };
        int gblk = 0;   // key blocks of all previous items of this CTA (stage = gblk % kStages)
        bool ok = true;
        uint32_t ring_full_bits = 0;
        int slot = 0;
        while (ok) {
            if (!(ok = mbar_wait(&bars.item_full[slot], (ring_full_bits >> slot) & 1u, abort, status,
                                 kStatusTimeout, p.wait_ns)))
                break;
            ring_full_bits ^= 1u << slot;
            const int idx = item_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.item_empty[slot]);
            slot = (slot + 1) % kRing;
            if (idx < 0) break;
            const Item it = decode_item(p, idx);
            const int item_blocks = (2 * it.pair + 1 < p.nqb) ? 2 * it.pair + 2 : 2 * it.pair + 1;
            const int gblk0 = gblk;
            gblk += item_blocks;
            const int qb = 2 * it.pair + g;
            if (qb >= p.nqb) continue;
            const int bh = it.b * p.H + it.h;
            const int row = qb * 128 + r;
            const int nblk = qb + 1;
            if (!it.frozen) {
                float m_used = -INFINITY, l = 0.f;
                for (int j = 0; j < nblk && ok; ++j) {
                    if (!(ok = mbar_wait(&bars.s_full[g], s_full_ph, abort, status, kStatusTimeout, p.wait_ns))) break;
                    s_full_ph ^= 1;
                    tc_fence_after();
                    uint32_t sr[128];   // this row of S (raw scores)
#pragma unroll
                    for (int c0 = 0; c0 < 128; c0 += 32) tmem_ld32(lane_base + c0, sr + c0);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.s_empty[g]);
                    if (j == qb) {
                        // causal mask on the diagonal tile: keys c > r are dropped
#pragma unroll
                        for (int c = 0; c < 128; ++c)
                            if (c > r) sr[c] = __float_as_uint(-INFINITY);
                    }
                    // row max of the raw scores (the scale is positive): two chains of 3-input max
                    float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 128; c += 4) {
                        ma = fmax3(ma, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                        mb = fmax3(mb, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                    }
                    const float mx = fmaxf(ma, mb) * kScaleLog2;
                    const float m_new = fmaxf(m_used, mx);
                    const bool need = m_new > m_used + kRescaleThreshold;
                    const float f = need ? fast_exp2(m_used - m_new) : 1.f;   // O and l rescale factor
                    if (need) {
                        l *= f;
                        m_used = m_new;
                    }
                    // P = 2^(S log2(e) / sqrt(d) - m), two columns per FFMA and per FADD, packed
                    // into registers while the previous block's P V may still run
                    const float2 sc2 = make_float2(kScaleLog2, kScaleLog2);
                    const float2 nm2 = make_float2(-m_used, -m_used);
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
                    uint32_t pk[64];   // packed bf16 pairs of the row's 128 columns of P
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const float2 x =
                            ffma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, nm2);
                        const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        if (c & 1)
                            acc1 = fadd2(acc1, e);
                        else
                            acc0 = fadd2(acc0, e);
                        pk[c] = pack_bf16(e.x, e.y);
                    }
                    if (j > 0) {   // P V of the previous block done: P is free, O is stable
                        if (!(ok = mbar_wait(&bars.o_done[g], o_done_ph, abort, status, kStatusTimeout, p.wait_ns))) break;
                        o_done_ph ^= 1;
                        tc_fence_after();
                    }
                    tmem_st32(lane_base + 128, pk);
                    tmem_st32(lane_base + 160, pk + 32);
                    l += (acc0.x + acc1.x) + (acc0.y + acc1.y);
                    // rescale O (stable: the previous P V is done) before this block's P V adds
                    // to it; done after the exp loop, when the row's scores no longer hold registers
                    if (j > 0 && __any_sync(0xffffffffu, need)) {
                        uint32_t ov[16];
#pragma unroll
                        for (int c0 = 0; c0 < 64; c0 += 16) {
                            tmem_ld16(lane_base + 192 + c0, ov);
                            tmem_ld_wait();
#pragma unroll
                            for (int c = 0; c < 16; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * f);
                            tmem_st16(lane_base + 192 + c0, ov);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.p_full[g]);
                }
                if (!ok) break;
                // epilogue: O = acc / l
                if (!(ok = mbar_wait(&bars.o_done[g], o_done_ph, abort, status, kStatusTimeout, p.wait_ns))) break;
                o_done_ph ^= 1;
                tc_fence_after();
                store_o(bh, row, 1.f / l, (m_used + log2f(l)) / kLog2e);
            } else {
                // frozen item: the exact or the factorised form of Eq. 3 (per-head flag)
                const bool exact = (p.hflag[it.h] & 2u) != 0;
                const float lz2 = row < p.T ? p.lz[(size_t)it.h * p.T + row] * kLog2e : INFINITY;   // log2 Z(i)
                for (int j = 0; j < nblk && ok; ++j) {
                    // Frozen tile of Eq. 3 from the key block's a values and the band of r values
                    // the producer staged in the K slot. Factorised form: W(i, k) Z'(i) =
                    // exp(r[i-k] - R) exp(a[k] - A), no exp per element (1 / Z' is applied to O).
                    // Exact form: W(i, k) = exp(a[k] + r[i - k] - log Z(i)).
                    const int G = gblk0 + j;
                    const int st = G % kStages;
                    if (!(ok = mbar_wait(&bars.kv_full[st], (uint32_t)(G / kStages) & 1u, abort, status,
                                         kStatusTimeout, p.wait_ns)))
                        break;
                    // W buffer j & 1 (P columns, or the S columns frozen items leave unused) is
                    // free once the P V of block j - 2 has read it
                    const int wb = j & 1;
                    if (!(ok = wait_w(wb))) break;
                    const uint32_t wcol = wb ? 0u : 128u;
                    const float* a2s = reinterpret_cast<const float*>(sm + SmemLayout::kv + st * SmemLayout::stage_bytes);
                    // bnd[-c] = r * log2(e) at offset i - k = (qb - j) * 128 + r - c
                    const float* bnd = reinterpret_cast<const float*>(sm + SmemLayout::kv + st * SmemLayout::stage_bytes +
                                                                      SmemLayout::frz_band) +
                                       128 * g + r + 127;
                    if (!exact) {
                        // W is Toeplitz up to the column factor exp(a[k] - A). In the 16x128b
                        // shape a thread holds rows 32 wq + rho + 8 m (m = 0..3) at packed
                        // columns 4 j + q, keys k = 8 j + 2 q + {0, 1} (j = 0..15): the band
                        // value of (row, k) depends on m - j alone, so 38 band loads serve
                        // the thread's 128 products (one per product in the row-per-thread
                        // shape).
                        const int wq = warp & 3, rho = lane >> 2, q = lane & 3;
                        const float* b0 = bnd - r + 32 * wq + rho - 2 * q;   // b0[8 (m - j) - v]
                        float e0[19], e1[19];   // index m - j + 15
#pragma unroll
                        for (int d = -15; d <= 3; ++d) {
                            e0[d + 15] = b0[8 * d];
                            e1[d + 15] = b0[8 * d - 1];
                        }
                        float2 ea[16];
#pragma unroll
                        for (int j2 = 0; j2 < 16; ++j2) ea[j2] = *reinterpret_cast<const float2*>(a2s + 8 * j2 + 2 * q);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            uint32_t pk[32];
#pragma unroll
                            for (int j2 = 0; j2 < 16; ++j2) {
#pragma unroll
                                for (int s2 = 0; s2 < 2; ++s2) {
                                    const int d = 2 * hh + s2 - j2 + 15;
                                    const float2 w = fmul2(make_float2(e0[d], e1[d]), ea[j2]);
                                    pk[2 * j2 + s2] = pack_bf16(w.x, w.y);
                                }
                            }
                            tmem_st_16x128b_x16(lane_base + ((uint32_t)(16 * hh) << 16) + wcol, pk);
                        }
                    } else {
#pragma unroll
                        for (int h4 = 0; h4 < 4; ++h4) {
                            uint32_t pk[16];
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const int cc = 32 * h4 + 2 * c;
                                const float w0 = fast_exp2(a2s[cc] + bnd[-cc] - lz2);
                                const float w1 = fast_exp2(a2s[cc + 1] + bnd[-cc - 1] - lz2);
                                pk[c] = pack_bf16(w0, w1);
                            }
                            tmem_st16(lane_base + wcol + 16 * h4, pk);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.w_full[g][j & 1]);
                    w_pend[j & 1] = true;
                }
                if (!ok) break;
                // the last P V (and, completing in order, every earlier one) is done; the next
                // item's S may now overwrite the W columns
                if (!(ok = wait_w((nblk - 1) & 1))) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.s_empty[g]);
                // epilogue: W rows sum to one in the exact form and carry the factor Z'(i) in
                // the factorised form
                const float inv = (exact || row >= p.T) ? 1.f : p.invz[(size_t)it.h * p.Tp + row];
                store_o(bh, row, inv, lz2 / kLog2e);
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

}  // namespace

cudaError_t launch_tc_fwd(const LayerArgs& a, cudaStream_t s) {
    FwdParams p;
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
        !make_tmap_bf16_3d(&p.tm_v, vbase, 64, a.T, BHkv, 64, 128))
        return cudaErrorInvalidValue;
    p.o = (__nv_bfloat16*)a.out;
    p.lse = a.lse_out;
    p.lz = a.lz;
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
    p.ld = a.ld_prior;
    p.nqb = (a.T + 127) / 128;
    p.Tp = p.nqb * 128;
    p.npairs = (p.nqb + 1) / 2;
    p.n_items = a.B * a.H * p.npairs;
    // K and V of every slice: 2 x T x 64 bf16 each. When all of them fit in part of
    // the L2 one group keeps the launch longest first (best balance); otherwise
    // groups of kSliceGroup slices keep each group's K and V in L2 while its
    // query pairs re-read them.
    const size_t kv_all = (size_t)BHkv * 2 * (size_t)a.T * 64 * 2;
    p.slice_group = kv_all <= kL2GroupBytes ? a.B * a.H : kSliceGroup;
    p.wait_ns = a.diag_wait_ns ? a.diag_wait_ns : kWaitLimitNs;
    p.withhold = a.diag_withhold;
    for (int h = 0; h < a.H; ++h) {
        if (head_frozen(a.mask, h))
            p.frz_heads[p.n_frz++] = (uint8_t)h;
        else
            p.ord_heads[p.n_ord++] = (uint8_t)h;
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = SmemLayout::total + 1024;
    cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // The register split inside the kernel draws on the registers the launch hands out: a
    // build that launches with fewer than kRegsLaunch per thread is refused here, since the
    // softmax warpgroups could then never obtain theirs.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fwd_tc_kernel);
    if (e != cudaSuccess) return e;
    if (2 * 128 * kRegsSoftmax + 128 * kRegsOther > kThreads * fa.numRegs) return cudaErrorInvalidConfiguration;
    const int grid = p.n_items < sms ? p.n_items : sms;
    before_launch(SAF_KERNEL_FWD, s);
    e = launch_ex(fwd_tc_kernel, dim3(grid), dim3(kThreads), smem, s, true, 1, p);
    after_launch(SAF_KERNEL_FWD, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace saf
