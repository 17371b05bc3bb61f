// Gradients of the frozen patterns' parameters on the tensor cores (bf16,
// d = 64), for the trainable-pattern variant ("When Can Attention Heads Be
// Statically Defined?", App. C.3.2: the patterns keep training and their
// normalisers are refreshed after each update).
//
// Eq. 3 is a row softmax of the logits L(i, j) = a(j) + r(i - j). With
// G(i, j) = dO_i . V_j and D_i = sum_j W(i, j) G(i, j) = dO_i . O_i,
//     dL(i, j) = W(i, j) (G(i, j) - D_i),
//     da(j) = sum_b sum_{i >= j} dL(i, j),   dr(d) = sum_b sum_{i >= d} dL(i, i - d).
//
// The causal 128 x 128 tiles (key block kb, query block qb >= kb) are taken
// band by band: a work item is (batch b, frozen head f, band = qb - kb) and
// runs over kb = 0 .. nqb - 1 - band. Each element a pattern thread holds lies
// at the same distance i - j in every tile of the band, so the thread sums its
// elements over the band in registers and the diagonal sums (dr) are formed
// once per band; the key-row sums (da) are formed per tile. In the factorised
// form of Eq. 3 (W = ea(j) er(i - j) / Z'(i), the layer's own form) er(i - j)
// is then also the same for all of a thread's terms of one element and is
// applied once, at the end of the band.
//
// Four launches, all enqueued on the caller's stream:
//   call_init_kernel    the layer's: maxima and padded slices of a and r
//   pg_prep_kernel      D_i of every frozen slice; 1 / Z' and log2 Z of every
//                       frozen head from the log Z rows of lse, and the
//                       exact-form flag
//   pg_tc_kernel        persistent, one CTA per SM; per tile
//                         G^T = V_kb dO_qb^T                 (tcgen05, TMEM, 2 buffers)
//                         dL^T(j, q) = W^T(j, q) (G^T(j, q) - D_q)
//                       writes one key-row sum per tile and 256 diagonal sums
//                       per band into per-item slots of the workspace
//   pg_reduce_kernel    da, dr: the slots summed in a fixed order, so the
//                       result has the same bits on every run
//
// pg_tc_kernel warp roles (320 threads): warps 0-7 pattern warps (warp w: key
// rows 32 (w % 4) .. + 31 = its TMEM lanes, query columns 64 (w / 4) .. + 63),
// warp 8 producer (per tile: V, dO and the row vectors), warp 9 tensor-memory
// owner and single-thread MMA issuer. A pattern thread reads G^T in the 16x256b
// shape: lane l = 4 rho + qq holds key rows rho + 8 m (m = 0..3) of its warp's
// 32 and query columns 8 jr + 2 qq + s (jr = 0..7, s = 0, 1) of its 64. Its 64
// elements then lie at only 22 distances, 8 (jr - m) + 2 qq - rho + s + const,
// so it keeps 22 band sums and 22 r factors in registers; the two columns s = 0, 1
// sit in adjacent registers at adjacent distances and are taken together by the
// paired fp32 instructions, and each column's D and 1 / Z' serve four elements.
#include <math.h>
#include <string.h>

#include "saf_internal.h"
#include "tc_common.cuh"

namespace saf {
namespace {

using namespace tc;

constexpr int kTileBytes = 128 * 64 * 2;   // one 128 x 64 bf16 tile
constexpr int kThreads = 320;
constexpr int kStagesMax = 5;   // load stages at d = 64 (PgSmem::stages for the wider heads)
constexpr int kRing = 4;
constexpr int kScrCols = 96;               // a warp's 95 distances, + 1
constexpr int kScrRows = 8;                // rows of a warp's skew buffer (4 rounds of 8 lanes)
constexpr int kScrStride = 98;             // its row stride in floats (spreads the banks)
constexpr float kLog2e = 1.4426950408889634f;

struct PgParams {
    CUtensorMap tm_v;
    CUtensorMap tm_do;
    // Row vectors in tile order (qperm / kperm below), per 128-block:
    float* yx;       // [B, F, Tp]: D_i = dO_i . O_i of the frozen slices (0 past T)   (exact form)
    float* yf;       // [B, F, Tp]: -D_i / Z'(i)                                    (factorised form)
    float* zx;       // [F, Tp]: log2 Z (+inf past T)
    float* zf;       // [F, Tp]: 1 / Z' (0 past T)
    float* ex;       // [F, Tp]: a * log2(e) (-inf past T)
    float* ef;       // [F, Tp]: exp(a - max a) (0 past T)
    // the layer's padded slices of r, read as 256-entry windows
    const float* r2p;      // [H, Tp + 256]: r * log2(e), + 127    (exact form)
    const float* erp;      // [H, Tp + 256]: exp(r - max r), + 127 (factorised form)
    const uint32_t* hflag; // per head: bit 1 = use the exact form
    float* da_part;        // [B, F, nqb (band), 2 (column half), Tp]: key-row sums of each tile
    float* dr_part;        // [B, F, nqb (band), 256]: entry e = distance 128 band + e - 128
    uint32_t* status;
    int B, H, T, Tp, nqb, F, n_items;
    int d;                 // head dimension (64, 96 or 128)
    uint8_t frz_heads[SAF_MAX_HEADS];
};

// Position of query column c (0..127) of a block in the tile order of the row
// vectors: a pattern thread with qq in column half c / 64 reads its 16 columns
// 8 jr + 2 qq + s (jr = 0..7, s = 0, 1) as four float4, jr = 2 i + e / 2,
// s = e % 2 at position 64 half + 16 i + 4 qq + e; the four qq of one float4
// index are 64 contiguous bytes (one shared-memory wavefront).
__host__ __device__ __forceinline__ int qperm(int c) {
    const int r = c & 63;
    return (c & 64) + (r >> 4) * 16 + ((r >> 1) & 3) * 4 + ((r >> 3) & 1) * 2 + (r & 1);
}
// Position of key row j (0..127) of a block: rows 32 quarter + rho + 8 m of a
// thread (m = 0..3) at 32 quarter + 4 rho + m, one float4 per thread.
__host__ __device__ __forceinline__ int kperm(int j) { return (j & 96) + (j & 7) * 4 + ((j >> 3) & 3); }

// Shared memory for head dimensions up to kD (64, or 128 for d = 96 and 128: a tile is
// then two 128-byte-swizzled atoms of 64 columns, and TMA fills the columns past d
// with zeros, which add nothing to G).
template <int kD>
struct PgSmem {
    static constexpr int atoms = kD / 64;
    static constexpr int stages = kD == 64 ? kStagesMax : 2;
    // per stage: V tile of key block kb, dO tile of query block kb + band, row vectors
    static constexpr int st_v = 0;
    static constexpr int st_do = atoms * kTileBytes;
    // row vectors, factorised form: 1/Z' [128] | -D/Z' [128] | ea [128] | er band [256];
    // exact form: log2 Z | D | a * log2(e) | r * log2(e) band (the first three in tile order)
    static constexpr int st_vec = 2 * atoms * kTileBytes;
    static constexpr int vec_bytes = 512 * 3 + 1024;
    static constexpr int st_bytes = 2 * atoms * kTileBytes + 3072;   // 1024-aligned
    static constexpr int scr = stages * st_bytes;                      // 8 warps x [8 x 98] fp32
    static constexpr int wsum = scr + 8 * kScrRows * kScrStride * 4;  // 2 (band parity) x 8 warps x 96 fp32
    static constexpr int total = wsum + 2 * 8 * kScrCols * 4;
    static_assert(st_bytes % 1024 == 0, "stage tiles must stay 1024-aligned");
    static_assert(total + 1024 <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// mbar_wait with a non-blocking test first: a phase that has already completed
// (the common case in the pattern warps' loop) costs one test.
__device__ __forceinline__ bool pg_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done ? true : mbar_wait(bar, parity, abort, status, kStatusTimeout);
}

// tcgen05.ld 16x256b, 8 repetitions: per repetition jr, r[4 jr + 2 h + s] = (lane
// l / 4 + 8 h, column 8 jr + 2 (l % 4) + s) of the 16 lanes starting at taddr's lane.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// One 16-lane block of a tile in the pattern thread's registers: elements (key row
// rho + 8 m, m = 2 blk + mm; query columns 8 jr + 2 qq + {0, 1}), a pair at
// adjacent distances, entry pi = jr - m + 3 of the band sums and r factors; two
// fp32 lanes per instruction.
//   factorised: x = (G - D) / Z' = G z + y (z = 1 / Z', y = -D / Z'),
//               acc += ea x (dr, before er), rs += er x (da, before ea)
//   exact:      dL = exp2(a2 + r2 - log2 Z) (G - D),  acc += dL, rs += dL
template <bool kExact>
__device__ __forceinline__ void pg_block(const uint32_t (&g)[32], int blk, const float2 (&zc)[8],
                                         const float2 (&yc)[8], const float (&ek)[4], const float2 (&bnd)[11],
                                         float2 (&acc)[11], float2 (&rs)[4]) {
#pragma unroll
    for (int jr = 0; jr < 8; ++jr) {
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            const int m = 2 * blk + mm, pi = jr - m + 3;
            const float2 gv = make_float2(__uint_as_float(g[4 * jr + 2 * mm]), __uint_as_float(g[4 * jr + 2 * mm + 1]));
            const float2 e2 = make_float2(ek[m], ek[m]);
            if (!kExact) {
                const float2 x = ffma2(gv, zc[jr], yc[jr]);
                acc[pi] = ffma2(e2, x, acc[pi]);
                rs[m] = ffma2(bnd[pi], x, rs[m]);
            } else {
                const float2 sx = fsub2(fadd2(e2, bnd[pi]), zc[jr]);
                const float2 dl = fmul2(make_float2(fast_exp2(sx.x), fast_exp2(sx.y)), fsub2(gv, yc[jr]));
                acc[pi] = fadd2(acc[pi], dl);
                rs[m] = fadd2(rs[m], dl);
            }
        }
    }
}

struct PgBarriers {
    uint64_t item_full[kRing], item_empty[kRing];
    uint64_t st_full[kStagesMax], st_empty[kStagesMax];
    uint64_t g_full[2], g_free[2];
    uint64_t band_sync;
    uint64_t mma_idle;
};

template <int kD>
__global__ void __launch_bounds__(kThreads, 1) pg_tc_kernel(const __grid_constant__ PgParams p) {
    using PgSmem = saf::PgSmem<kD>;
    constexpr int kStages = PgSmem::stages;
    constexpr int kAtoms = PgSmem::atoms;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ PgBarriers bars;
    __shared__ int item_ring[kRing];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    grid_dep_wait();
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bars.item_full[i], 1);
            mbar_init(&bars.item_empty[i], 9);   // MMA warp + 8 pattern warps
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars.st_full[i], 1);
            mbar_init(&bars.st_empty[i], 9);     // MMA commit + 8 pattern warps (row vectors read)
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.g_full[i], 1);
            mbar_init(&bars.g_free[i], 8);
        }
        mbar_init(&bars.band_sync, 8);
        mbar_init(&bars.mma_idle, 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&tmem_base_sh, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abort = &abort_flag;
    uint32_t* status = p.status;
    const int nqb = p.nqb;
    auto decode = [&](int idx, int& b, int& f, int& band) {
        const int per = p.B * p.F;
        band = idx / per;
        const int rem = idx - band * per;
        b = rem / p.F;
        f = rem - b * p.F;
    };

    if (warp == 8) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_do);
            uint32_t ring_empty_bits = (1u << kRing) - 1, st_empty_bits = (1u << kStages) - 1;
            int slot = 0, stage = 0;
            bool ok = true;
            while (ok) {
                if (!(ok = mbar_wait(&bars.item_empty[slot], (ring_empty_bits >> slot) & 1u, abort, status,
                                     kStatusTimeout)))
                    break;
                ring_empty_bits ^= 1u << slot;
                // bands in ascending order: the longest items first
                int idx = (int)atomicAdd(status + kCounterBwd, 1u);
                if (idx >= p.n_items) idx = -1;
                item_ring[slot] = idx;
                mbar_arrive(&bars.item_full[slot]);
                slot = (slot + 1) % kRing;
                if (idx < 0) break;
                int b, f, band;
                decode(idx, b, f, band);
                const int h = p.frz_heads[f];
                const int bh = b * p.H + h;
                const bool exact = (p.hflag[h] & 2u) != 0;
                const float* zrow = (exact ? p.zx : p.zf) + (size_t)f * p.Tp;
                const float* yrow = (exact ? p.yx : p.yf) + (size_t)(b * p.F + f) * p.Tp;
                const float* erow = (exact ? p.ex : p.ef) + (size_t)f * p.Tp;
                const float* brow = (exact ? p.r2p : p.erp) + (size_t)h * (p.Tp + 256) + (size_t)band * 128;
                for (int kb = 0; kb + band < nqb; ++kb) {
                    const int qb = kb + band;
                    if (!(ok = mbar_wait(&bars.st_empty[stage], (st_empty_bits >> stage) & 1u, abort, status,
                                         kStatusTimeout)))
                        break;
                    st_empty_bits ^= 1u << stage;
                    uint8_t* st = sm + stage * PgSmem::st_bytes;
                    float* vec = reinterpret_cast<float*>(st + PgSmem::st_vec);
                    uint64_t* full = &bars.st_full[stage];
                    mbar_expect_tx(full, 2 * kAtoms * kTileBytes + PgSmem::vec_bytes);
#pragma unroll
                    for (int at = 0; at < kAtoms; ++at) {   // 64 columns per atom
                        tma_load_3d(st + PgSmem::st_v + at * kTileBytes, &p.tm_v, full, 64 * at, kb * 128, bh);
                        tma_load_3d(st + PgSmem::st_do + at * kTileBytes, &p.tm_do, full, 64 * at, qb * 128, bh);
                    }
                    bulk_load(vec, zrow + (size_t)qb * 128, 512, full);
                    bulk_load(vec + 128, yrow + (size_t)qb * 128, 512, full);
                    bulk_load(vec + 256, erow + (size_t)kb * 128, 512, full);
                    bulk_load(vec + 384, brow, 1024, full);
                    stage = (stage + 1) % kStages;
                }
            }
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_g = idesc_bf16(128, 128, 0, 0);   // G^T = V dO^T, both K-major
            uint32_t ring_full_bits = 0, st_full_bits = 0, g_free_bits = 3;
            int slot = 0, stage = 0, tile = 0;
            bool ok = true;
            while (ok) {
                if (!(ok = mbar_wait(&bars.item_full[slot], (ring_full_bits >> slot) & 1u, abort, status,
                                     kStatusTimeout)))
                    break;
                ring_full_bits ^= 1u << slot;
                const int idx = item_ring[slot];
                mbar_arrive(&bars.item_empty[slot]);
                slot = (slot + 1) % kRing;
                if (idx < 0) break;
                int b, f, band;
                decode(idx, b, f, band);
                for (int kb = 0; kb + band < nqb; ++kb) {
                    const int s = stage, gb = tile & 1;
                    if (!(ok = mbar_wait(&bars.st_full[s], (st_full_bits >> s) & 1u, abort, status, kStatusTimeout)))
                        break;
                    st_full_bits ^= 1u << s;
                    // buffer gb is free once the pattern warps have read the tile before last
                    if (!(ok = mbar_wait(&bars.g_free[gb], (g_free_bits >> gb) & 1u, abort, status, kStatusTimeout)))
                        break;
                    g_free_bits ^= 1u << gb;
                    tc_fence_after();
                    const uint32_t st = smem_u32(sm + s * PgSmem::st_bytes);
                    const uint64_t d_v = sdesc_sw128(st + PgSmem::st_v, 16, 1024);
                    const uint64_t d_do = sdesc_sw128(st + PgSmem::st_do, 16, 1024);
#pragma unroll
                    for (int k = 0; k < 4 * kAtoms; ++k) {   // K = 16 per step, 4 steps per atom
                        const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                        mma_ss(tmem + 128 * gb, sdesc_advance(d_v, off), sdesc_advance(d_do, off), id_g, k > 0);
                    }
                    mma_commit(&bars.g_full[gb]);
                    mma_commit(&bars.st_empty[s]);
                    stage = (stage + 1) % kStages;
                    ++tile;
                }
            }
            // every MMA issued has completed before the tensor memory is released
            mma_commit(&bars.mma_idle);
            mbar_wait_bounded(&bars.mma_idle, 0, kWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------------- pattern warps
        const int quarter = warp & 3, half = warp >> 2;
        const int rho = lane >> 2, qq = lane & 3;
        // my key rows 32 quarter + rho + 8 m (m = 0..3): TMEM lanes of the two 16-lane loads
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        float* scr = reinterpret_cast<float*>(sm + PgSmem::scr) + warp * kScrRows * kScrStride;
        float* wsum = reinterpret_cast<float*>(sm + PgSmem::wsum);
        uint32_t ring_full_bits = 0, st_full_bits = 0, g_full_bits = 0, band_ph = 0;
        int slot = 0, stage = 0, tile = 0, nband = 0;
        bool ok = true;
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
            int b, f, band;
            decode(idx, b, f, band);
            const int h = p.frz_heads[f];
            const bool exact = (p.hflag[h] & 2u) != 0;
            const size_t slot_row = ((size_t)b * p.F + f) * nqb + band;
            // Element (row rho + 8 m, column 8 jr + 2 qq + s) lies at distance
            //   128 band + 64 half - 32 quarter + 8 (pi - 3) + 2 qq - rho + s,   pi = jr - m + 3.
            // acc[pi].s: my elements at that distance summed over the band (factorised form:
            // without their common er factor); bnd[pi].s: er, or r * log2(e), there.
            float2 acc[11], bnd[11];
#pragma unroll
            for (int i = 0; i < 11; ++i) acc[i] = make_float2(0.f, 0.f);
            for (int kb = 0; kb + band < nqb; ++kb) {
                const int gb = tile & 1;
                if (!(ok = pg_wait(&bars.st_full[stage], (st_full_bits >> stage) & 1u, abort, status))) break;
                st_full_bits ^= 1u << stage;
                const float* vec = reinterpret_cast<const float*>(sm + stage * PgSmem::st_bytes + PgSmem::st_vec);
                if (kb == 0) {
                    // entry 127 + (distance - 128 band) of the band window
                    const float* bw = vec + 384 + 103 + 64 * half - 32 * quarter + 2 * qq - rho;
#pragma unroll
                    for (int i = 0; i < 11; ++i) bnd[i] = make_float2(bw[8 * i], bw[8 * i + 1]);
                }
                // ea, or a * log2(e), of my four keys; 1 / Z' and -D / Z' (or log2 Z and D) of my
                // 16 queries, in pairs of columns
                float2 zc[8], yc[8];
                const float4 e4 = *reinterpret_cast<const float4*>(vec + 256 + 32 * quarter + 4 * rho);
                const float ek[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 z4 = *reinterpret_cast<const float4*>(vec + 64 * half + 16 * i + 4 * qq);
                    const float4 y4 = *reinterpret_cast<const float4*>(vec + 128 + 64 * half + 16 * i + 4 * qq);
                    zc[2 * i] = make_float2(z4.x, z4.y);
                    zc[2 * i + 1] = make_float2(z4.z, z4.w);
                    yc[2 * i] = make_float2(y4.x, y4.y);
                    yc[2 * i + 1] = make_float2(y4.z, y4.w);
                }
                // the stage's row vectors are in registers: with the MMA's commit, the
                // producer may refill it
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.st_empty[stage]);
                if (!(ok = pg_wait(&bars.g_full[gb], (g_full_bits >> gb) & 1u, abort, status))) break;
                g_full_bits ^= 1u << gb;
                tc_fence_after();
                float2 rs[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) rs[m] = make_float2(0.f, 0.f);
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    uint32_t g[32];
                    tmem_ld_16x256b_x8(lane_base + ((uint32_t)(16 * blk) << 16) + 128 * gb + 64 * half, g);
                    tmem_ld_wait();
                    if (blk == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars.g_free[gb]);
                    }
                    if (exact)
                        pg_block<true>(g, blk, zc, yc, ek, bnd, acc, rs);
                    else
                        pg_block<false>(g, blk, zc, yc, ek, bnd, acc, rs);
                }
                stage = (stage + 1) % kStages;
                ++tile;
                // Row sums over the four lanes of each rho, so that lane qq ends with row
                // rho + 8 qq: the lanes exchange halves of their four sums (xor 1: rows with
                // m % 2 = qq % 2 stay; xor 2: the row m = qq stays), three shuffles.
                const float r0 = rs[0].x + rs[0].y, r1 = rs[1].x + rs[1].y;
                const float r2 = rs[2].x + rs[2].y, r3 = rs[3].x + rs[3].y;
                const bool b0 = (qq & 1) != 0, b1 = (qq & 2) != 0;
                const float ka = (b0 ? r1 : r0) + __shfl_xor_sync(0xffffffffu, b0 ? r0 : r1, 1);   // row b0
                const float kc = (b0 ? r3 : r2) + __shfl_xor_sync(0xffffffffu, b0 ? r2 : r3, 1);   // row b0 + 2
                const float rm = (b1 ? kc : ka) + __shfl_xor_sync(0xffffffffu, b1 ? ka : kc, 2);   // row qq
                const float em = b1 ? (b0 ? ek[3] : ek[2]) : (b0 ? ek[1] : ek[0]);
                p.da_part[(slot_row * 2 + half) * p.Tp + kb * 128 + 32 * quarter + rho + 8 * qq] =
                    exact ? rm : em * rm;
            }
            if (!ok) break;
            // Diagonal sums of the band. My sum acc[pi].s lies at distance (128 band + 64 half -
            // 32 quarter) + col - 31, col = 8 pi + s + dd, dd = 2 qq - rho + 7. In round rd,
            // lanes 8 rd .. 8 rd + 7 (rho = 2 rd + rr) write their 22 sums to row 4 rr + qq of
            // the warp's buffer at column col; then lane c adds up columns c, c + 32, c + 64:
            // for each rho of the round, column col holds an entry in exactly one row, the one
            // with 2 qq = col + rho - 7 - s (mod 8), s = (col + rho - 7) mod 2, when
            // 0 <= col - dd <= 81. Rows in round order: the same sums on every run.
            float s0 = 0.f, s1 = 0.f, s2 = 0.f;
            const int dd = 2 * qq - rho + 7;
#pragma unroll 1
            for (int rd = 0; rd < 4; ++rd) {
                if ((lane >> 3) == rd) {
                    float* row = scr + (lane & 7) * kScrStride + dd;
#pragma unroll
                    for (int i = 0; i < 11; ++i) {
                        const float2 v = exact ? acc[i] : fmul2(acc[i], bnd[i]);
                        row[8 * i] = v.x;
                        row[8 * i + 1] = v.y;
                    }
                }
                __syncwarp();
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int rh = 2 * rd + rr;
#pragma unroll
                    for (int cc = 0; cc < 3; ++cc) {
                        const int col = lane + 32 * cc;
                        const int t0 = col + rh - 7;
                        const int q2 = ((t0 - (t0 & 1)) >> 1) & 3;
                        const int kk = t0 - 2 * q2;
                        const float v = (kk >= 0 && kk <= 81) ? scr[(4 * rr + q2) * kScrStride + col] : 0.f;
                        if (cc == 0) s0 += v;
                        else if (cc == 1) s1 += v;
                        else s2 += v;
                    }
                }
                __syncwarp();
            }
            // two sets of warp sums, by band parity: a warp can reach the next band's end
            // only after every warp has read this band's sums
            float* ws = wsum + (nband & 1) * 8 * kScrCols;
            ws[warp * kScrCols + lane] = s0;
            ws[warp * kScrCols + 32 + lane] = s1;
            ws[warp * kScrCols + 64 + lane] = s2;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.band_sync);
            if (!(ok = mbar_wait(&bars.band_sync, band_ph, abort, status, kStatusTimeout))) break;
            band_ph ^= 1;
            ++nband;
            // entry e = threadIdx.x: distance 128 band + e - 128; warp w holds it in column
            // e - 128 - 64 (w / 4) + 32 (w % 4) + 31. A fixed order over the warps.
            const int e = threadIdx.x;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const int col = e - 128 - 64 * (w >> 2) + 32 * (w & 3) + 31;
                if (col >= 0 && col < kScrCols) sum += ws[w * kScrCols + col];
            }
            p.dr_part[slot_row * 256 + e] = sum;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// 1 / Z'(u) = exp(max a + max r - log Z(u)) from the frozen row of lse (batch
// entry 0: identical for every batch entry), as the layer's backward derives it;
// sets the head's exact-form flag when log Z' < -64.
__device__ __forceinline__ float pg_invz(const float* lse, const float* amax, uint32_t* hflag, int H, int T, int h,
                                         int u, float* lz_out) {
    const float lz = lse[(size_t)h * T + u];
    *lz_out = lz;
    const float sh = lz - amax[h] - amax[H + h];   // log Z'(u)
    if (!(sh >= -64.f)) atomicOr(hflag + h, 2u);
    return expf(fminf(-sh, 80.f));
}

// The row vectors of the tiles, in tile order. 256 threads.
//  * Blocks [0, B F Tp / 64): 64 query rows of slice (b, f), four threads per
//    row, each reading 32 contiguous bytes of o and of dO (a warp reads 1 KB of
//    each): D = sum_c dO_c o_c and -D / Z' (0 past T).
//  * Then ceil(Tp / 256) blocks per frozen head f: log2 Z (+inf past T) and
//    1 / Z' (0 past T) of each query, with the exact-form flag; a * log2(e) and
//    exp(a - max a) of each key, from the layer's padded slices.
__global__ void __launch_bounds__(256)
pg_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
               const float* __restrict__ lse, const __grid_constant__ PgParams p, const float* __restrict__ amax,
               const float* __restrict__ a2p, const float* __restrict__ eap, uint32_t* __restrict__ hflag) {
    grid_dep_wait();
    grid_dep_launch();
    const int per_slice = p.Tp / 64;
    const long long nd = (long long)p.B * p.F * per_slice;
    if ((long long)blockIdx.x < nd) {
        const int slice = (int)(blockIdx.x / (unsigned)per_slice);
        const int i = (int)(blockIdx.x - (unsigned)(slice * per_slice)) * 64 + (threadIdx.x >> 2);
        const int part = threadIdx.x & 3;
        const int b = slice / p.F, f = slice - b * p.F;
        const int h = p.frz_heads[f];
        // log Z(i) and the maxima are loaded with o and dO, not after the dot product
        float lz = 0.f, am = 0.f, rm = 0.f;
        if (part == 0 && i < p.T) {
            lz = lse[(size_t)h * p.T + i];
            am = amax[h];
            rm = amax[p.H + h];
        }
        float d = 0.f;
        if (i < p.T) {
            const size_t row = ((size_t)b * p.H + h) * p.T + i;
            // 4 threads per row, d / 4 elements (d / 32 chunks of 8) each
            const int nc = p.d >> 5;
            const uint4* po = reinterpret_cast<const uint4*>(o + row * p.d) + nc * part;
            const uint4* pd = reinterpret_cast<const uint4*>(dO + row * p.d) + nc * part;
            uint4 xv[4], yv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (c < nc) {
                    xv[c] = __ldg(po + c);
                    yv[c] = __ldg(pd + c);
                }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (c < nc) {
                    const uint32_t xs[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
                    const uint32_t ys[4] = {yv[c].x, yv[c].y, yv[c].z, yv[c].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        d = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), d);
                        d = fmaf(__uint_as_float(xs[e] & 0xffff0000u), __uint_as_float(ys[e] & 0xffff0000u), d);
                    }
                }
        }
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        if (part == 0) {
            // 1 / Z'(i) as pg_invz forms it (the head blocks below raise the exact-form flag)
            const float y = i < p.T ? -d * expf(fminf(-(lz - am - rm), 80.f)) : 0.f;
            const size_t at = (size_t)slice * p.Tp + (i & ~127) + qperm(i & 127);
            p.yx[at] = d;
            p.yf[at] = y;
        }
        return;
    }
    const int per_head = (p.Tp + 255) / 256;
    const int v = (int)((long long)blockIdx.x - nd);
    const int f = v / per_head;
    const int u = (v - f * per_head) * 256 + threadIdx.x;
    if (f >= p.F || u >= p.Tp) return;
    const int h = p.frz_heads[f];
    float l2 = INFINITY, iz = 0.f;
    if (u < p.T) {
        float lz;
        iz = pg_invz(lse, amax, hflag, p.H, p.T, h, u, &lz);
        l2 = lz * kLog2e;
    }
    const size_t row = (size_t)f * p.Tp + (u & ~127);
    p.zx[row + qperm(u & 127)] = l2;
    p.zf[row + qperm(u & 127)] = iz;
    p.ex[row + kperm(u & 127)] = a2p[(size_t)h * p.Tp + u];
    p.ef[row + kperm(u & 127)] = eap[(size_t)h * p.Tp + u];
}

// da[h, x] = sum_b sum_band sum_half da_part[b, f, band, half, x] over the tiles
// that exist (band < nqb - x / 128); dr[h, x] = sum_b of the two bands that hold
// distance x (band x / 128: entry x mod 128 + 128; band x / 128 + 1: entry
// x mod 128). Ordinary heads get zeros.
// Grid (ceil(T / 32), H), 512 threads: 32 keys x 16 groups. Group g = 2 c + half
// adds, for b = 0.. and then band = c, c + 8, ..., the terms of its column half;
// group 0 then adds the sixteen partial sums in group order, and group 1 the dr
// terms in batch order. Every result has the same bits on every run.
__global__ void __launch_bounds__(512)
pg_reduce_kernel(const __grid_constant__ PgParams p, float* __restrict__ da, float* __restrict__ dr) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int kGroups = 16, kPhases = kGroups / 2;
    __shared__ float part[kGroups][32];
    const int h = blockIdx.y;
    const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
    const int x = blockIdx.x * 32 + lane;
    int f = 0;
    while (f < p.F && p.frz_heads[f] != h) ++f;
    if (f == p.F) {   // ordinary head
        if (grp == 0 && x < p.T) {
            da[(size_t)h * p.T + x] = 0.f;
            dr[(size_t)h * p.T + x] = 0.f;
        }
        return;
    }
    const int xb = (blockIdx.x * 32) >> 7, xr = x & 127;
    const int nb = p.nqb - xb;   // bands whose tiles hold key block xb
    float sa = 0.f;
    if (x < p.T && (grp >> 1) < nb) {
        // the group's terms in order, eight loads in flight at a time (past the last
        // term they read nothing and add +0)
        const size_t stride_band = 2 * (size_t)p.Tp, stride_b = (size_t)p.F * p.nqb * stride_band;
        const float* base = p.da_part + (size_t)f * p.nqb * stride_band + (grp & 1) * (size_t)p.Tp + x;
        int b = 0, band = grp >> 1;
        while (b < p.B) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool in = b < p.B;
                v[u] = in ? base[b * stride_b + band * stride_band] : 0.f;
                if (in && (band += kPhases) >= nb) {
                    band = grp >> 1;
                    ++b;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) sa += v[u];
        }
    }
    part[grp][lane] = sa;
    __syncthreads();
    if (x >= p.T) return;
    if (grp == 0) {
        float t = part[0][lane];
#pragma unroll
        for (int g = 1; g < kGroups; ++g) t += part[g][lane];
        da[(size_t)h * p.T + x] = t;
    } else if (grp == 1) {
        float sr = 0.f;
        for (int b = 0; b < p.B; ++b) {
            const size_t rows = ((size_t)b * p.F + f) * p.nqb;
            sr += p.dr_part[(rows + xb) * 256 + xr + 128];
            if (xb + 1 < p.nqb) sr += p.dr_part[(rows + xb + 1) * 256 + xr];
        }
        dr[(size_t)h * p.T + x] = sr;
    }
}

// Workspace: the layer's forward regions (status words, flags, maxima, padded
// slices), then the row vectors in tile order and the per-item slots.
struct PgLayout {
    size_t yx, yf, zx, zf, ex, ef, da_part, dr_part, total;
};
PgLayout pg_layout(int B, int H, int F, int T) {
    const size_t Tp = (size_t)(T + 127) / 128 * 128;
    const size_t nqb = Tp / 128;
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    PgLayout L;
    size_t off = up(workspace_layout(0, H, T, 0, 1).total);
    L.yx = off;
    off = up(off + (size_t)B * F * Tp * sizeof(float));
    L.yf = off;
    off = up(off + (size_t)B * F * Tp * sizeof(float));
    L.zx = off;
    off = up(off + (size_t)F * Tp * sizeof(float));
    L.zf = off;
    off = up(off + (size_t)F * Tp * sizeof(float));
    L.ex = off;
    off = up(off + (size_t)F * Tp * sizeof(float));
    L.ef = off;
    off = up(off + (size_t)F * Tp * sizeof(float));
    L.da_part = off;
    off = up(off + (size_t)B * F * nqb * 2 * Tp * sizeof(float));
    L.dr_part = off;
    off = up(off + (size_t)B * F * nqb * 256 * sizeof(float));
    L.total = off;
    return L;
}

}  // namespace
}  // namespace saf

using namespace saf;

extern "C" size_t saf_pattern_grad_tc_workspace_bytes(int B, int H, int T, int n_frozen) {
    if (B < 0 || H <= 0 || H > SAF_MAX_HEADS || T < 0 || n_frozen < 0 || n_frozen > H) return 0;
    return pg_layout(B, H, n_frozen, T).total;
}

extern "C" int saf_pattern_grad_tc(const void* v, const void* dO, const void* o, const float* lse, const float* a,
                                   const float* r, int ld_prior, const uint8_t* frozen, int B, int H, int T, int d,
                                   float* da, float* dr, void* workspace, size_t ws_bytes, void* stream) {
    if (B < 0 || H <= 0 || H > SAF_MAX_HEADS || T < 0) return SAF_EINVAL;
    if (d != 64 && d != 96 && d != 128) return SAF_EUNSUPPORTED;
    if ((long long)B * H * T * d > (1ll << 40)) return SAF_EINVAL;
    if (!da || !dr) return SAF_EINVAL;
    if (((uintptr_t)da & 3u) || ((uintptr_t)dr & 3u)) return SAF_EALIGN;
    PgParams p;
    memset(&p, 0, sizeof(p));
    HeadMask mask;
    memset(&mask, 0, sizeof(mask));
    int F = 0;
    for (int h = 0; h < H; ++h)
        if (frozen && frozen[h]) {
            mask.w[h >> 6] |= 1ull << (h & 63);
            p.frz_heads[F++] = (uint8_t)h;
        }
    if (T == 0) return SAF_OK;
    // every argument and the device are checked before the first work is enqueued
    const bool work = B > 0 && F > 0;
    const PgLayout L = pg_layout(B, H, F, T);
    if (work) {
        if (!v || !dO || !o || !lse || !a || !r || ld_prior < T) return SAF_EINVAL;
        if (((uintptr_t)v | (uintptr_t)dO | (uintptr_t)o | (uintptr_t)lse) & 15u) return SAF_EALIGN;
        if (((uintptr_t)a | (uintptr_t)r) & 3u) return SAF_EALIGN;
        if (!workspace) return SAF_EWORKSPACE;
        if ((uintptr_t)workspace & 255u) return SAF_EALIGN;
        if (ws_bytes < L.total) return SAF_EWORKSPACE;
    }
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        return SAF_ECUDA;
    }
    if (!(prop.major == 10 && prop.minor == 3)) return SAF_EUNSUPPORTED;
    const int sms = prop.multiProcessorCount;
    cudaStream_t s = (cudaStream_t)stream;
    if (!work) {
        if (cudaMemsetAsync(da, 0, (size_t)H * T * sizeof(float), s) != cudaSuccess ||
            cudaMemsetAsync(dr, 0, (size_t)H * T * sizeof(float), s) != cudaSuccess) {
            cudaGetLastError();
            return SAF_ELAUNCH;
        }
        return SAF_OK;
    }

    const WorkspaceLayout W = workspace_layout(0, H, T, 0, 1);
    char* ws = (char*)workspace;
    LayerArgs la;
    memset(&la, 0, sizeof(la));
    la.v = v;
    la.dO = dO;
    la.o = o;
    la.lse = lse;
    la.a = a;
    la.r = r;
    la.ld_prior = ld_prior;
    la.B = B;
    la.H = H;
    la.Hkv = H;
    la.T = T;
    la.d = d;
    la.mask = mask;
    la.status = (uint32_t*)(ws + W.status);
    la.hflag = (uint32_t*)(ws + W.hflag);
    la.amax = (float*)(ws + W.amax);
    la.a2p = (float*)(ws + W.a2p);
    la.r2p = (float*)(ws + W.r2p);
    la.eap = (float*)(ws + W.eap);
    la.erp = (float*)(ws + W.erp);

    const int BH = B * H;
    if (!make_tmap_bf16_3d(&p.tm_v, v, d, T, BH, 64, 128) || !make_tmap_bf16_3d(&p.tm_do, dO, d, T, BH, 64, 128))
        return SAF_ELAUNCH;
    p.yx = (float*)(ws + L.yx);
    p.yf = (float*)(ws + L.yf);
    p.zx = (float*)(ws + L.zx);
    p.zf = (float*)(ws + L.zf);
    p.ex = (float*)(ws + L.ex);
    p.ef = (float*)(ws + L.ef);
    p.r2p = la.r2p;
    p.erp = la.erp;
    p.hflag = la.hflag;
    p.da_part = (float*)(ws + L.da_part);
    p.dr_part = (float*)(ws + L.dr_part);
    p.status = la.status;
    p.B = B;
    p.H = H;
    p.T = T;
    p.nqb = (T + 127) / 128;
    p.Tp = p.nqb * 128;
    p.F = F;
    p.n_items = B * F * p.nqb;
    p.d = d;

    trace_begin(SAF_KERNEL_PATTERN_GRAD, s);
    cudaError_t e = launch_call_init(la, true, false, s);
    if (e == cudaSuccess) {
        note_launch();
        const long long blocks = (long long)B * F * (p.Tp / 64) + (long long)F * ((p.Tp + 255) / 256);
        e = launch_ex(pg_prep_kernel, dim3((unsigned)blocks), dim3(256), 0, s, true, 1,
                      (const __nv_bfloat16*)o, (const __nv_bfloat16*)dO, lse, p, (const float*)la.amax,
                      (const float*)la.a2p, (const float*)la.eap, la.hflag);
    }
    const bool wide = d > 64;
    const int smem = (wide ? PgSmem<128>::total : PgSmem<64>::total) + 1024;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(wide ? pg_tc_kernel<128> : pg_tc_kernel<64>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) {
        note_launch();
        e = launch_ex(wide ? pg_tc_kernel<128> : pg_tc_kernel<64>, dim3((unsigned)(p.n_items < sms ? p.n_items : sms)),
                      dim3(kThreads), (size_t)smem, s, true, 1, p);
    }
    if (e == cudaSuccess) {
        note_launch();
        e = launch_ex(pg_reduce_kernel, dim3((unsigned)((T + 31) / 32), (unsigned)H), dim3(512), 0, s, true, 1, p,
                      da, dr);
    }
    after_launch(SAF_KERNEL_PATTERN_GRAD, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SAF_ELAUNCH;
    }
    return SAF_OK;
}
