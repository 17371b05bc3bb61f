/*
 * saf.h - C ABI of the hybrid causal-attention layer of Selective Attention
 * Freezing (SAF), forward and backward, on one NVIDIA GB300 (sm_103a).
 *
 * Source: "When Can Attention Heads Be Statically Defined?" (arXiv 2609.34650).
 *
 *   Ordinary head (App. A.1, Eqs. 5-7):
 *       S = Q K^T / sqrt(d),  A = softmax_causal(S),  O = A V.
 *   Frozen head (§3.2, Eq. 3; §3.3 "Fused computation"):
 *       W(i, j) = exp(a[j] + r[i - j]) / Z(i) for j <= i, 0 for j > i,
 *       Z(i)    = sum_{k <= i} exp(a[k] + r[i - k]),        O = W V.
 *     The pattern never looks at Q or K. Its backward pass is only
 *     dV = W^T dO (§3.3, App. D.2); a frozen head has no query/key slot, so
 *     its dQ and dK are zero, and a, r and the normalisers take no gradient.
 *   Both kinds of head run in one fused launch per pass and write their
 *   outputs in the original head order (App. D.2).
 *
 * Indexing is 0-based: the paper's alpha(j) (keys 1..T) is a[j-1] and its
 * rho(delta) (offsets 0..T-1) is r[delta].
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors q, k, v, o, dO, dq, dk, dv have layout [B, H, T, d], contiguous,
 *    element type `dt` (bf16 or fp32). lse and the normalisers are fp32.
 *    d = 64, 96 or 128. SAF_BF16 runs on tensor-core kernels, SAF_FP32 on
 *    CUDA-core kernels, for the multi-head and grouped-query layouts, with
 *    per-call or prepared normalisers. Other values return SAF_EUNSUPPORTED.
 *    Every tensor pointer must be 16-byte aligned (SAF_EALIGN otherwise).
 *  - a, r: fp32 [H, ld_prior] device arrays, ld_prior >= T; row h holds the
 *    absolute-key preference a and the relative-distance preference r of
 *    head h. Only a[h, 0..T-1], r[h, 0..T-1] of frozen heads are read, so a
 *    stored prior longer than T may be passed (App. D.2 tests prior length
 *    192 at T = 129). a and r may be NULL when no head is frozen.
 *  - frozen: HOST array of H bytes, nonzero = frozen head. NULL means no
 *    frozen head. H <= SAF_MAX_HEADS.
 *  - q and k of frozen heads are never read (they may hold anything,
 *    including NaN); q and k may be NULL only when every head is frozen.
 *  - workspace: caller-owned DEVICE scratch of at least
 *    saf_attn_workspace_bytes(...) bytes, 256-byte aligned. The library
 *    allocates no memory and keeps no state across calls other than cached
 *    device attributes, CUDA function attributes, a launch counter and the
 *    optional trace hook below. Calls that share a workspace must be
 *    ordered on one stream.
 *  - stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All device work is enqueued on it; no entry point synchronises except
 *    saf_device_status.
 *  - Return value: SAF_OK (0) or a negative saf_status_t. Argument, shape,
 *    alignment and device errors are returned synchronously before any
 *    work is enqueued. An error raised while kernels run (a bounded device
 *    wait that expired) is recorded in the workspace and reported by
 *    saf_device_status.
 *  - T == 0 or B == 0 is a valid empty call: nothing is launched.
 */
#ifndef SAF_H_
#define SAF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SAF_MAX_HEADS 256

#if defined(__GNUC__)
#define SAF_API __attribute__((visibility("default")))
#else
#define SAF_API
#endif

typedef enum { SAF_BF16 = 0, SAF_FP32 = 1 } saf_dtype_t;

typedef enum {
    SAF_OK = 0,
    SAF_EINVAL = -1,        /* null pointer, bad shape, ld_prior < T, H > SAF_MAX_HEADS   */
    SAF_EALIGN = -2,        /* a tensor or the workspace is not aligned                   */
    SAF_EUNSUPPORTED = -3,  /* device is not sm_103, or d / dtype not supported          */
    SAF_ELAUNCH = -4,       /* a kernel launch or an async CUDA call failed               */
    SAF_EWORKSPACE = -5,    /* workspace NULL or smaller than saf_attn_workspace_bytes    */
    SAF_ETIMEOUT = -6,      /* a bounded device wait expired (from saf_device_status)    */
    SAF_ECUDA = -8,         /* a CUDA runtime query failed (no device, driver error)    */
    SAF_ESCRATCH = -9       /* saf_attn_fwd_noalloc: the problem needs more workspace
                               than its fixed device scratch holds                     */
} saf_status_t;

/* Bytes of device workspace that saf_attn_fwd (backward = 0) or
 * saf_attn_bwd (backward = 1) needs for these sizes. Returns 0 for an
 * invalid size. */
SAF_API size_t saf_attn_workspace_bytes(int B, int H, int T, int d, saf_dtype_t dt, int backward);

/* Forward pass of the hybrid layer.
 *
 * In:  q, k, v [B,H,T,d] (dt); a, r [H, ld_prior] fp32; frozen [H] host bytes.
 * Out: o [B,H,T,d] (dt): ordinary heads A V (Eqs. 5-7), frozen heads W V
 *      (Eq. 3); lse [B,H,T] fp32: for ordinary rows the natural-log
 *      normaliser of the scaled scores, m_i + log sum_j exp(S_ij - m_i); for
 *      frozen rows log Z(i). saf_attn_bwd consumes lse.
 * The normalisers log Z of the frozen heads are computed here ("precomputed
 * normalisers", §3.3), once per head, independent of the batch.
 * Supported: d in {64, 96, 128}; SAF_BF16 on the tensor cores with fp32
 * accumulation (App. C.5's 1B model has d_h = 96), SAF_FP32 in fp32 arithmetic
 * throughout on CUDA cores. */
SAF_API int saf_attn_fwd(const void* q, const void* k, const void* v,
                 const float* a, const float* r, int ld_prior, const uint8_t* frozen,
                 int B, int H, int T, int d, saf_dtype_t dt,
                 void* o, float* lse,
                 void* workspace, size_t ws_bytes, void* stream);

/* Forward pass for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot hand the library a workspace: code that runs where
 * cudaMalloc is not allowed (for example inside a framework that owns every
 * allocation and passes plugins only their input and output buffers, or in
 * a context where allocating could deadlock or fragment a caching
 * allocator). It computes exactly what saf_attn_fwd computes, with the same
 * kernels, arguments and outputs, but takes its workspace from a fixed
 * array of 8 MiB in device memory that the library declares statically;
 * every GPU that loads the library holds that array until the process
 * exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *  - Size limit: saf_attn_workspace_bytes(B, H, T, d, dt, 0) must be at most
 *    8 MiB: about H * T <= 340,000 for SAF_BF16 (for example 12 heads of
 *    16,384 tokens) and H * T <= 2,000,000 for SAF_FP32, independent of B;
 *    larger problems return SAF_ESCRATCH and enqueue nothing.
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress, with that device current) and caches
 *    it. Make that first call before any stream capture begins. The cached
 *    address belongs to the device's primary context: after
 *    cudaDeviceReset (or anything else that ends that context) it is stale,
 *    so a process that resets a device must not call this entry point on
 *    that device again.
 *  - Sharing: every call on a device uses the same array, which keeps the
 *    contents the last call left. Each call's first kernel clears the parts
 *    that must start at zero before anything reads them. Calls whose work overlaps on the
 *    GPU (two streams, or two host threads) race on the array: order them
 *    on one stream.
 *  - Device-side status words live in that array and are not reported;
 *    callers that need saf_device_status use saf_attn_fwd with a workspace. */
SAF_API int saf_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                 const float* a, const float* r, int ld_prior, const uint8_t* frozen,
                                 int B, int H, int T, int d, saf_dtype_t dt,
                                 void* o, float* lse, void* stream);

/* Backward pass of the hybrid layer, given dO = dL/dO.
 *
 * In:  q, k, v, o, dO [B,H,T,d] (dt), lse [B,H,T] from saf_attn_fwd with the
 *      same inputs; a, r, frozen as in saf_attn_fwd.
 * Out: dq, dk, dv [B,H,T,d] (dt). Ordinary heads: the gradient of Eqs. 5-7.
 *      Frozen heads: dv = W^T dO; dq and dk are written as exact zeros
 *      (§3.3, App. D.2).
 * Supported: d in {64, 96, 128} for both types. */
SAF_API int saf_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, const float* a, const float* r, int ld_prior,
                 const uint8_t* frozen, int B, int H, int T, int d, saf_dtype_t dt,
                 void* dq, void* dk, void* dv,
                 void* workspace, size_t ws_bytes, void* stream);

/* Grouped-query forward pass (§3.3: the grouped-query path keeps the shared
 * key and value projections and drops the replaced heads' query projections;
 * App. C.6: Qwen3-4B shares 8 key/value heads among 32 query heads; App. D.2:
 * each ordinary query head is mapped to its retained key/value group).
 *
 * Same as saf_attn_fwd, except that k and v have Hkv heads:
 * In:  q [B,H,T,d], k, v [B,Hkv,T,d] (dt), H a multiple of Hkv; query head h
 *      reads key/value head h / (H / Hkv). a, r, frozen are per query head
 *      ([H, ld_prior], H bytes): a frozen query head applies its own Eq. 3
 *      pattern to the values of its group and reads no q or k.
 * Out: o [B,H,T,d], lse [B,H,T] as for saf_attn_fwd.
 * Workspace: saf_attn_workspace_bytes(B, H, T, d, dt, 0) (query heads).
 * Errors: as saf_attn_fwd; SAF_EINVAL also for Hkv <= 0 or H % Hkv != 0.
 * saf_attn_fwd(...) equals saf_attn_fwd_gqa(..., Hkv = H, ...). */
SAF_API int saf_attn_fwd_gqa(const void* q, const void* k, const void* v,
                     const float* a, const float* r, int ld_prior, const uint8_t* frozen,
                     int B, int H, int Hkv, int T, int d, saf_dtype_t dt,
                     void* o, float* lse,
                     void* workspace, size_t ws_bytes, void* stream);

/* Grouped-query backward pass (§3.3, App. C.6, App. D.2), given dO.
 *
 * In:  q, o, dO [B,H,T,d]; k, v [B,Hkv,T,d]; lse [B,H,T] from
 *      saf_attn_fwd_gqa with the same inputs; a, r, frozen per query head.
 * Out: dq [B,H,T,d]: the gradient of Eqs. 5-7 for ordinary query heads,
 *      exact zeros for frozen ones. dk, dv [B,Hkv,T,d]: the gradient of a
 *      shared head is the sum over the query heads of its group; frozen query
 *      heads add W^T dO to dv only, so a group with no ordinary query head
 *      gets dk = 0 exactly.
 * Workspace: saf_attn_workspace_bytes(B, H, T, d, dt, 1).
 * Errors: as saf_attn_bwd; SAF_EINVAL also for Hkv <= 0 or H % Hkv != 0.
 * saf_attn_bwd(...) equals saf_attn_bwd_gqa(..., Hkv = H, ...). */
SAF_API int saf_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, const float* a, const float* r, int ld_prior,
                     const uint8_t* frozen, int B, int H, int Hkv, int T, int d, saf_dtype_t dt,
                     void* dq, void* dk, void* dv,
                     void* workspace, size_t ws_bytes, void* stream);

/* ---- Prepared frozen-pattern state -------------------------------------------
 * A frozen head's pattern depends on a and r alone (§3.2, Eq. 3), so its
 * normalisers can be computed once and kept: the paper's persistent state per
 * replaced head is alpha, rho, the normalisers and a small relative-distance
 * band (§3.3 "precomputed normalisers"; App. D.2). saf_attn_fwd / saf_attn_bwd
 * recompute them in every call; the calls below take them from a state that
 * saf_frozen_prepare filled once for fixed (a, r).
 *
 * saf_frozen_state_bytes: bytes of DEVICE state for H heads of length T
 * (0 for invalid sizes). It does not depend on B.
 *
 * saf_frozen_prepare: fills `state` (caller-owned, 256-byte aligned) for the
 * frozen heads of `frozen` from a, r [H, ld_prior]. Enqueued on `stream`.
 * Prepare again after a or r change (the trainable variant of App. C.3.2
 * refreshes its normalisers after each update).
 *
 * saf_attn_fwd_prepared / saf_attn_bwd_prepared: saf_attn_fwd_gqa /
 * saf_attn_bwd_gqa (Hkv = H for the multi-head layer) with the frozen-pattern
 * data read from `state`. a, r, ld_prior and frozen must be the ones the state
 * was prepared with (the fp32 path still reads a and r). `workspace` is the
 * per-call workspace of saf_attn_workspace_bytes. Calls may share one state
 * while nothing prepares it again. Results equal those of the unprepared
 * calls up to rounding (the forward's exactly). Errors as the unprepared
 * calls, and SAF_EWORKSPACE for a NULL state. */
SAF_API size_t saf_frozen_state_bytes(int H, int T, saf_dtype_t dt);
SAF_API int saf_frozen_prepare(const float* a, const float* r, int ld_prior, const uint8_t* frozen, int H, int T,
                               saf_dtype_t dt, void* state, size_t state_bytes, void* stream);
SAF_API int saf_attn_fwd_prepared(const void* q, const void* k, const void* v, const float* a, const float* r,
                                  int ld_prior, const uint8_t* frozen, const void* state, int B, int H, int Hkv,
                                  int T, int d, saf_dtype_t dt, void* o, float* lse, void* workspace,
                                  size_t ws_bytes, void* stream);
SAF_API int saf_attn_bwd_prepared(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                  const float* lse, const float* a, const float* r, int ld_prior,
                                  const uint8_t* frozen, const void* state, int B, int H, int Hkv, int T, int d,
                                  saf_dtype_t dt, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                  void* stream);

/* Diagnostic forward pass for testing failure detection (the paper has no
 * counterpart; it exercises this library's bounded waits).
 *
 * Every wait inside the tensor-core kernels is bounded: when it expires, the
 * kernel records SAF_ETIMEOUT in the workspace's error word, its other warps
 * give up too, it frees its tensor memory and returns, so the CUDA context
 * stays usable. This entry point makes that happen on purpose, without any
 * fault: it is saf_attn_fwd (SAF_BF16 only, else SAF_EUNSUPPORTED) with
 *  - withhold = 1: the forward kernel's producer publishes no work item, so
 *    every other role's first wait expires (o and lse are not written);
 *    withhold = 0 runs the normal pass;
 *  - wait_limit_us: the limit of every bounded wait in the forward kernel,
 *    in microseconds (0: the default of 2 s). A wait ends at most one
 *    suspend interval (about 10 ms) after its limit.
 * The next saf_device_status on `workspace` reports SAF_ETIMEOUT after a
 * withheld call; the next normal call clears the word. */
SAF_API int saf_attn_fwd_diag(const void* q, const void* k, const void* v,
                              const float* a, const float* r, int ld_prior, const uint8_t* frozen,
                              int B, int H, int T, int d, saf_dtype_t dt,
                              void* o, float* lse,
                              void* workspace, size_t ws_bytes, void* stream,
                              int withhold, unsigned wait_limit_us);

/* Waits for `stream`, then reads the error word that the kernels of the last
 * call on `workspace` left there. Returns SAF_OK, SAF_ETIMEOUT, or
 * SAF_ECUDA if the stream reported a CUDA error. */
SAF_API int saf_device_status(const void* workspace, void* stream);

/* Static, human-readable text for a status code. Never NULL. */
SAF_API const char* saf_error_string(int status);

/* ABI version of this library (major * 100 + minor). */
SAF_API int saf_version(void);

/* ---- Compact fitting of a frozen pattern -----------------------------------
 * Fits a, r of Eq. 3 to a target pattern P, given only P's sufficient
 * statistics (§3.2 "Fitting", Eq. 4; App. D.1, Eq. 20):
 *   eta_abs(j)   = sum_{i >= j} P(i, j)          (key-column sums)
 *   eta_rel(d)   = sum_{i - d >= 0} P(i, i - d)  (diagonal sums)
 * It starts from a = 0, r(d) = log max(eta_rel(d) / (T - d), 1e-9) and takes
 * `steps` Adam steps (moment decays 0.9 and 0.999, epsilon 1e-8, bias-corrected)
 * at learning rate `lr` on
 *   L(a, r) = (1/T) [sum_i log Z(i) - sum_j eta_abs(j) a(j) - sum_d eta_rel(d) r(d)],
 * whose gradient is the fitted pattern's marginals minus the target's, over T.
 * The paper's settings are steps = 400, lr = 0.05 (App. C.1).
 *
 * In:  eta_abs, eta_rel: DEVICE fp32 [H, T] (row h: head h); H <= SAF_MAX_HEADS.
 * Out: a, r: DEVICE fp32 [H, T], the fitted parameters (row stride T, ready to
 *      pass to saf_attn_fwd with ld_prior = T); loss: DEVICE fp32 [H], L at the
 *      result. The paper's acceptance statistic kappa (mean KL per row of the
 *      target from the fit) is loss[h] + (1/T) sum P log P of the target
 *      (saf_fit_target_stats computes that term; saf_fit_from_target runs the
 *      whole path); a fit passes when kappa <= 0.2.
 * workspace: DEVICE scratch of saf_fit_workspace_bytes(H, T) bytes, 256-byte
 * aligned. fp32 pointers must be 4-byte aligned. Work is enqueued on `stream`;
 * errors in the arguments return before any work is enqueued. */
SAF_API size_t saf_fit_workspace_bytes(int H, int T);
SAF_API int saf_fit_compact(const float* eta_abs, const float* eta_rel, int H, int T, int steps, float lr,
                            float* a, float* r, float* loss, void* workspace, size_t ws_bytes, void* stream);

/* ---- From a measured target to accept / reject ------------------------------
 * The selection algorithm's target steps (§3.2 "Fitting"; App. A.2; App. C.1):
 * the measured mean attention matrix A of a head has its causal entries
 * floored at 1e-9 and every row normalised, P = floor-and-normalise(A); Eq. 4
 * needs only P's key-column sums eta_abs(j) = sum_{i >= j} P(i, j) and diagonal
 * sums eta_rel(d) = sum_{i >= d} P(i, i - d); a fitted head is accepted when
 * kappa = (1/T) sum_i KL(P(i, .) || W(i, .)) <= 0.2 nats (App. C.1). Since
 * kappa = (1/T) sum_i sum_j P log P + L(a, r) with L the Eq. 4 loss, the
 * target's negative entropy per row, negent = (1/T) sum P log P, completes it.
 *
 * saf_fit_target_stats
 * In:  A: DEVICE fp32 [H, T, T] row-major; entries above the diagonal are not
 *      read. P is never stored.
 * Out: eta_abs, eta_rel: DEVICE fp32 [H, T]; negent: DEVICE fp32 [H].
 * Sums run in a fixed order: results are the same on every run.
 * workspace: DEVICE scratch of saf_fit_stats_workspace_bytes(H, T) bytes,
 * 256-byte aligned. Errors: SAF_EINVAL (sizes, NULL), SAF_EALIGN, SAF_EWORKSPACE,
 * SAF_EUNSUPPORTED (device), all before any work is enqueued.
 *
 * saf_fit_from_target: the whole path on the device: the statistics above,
 * saf_fit_compact's `steps` Adam steps at rate `lr`, then kappa.
 * Out: a, r: DEVICE fp32 [H, T] (the fitted pattern); kappa: DEVICE fp32 [H];
 *      accept: DEVICE uint8 [H], 1 when kappa <= tol (the paper: 0.2).
 * workspace: saf_fit_from_target_workspace_bytes(H, T) bytes, 256-byte aligned.
 * Errors as above, and SAF_EINVAL for steps < 0, lr <= 0 or tol < 0. */
SAF_API size_t saf_fit_stats_workspace_bytes(int H, int T);
SAF_API int saf_fit_target_stats(const float* A, int H, int T, float* eta_abs, float* eta_rel, float* negent,
                                 void* workspace, size_t ws_bytes, void* stream);
SAF_API size_t saf_fit_from_target_workspace_bytes(int H, int T);
SAF_API int saf_fit_from_target(const float* A, int H, int T, int steps, float lr, float tol, float* a, float* r,
                                float* kappa, uint8_t* accept, void* workspace, size_t ws_bytes, void* stream);

/* ---- Gradients of trainable patterns ---------------------------------------
 * For the variant whose patterns keep training (App. C.3.2): the gradients of
 * the loss with respect to a and r of every frozen head, given the forward
 * output and the output gradient. Eq. 3 is a row softmax of the logits
 * a(j) + r(i - j); with G(i, j) = dO_i . V_j and D_i = dO_i . O_i,
 *   dL(i, j) = W(i, j) (G(i, j) - D_i),
 *   da(j) = sum_b sum_{i >= j} dL(i, j),   dr(d) = sum_b sum_{i >= d} dL(i, i - d).
 *
 * In:  v, dO, o [B, H, T, d] (dt, d = 64, 96 or 128), lse [B, H, T] as
 *      saf_attn_fwd wrote it (the frozen rows hold log Z), a, r, ld_prior,
 *      frozen as for saf_attn_fwd.
 * Out: da, dr: DEVICE fp32 [H, T]; rows of ordinary heads are zero. They are
 *      overwritten (cleared on `stream` first).
 * fp32 arithmetic on CUDA cores; the additions into da and dr are atomic, so
 * their last bits vary from run to run. No workspace. */
SAF_API int saf_pattern_grad(const void* v, const void* dO, const void* o, const float* lse, const float* a,
                             const float* r, int ld_prior, const uint8_t* frozen, int B, int H, int T, int d,
                             saf_dtype_t dt, float* da, float* dr, void* stream);

/* The same gradients on the tensor cores (bf16 inputs, d = 64, 96 or 128), with
 * sums in a fixed order: the results have the same bits on every run.
 * G^T = V dO^T is formed per causal 128 x 128 tile with tcgen05 MMAs (fp32 in
 * tensor memory); W is rebuilt from a, r and the log Z rows of lse in the form
 * the layer's backward uses (factorised, or exact when a head's log Z' falls
 * below -64); tiles are visited band by band (band = query block - key block),
 * each thread summing its elements of one distance i - j over the band in
 * registers, and the per-tile key sums and per-band distance sums are written
 * to the workspace and added up by a last kernel.
 * In:  v, dO, o [B, H, T, d] bf16, 16-byte aligned; lse [B, H, T] fp32 as
 *      saf_attn_fwd wrote it; a, r, ld_prior, frozen as for saf_attn_fwd.
 * Out: da, dr: DEVICE fp32 [H, T], overwritten; rows of ordinary heads zero.
 * workspace: DEVICE scratch of saf_pattern_grad_tc_workspace_bytes(B, H, T,
 * n_frozen) bytes (n_frozen = number of nonzero entries of `frozen`), 256-byte
 * aligned; clobbered. Its first 256 bytes are the status words that
 * saf_device_status reads after the call (SAF_ETIMEOUT when a bounded
 * wait of the kernel expired).
 * Errors: SAF_EINVAL (sizes, NULL), SAF_EALIGN, SAF_EWORKSPACE,
 * SAF_EUNSUPPORTED (d not 64, 96 or 128; device), all before any work is
 * enqueued; SAF_ELAUNCH. saf_pattern_grad_tc_workspace_bytes returns 0 for
 * invalid sizes. */
SAF_API size_t saf_pattern_grad_tc_workspace_bytes(int B, int H, int T, int n_frozen);
SAF_API int saf_pattern_grad_tc(const void* v, const void* dO, const void* o, const float* lse, const float* a,
                                const float* r, int ld_prior, const uint8_t* frozen, int B, int H, int T, int d,
                                float* da, float* dr, void* workspace, size_t ws_bytes, void* stream);

/* ---- Profiling hooks (not part of the layer's arithmetic) ----------------
 * Kernel identifiers for saf_set_trace_events. */
typedef enum {
    SAF_KERNEL_NONE = 0,
    SAF_KERNEL_LOGNORM = 1,     /* forward: init kernel, log Z of frozen heads  */
    SAF_KERNEL_FWD = 2,         /* fused forward (both kinds of head)           */
    SAF_KERNEL_BWD_DELTA = 3,   /* D_i = sum_c dO_ic O_ic (bf16: also the row   *
                                 * vectors, dQ accumulator zeroing and 1 / Z')  */
    SAF_KERNEL_BWD_KV = 4,      /* backward key-block pass (dV, dK)            */
    SAF_KERNEL_BWD_Q = 5,       /* backward query-block pass (dQ)              */
    SAF_KERNEL_BWD = 6,         /* fused backward (dQ, dK, dV in one launch)   */
    SAF_KERNEL_DQ_FINISH = 7,   /* dQ accumulator -> dq (scale, dtype, zeros)  */
    SAF_KERNEL_PATTERN_PREP = 8, /* backward: init kernel (clears the status   *
                                  * words; maxima and padded a, r slices)       */
    SAF_KERNEL_PATTERN_GRAD = 9  /* saf_pattern_grad_tc: all of its launches    */
} saf_kernel_t;

/* From the next call on, record `start` (a cudaEvent_t as void*) on the
 * call's stream right before the launches that `kernel` names, and `stop`
 * right after them. Each kernel id has its own pair; NULL events switch that id
 * off, SAF_KERNEL_NONE switches every id off. The hook is process-wide and
 * not thread-safe; it is meant for benchmarks. Returns SAF_OK or
 * SAF_EINVAL for an unknown id. */
SAF_API int saf_set_trace_events(int kernel, void* start, void* stop);

/* Number of kernels this library has launched since it was loaded
 * (host-side counter, all devices and streams). */
SAF_API unsigned long long saf_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SAF_H_ */
