"""Plain fp64 reference for the hybrid causal-attention layer of Selective
Attention Freezing (SAF).

TEST INFRASTRUCTURE ONLY: called by tests/, by __graft_entry__.smoke() and by
bench.py's CPU-baseline leg; never by the library. It is deliberately slow
and literal: dense matrices, one exp per element, NumPy matmuls.

Source: "When Can Attention Heads Be Statically Defined?" (arXiv 2609.34650).

* Ordinary heads (App. A.1, Eqs. 5-7): S = Q K^T / sqrt(d_h),
  A = softmax_causal(S), Z = A V. softmax_causal masks keys j > i and
  normalises each query row.
* Frozen heads (§3.2, Eq. 3): P(i, j) = exp(alpha(j) + rho(i - j)) / Z(i) for
  j <= i, else 0, with Z(i) = sum_{k <= i} exp(alpha(k) + rho(i - k)). The head
  output is P V (§3, "the head output"). The pattern does not look at Q or K.
* Backward of a frozen head (§3.3 "Fused computation", App. D.2): only
  dV = P^T dZ; alpha, rho and the normalisers receive no gradient (§3.3), and
  a frozen head has no query/key slot, so dQ = dK = 0.
* Backward of an ordinary head: the gradient of Eqs. 5-7 by the chain rule,
  dV = A^T dO, dP = dO V^T, D_i = sum_j A_ij dP_ij, dS = A o (dP - D),
  dQ = dS K / sqrt(d_h), dK = dS^T Q / sqrt(d_h).

Indexing: the paper is 1-based (alpha over keys 1..T, rho over offsets
0..T-1). Here everything is 0-based: alpha(j) -> a[j], rho(delta) -> r[delta],
and Z(i) sums over j = 0..i. a and r may be longer than T (a stored prior of
length >= T, App. D.2 tests prior length 192 with T = 129); only their first
T entries are used.

lse: for ordinary rows the natural-log normaliser of the scaled scores,
m_i + log sum_j exp(S_ij - m_i); for frozen rows log Z(i).

Row blocking: every quantity except dV and dK is local to one query row, so
the functions below process query rows in blocks to bound memory at large T.
dV and dK sum over query rows; blocking only changes the order of that sum.

Trainable patterns (App. C.3.2: the trainable variant "computes pattern
gradients and refreshes the normalisers after each update"): Eq. 3 is a row
softmax of the logits L(i, j) = alpha(j) + rho(i - j), so the gradient of the
loss with respect to those logits is the softmax Jacobian applied to
G = dZ V^T, dL(i, j) = P(i, j) (G(i, j) - D_i) with D_i = sum_j P(i, j) G(i, j),
and alpha(j) collects column j, rho(delta) the diagonal i - j = delta.
"""
from __future__ import annotations

import concurrent.futures as _cf
import math

import numpy as np

_NEG_INF = -np.inf


def _as64(x):
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Frozen-head pattern, Eq. 3
# ---------------------------------------------------------------------------

def frozen_logits(a, r, T, rows=None):
    """L[i, j] = a[j] + r[i - j] for j <= i, -inf for j > i (Eq. 3 exponent).

    Returns an array of shape [len(rows), T] (rows default to 0..T-1).
    """
    a = _as64(a)[:T]
    r = _as64(r)[:T]
    i = np.arange(T) if rows is None else np.asarray(rows)
    j = np.arange(T)
    delta = i[:, None] - j[None, :]
    L = np.full(delta.shape, _NEG_INF)
    keep = delta >= 0
    L[keep] = (a[None, :] + r[np.where(keep, delta, 0)])[keep]
    return L


def _row_softmax(L):
    """Row-wise softmax of a matrix whose masked entries are -inf."""
    m = np.max(L, axis=1, keepdims=True)
    e = np.exp(L - m)
    return e / np.sum(e, axis=1, keepdims=True)


def _row_logsumexp(L):
    m = np.max(L, axis=1)
    return m + np.log(np.sum(np.exp(L - m[:, None]), axis=1))


def frozen_pattern(a, r, T, rows=None):
    """Dense P-hat of Eq. 3 for the given query rows.

    P(i, j) = exp(a[j] + r[i - j]) / Z(i), j <= i. Z(i) is the row sum of the
    numerators, so P is the row softmax of frozen_logits; the row maximum is
    subtracted before exp, which leaves every ratio unchanged.
    """
    return _row_softmax(frozen_logits(a, r, T, rows))


def log_normaliser(a, r, T):
    """log Z(i), i = 0..T-1, with Z(i) = sum_{k <= i} exp(a[k] + r[i - k]) (Eq. 3)."""
    return _row_logsumexp(frozen_logits(a, r, T))


# ---------------------------------------------------------------------------
# Ordinary head, Eqs. 5-7
# ---------------------------------------------------------------------------

def _causal_scores(q_rows, k, rows, scale):
    """S = Q K^T * scale on the given query rows, keys j > i set to -inf."""
    S = (q_rows @ k.T) * scale
    T = k.shape[0]
    S[np.arange(T)[None, :] > np.asarray(rows)[:, None]] = _NEG_INF
    return S


def ordinary_pattern(q, k, rows=None):
    """A = softmax_causal(Q K^T / sqrt(d)) on the given query rows (Eqs. 5-6)."""
    q = _as64(q)
    k = _as64(k)
    T, d = k.shape
    rows = np.arange(T) if rows is None else np.asarray(rows)
    return _row_softmax(_causal_scores(q[rows], k, rows, 1.0 / math.sqrt(d)))


# ---------------------------------------------------------------------------
# One (batch, head) slice
# ---------------------------------------------------------------------------

def _blocks(rows, block):
    for s in range(0, len(rows), block):
        yield rows[s:s + block]


def head_fwd(q, k, v, a, r, frozen, rows=None, block=1024):
    """Forward of one head on one sequence.

    q, k, v: [T, d]; a, r: [>= T]; frozen: bool. Returns (o, lse) on the given
    query rows (default all): o [len(rows), d], lse [len(rows)]. Frozen heads
    never read q or k.
    """
    v = _as64(v)
    T, d = v.shape
    rows = np.arange(T) if rows is None else np.asarray(rows)
    o = np.empty((len(rows), d))
    lse = np.empty(len(rows))
    if not frozen:
        q = _as64(q)
        k = _as64(k)
        scale = 1.0 / math.sqrt(d)
    pos = 0
    for blk in _blocks(rows, block):
        if frozen:
            L = frozen_logits(a, r, T, blk)                 # Eq. 3 exponent
        else:
            L = _causal_scores(q[blk], k, blk, scale)       # Eq. 5 + causal mask
        P = _row_softmax(L)                                 # Eq. 3 / Eq. 6
        o[pos:pos + len(blk)] = P @ v                       # P V / Eq. 7
        lse[pos:pos + len(blk)] = _row_logsumexp(L)
        pos += len(blk)
    return o, lse


def head_bwd(q, k, v, do, a, r, frozen, block=1024):
    """Backward of one head on one sequence, given the output gradient dO.

    Returns (dq, dk, dv), each [T, d]. For a frozen head dq = dk = 0 exactly
    and dv = P^T dO; for an ordinary head the chain rule through Eqs. 5-7.
    """
    v = _as64(v)
    do = _as64(do)
    T, d = v.shape
    rows = np.arange(T)
    dv = np.zeros((T, d))
    dq = np.zeros((T, d))
    dk = np.zeros((T, d))
    if frozen:
        for blk in _blocks(rows, block):
            P = frozen_pattern(a, r, T, blk)
            dv += P.T @ do[blk]                             # dV = P^T dZ
        return dq, dk, dv
    q = _as64(q)
    k = _as64(k)
    scale = 1.0 / math.sqrt(d)
    for blk in _blocks(rows, block):
        A = _row_softmax(_causal_scores(q[blk], k, blk, scale))
        dv += A.T @ do[blk]                                 # dV = A^T dO
        dP = do[blk] @ v.T                                  # dP = dO V^T
        D = np.sum(A * dP, axis=1, keepdims=True)           # D_i = sum_j A_ij dP_ij
        dS = A * (dP - D)                                   # softmax Jacobian
        dq[blk] = (dS @ k) * scale                          # dQ = dS K / sqrt(d)
        dk += (dS.T @ q[blk]) * scale                       # dK = dS^T Q / sqrt(d)
    return dq, dk, dv


def pattern_grad(v, do, a, r, block=1024):
    """Gradients of the loss with respect to a and r of one frozen head on one
    sequence, given the output gradient dO (trainable patterns, App. C.3.2).

    With P from Eq. 3, G = dO V^T and D_i = sum_j P_ij G_ij, the logit gradient
    is dL_ij = P_ij (G_ij - D_i); a[j] appears in every logit of key column j and
    r[delta] in every logit of the diagonal i - j = delta, so
        da[j] = sum_{i >= j} dL_ij,   dr[delta] = sum_{i >= delta} dL_{i, i - delta}.
    Returns (da [T], dr [T]).
    """
    v = _as64(v)
    do = _as64(do)
    T = v.shape[0]
    da = np.zeros(T)
    dr = np.zeros(T)
    for blk in _blocks(np.arange(T), block):
        P = frozen_pattern(a, r, T, blk)                    # Eq. 3
        G = do[blk] @ v.T                                   # dL/dP = dO V^T
        D = np.sum(P * G, axis=1, keepdims=True)            # D_i = sum_j P_ij G_ij
        dL = P * (G - D)                                    # row-softmax Jacobian
        da += np.sum(dL, axis=0)                            # column sums
        for t, i in enumerate(blk):
            dr[:i + 1] += dL[t, i::-1]                      # entry (i, j) -> delta = i - j
    return da, dr


# ---------------------------------------------------------------------------
# Whole layer [B, H, T, d]
# ---------------------------------------------------------------------------

def _map(fn, items, threads):
    if threads <= 1:
        return [fn(x) for x in items]
    with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


def attn_fwd(q, k, v, a, r, frozen, threads=1):
    """Layer forward. q, k, v [B, H, T, d]; a, r [H, >= T]; frozen: H flags.

    Returns o [B, H, T, d] and lse [B, H, T] in fp64. Output heads keep their
    original order (App. D.2).
    """
    v = _as64(v)
    B, H, T, d = v.shape
    q = _as64(q)
    k = _as64(k)
    a = _as64(a)
    r = _as64(r)
    o = np.empty((B, H, T, d))
    lse = np.empty((B, H, T))

    def one(bh):
        b, h = bh
        o[b, h], lse[b, h] = head_fwd(q[b, h], k[b, h], v[b, h], a[h], r[h], bool(frozen[h]))

    _map(one, [(b, h) for b in range(B) for h in range(H)], threads)
    return o, lse


def attn_bwd(q, k, v, do, a, r, frozen, threads=1):
    """Layer backward. Returns dq, dk, dv [B, H, T, d] in fp64."""
    v = _as64(v)
    B, H, T, d = v.shape
    q = _as64(q)
    k = _as64(k)
    do = _as64(do)
    a = _as64(a)
    r = _as64(r)
    dq = np.empty((B, H, T, d))
    dk = np.empty((B, H, T, d))
    dv = np.empty((B, H, T, d))

    def one(bh):
        b, h = bh
        dq[b, h], dk[b, h], dv[b, h] = head_bwd(q[b, h], k[b, h], v[b, h], do[b, h],
                                                a[h], r[h], bool(frozen[h]))

    _map(one, [(b, h) for b in range(B) for h in range(H)], threads)
    return dq, dk, dv


def attn_pattern_grad(v, do, a, r, frozen, threads=1):
    """Gradients of a and r for every frozen head, summed over the batch (the
    pattern of a head is shared by all batch entries, §3.2). v, do [B, H, T, d];
    a, r [H, >= T]. Returns da, dr [H, T] in fp64; rows of ordinary heads are 0.
    """
    v = _as64(v)
    do = _as64(do)
    B, H, T, d = v.shape
    a = _as64(a)
    r = _as64(r)
    da = np.zeros((H, T))
    dr = np.zeros((H, T))
    heads = [h for h in range(H) if frozen[h]]
    parts = _map(lambda bh: pattern_grad(v[bh[0], bh[1]], do[bh[0], bh[1]], a[bh[1]], r[bh[1]]),
                 [(b, h) for h in heads for b in range(B)], threads)
    for (b, h), (ga, gr) in zip([(b, h) for h in heads for b in range(B)], parts):
        da[h] += ga
        dr[h] += gr
    return da, dr


def attn_pattern_grad_at(v, do, o, a, r, frozen, cols, dists):
    """Chosen entries of the pattern gradients of every frozen head, summed over
    the batch, with D_i = dO_i . o_i taken from a given layer output o
    (trainable patterns, App. C.3.2).

    For o = P V, the output of Eq. 3, D_i = sum_j P_ij G_ij and the entries are
    those of attn_pattern_grad. A layer output that carries rounding (a bf16 o)
    gives the gradient that the same formula yields with that D:
        da[j] = sum_b sum_{i >= j} P_ij (G_ij - D_i),
        dr[d] = sum_b sum_{i >= d} P_{i,i-d} (G_{i,i-d} - D_i),   G = dO V^T.
    Each entry is formed on its own from log Z (Eq. 3), one column or diagonal
    of P and the matching dot products, so full-length sequences stay cheap.
    v, do, o [B, H, T, d]; a, r [H, >= T]; cols, dists: indices into [0, T).
    Returns da [H, len(cols)], dr [H, len(dists)] in fp64; ordinary heads 0.
    """
    v = _as64(v)
    do = _as64(do)
    o = _as64(o)
    a = _as64(a)
    r = _as64(r)
    B, H, T, d = v.shape
    cols = [int(j) for j in cols]
    dists = [int(x) for x in dists]
    da = np.zeros((H, len(cols)))
    dr = np.zeros((H, len(dists)))
    for h in range(H):
        if not frozen[h]:
            continue
        lz = log_normaliser(a[h], r[h], T)                   # Eq. 3 normalisers
        for b in range(B):
            D = np.sum(do[b, h] * o[b, h], axis=1)           # D_i = dO_i . o_i
            for n, j in enumerate(cols):
                i = np.arange(j, T)
                p = np.exp(a[h, j] + r[h, i - j] - lz[i])    # column j of P
                g = do[b, h, i] @ v[b, h, j]                 # G(i, j)
                da[h, n] += np.sum(p * (g - D[i]))
            for n, x in enumerate(dists):
                i = np.arange(x, T)
                p = np.exp(a[h, i - x] + r[h, x] - lz[i])    # diagonal i - j = x of P
                g = np.sum(do[b, h, i] * v[b, h, i - x], axis=1)
                dr[h, n] += np.sum(p * (g - D[i]))
    return da, dr


# ---------------------------------------------------------------------------
# Compact fitting (§3.2 "Fitting", Eq. 4; App. D.1, Eq. 20; the selection
# algorithm's fitting steps; settings of App. C.1)
# ---------------------------------------------------------------------------

FIT_STEPS = 400        # J, Adam steps without early stopping
FIT_LR = 0.05          # gamma
FIT_TOL = 0.2          # epsilon_fit, nats per row
FIT_FLOOR = 1e-9       # floor of causal entries before row normalisation


def floor_and_normalise(A):
    """Target pattern from a measured mean attention matrix: causal entries
    floored at 1e-9, then every row normalised (the algorithm's step before the
    marginals). Entries above the diagonal are 0."""
    A = _as64(A)
    T = A.shape[0]
    causal = np.tril(np.ones((T, T), dtype=bool))
    P = np.where(causal, np.maximum(A, FIT_FLOOR), 0.0)
    return P / np.sum(P, axis=1, keepdims=True)


def target_marginals(P):
    """eta_abs(j) = sum_{i >= j} P(i, j) and eta_rel(delta) = sum_{i - j = delta} P(i, j)
    of a causal target P (Eq. 4): its key-column sums and its diagonal sums."""
    P = np.tril(_as64(P))
    T = P.shape[0]
    eta_abs = np.sum(P, axis=0)
    eta_rel = np.array([np.trace(P, offset=-delta) for delta in range(T)])
    return eta_abs, eta_rel


def fit_loss(a, r, eta_abs, eta_rel):
    """Eq. 4: (1/T) [sum_i log Z(i) - sum_j eta_abs(j) a(j) - sum_delta eta_rel(delta) r(delta)]."""
    T = len(eta_abs)
    a = _as64(a)[:T]
    r = _as64(r)[:T]
    return (np.sum(log_normaliser(a, r, T)) - np.dot(eta_abs, a) - np.dot(eta_rel, r)) / T


def fit_grad(a, r, eta_abs, eta_rel):
    """Eq. 20 and its analogue for r: the fitted prior's marginals minus the
    target's, over T."""
    T = len(eta_abs)
    fa, fr = target_marginals(frozen_pattern(a, r, T))
    return (fa - eta_abs) / T, (fr - eta_rel) / T


def fit_compact(eta_abs, eta_rel, steps=FIT_STEPS, lr=FIT_LR, betas=(0.9, 0.999), eps=1e-8):
    """Fit (a, r) of Eq. 3 to the target marginals: a = 0 and
    r(delta) = log max(eta_rel(delta) / (T - delta), 1e-9) to start, then `steps`
    Adam steps (Kingma and Ba, bias-corrected moments) on Eq. 4."""
    eta_abs = _as64(eta_abs)
    eta_rel = _as64(eta_rel)
    T = len(eta_abs)
    a = np.zeros(T)
    r = np.log(np.maximum(eta_rel / (T - np.arange(T)), FIT_FLOOR))
    b1, b2 = betas
    m = [np.zeros(T), np.zeros(T)]
    v = [np.zeros(T), np.zeros(T)]
    for t in range(1, steps + 1):
        g = fit_grad(a, r, eta_abs, eta_rel)
        for k, x in enumerate((a, r)):
            m[k] = b1 * m[k] + (1 - b1) * g[k]
            v[k] = b2 * v[k] + (1 - b2) * g[k] ** 2
            mh = m[k] / (1 - b1 ** t)
            vh = v[k] / (1 - b2 ** t)
            x -= lr * mh / (np.sqrt(vh) + eps)
    return a, r


def target_negentropy(P):
    """(1/T) sum_i sum_{j <= i} P(i, j) log P(i, j) of a causal target (terms with
    P = 0 contribute 0): the part of kappa that depends on the target alone, since
    kappa = (1/T) sum_i KL(P(i, .) || P-hat(i, .)) splits into this and the cross
    entropy of Eq. 4."""
    P = np.tril(_as64(P))
    T = P.shape[0]
    pos = P > 0
    return float(np.sum(P[pos] * np.log(P[pos]))) / T


def fit_kl(P, a, r):
    """kappa = (1/T) sum_i KL(P(i, 0..i) || P-hat(i, 0..i)), P-hat from Eq. 3."""
    P = _as64(P)
    T = P.shape[0]
    Ph = frozen_pattern(a, r, T)
    causal = np.tril(np.ones((T, T), dtype=bool)) & (P > 0)
    return float(np.sum(P[causal] * (np.log(P[causal]) - np.log(Ph[causal])))) / T


# ---------------------------------------------------------------------------
# Grouped-query layout (§3.3: the grouped-query path drops the replaced heads'
# query projections and keeps the shared key and value projections; App. C.6:
# 32 query heads share 8 key/value heads)
# ---------------------------------------------------------------------------

def gqa_fwd(q, k, v, a, r, frozen, threads=1):
    """Layer forward with H query heads over Hkv shared key/value heads: query
    head h reads key/value head h // (H / Hkv). q [B, H, T, d]; k, v
    [B, Hkv, T, d]; a, r [H, >= T]; frozen: H flags (a frozen head reads only
    the values of its group). Returns o [B, H, T, d], lse [B, H, T]."""
    q = _as64(q)
    k = _as64(k)
    v = _as64(v)
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    assert H % Hkv == 0, "the query heads must split evenly over the key/value heads"
    g = H // Hkv
    a = _as64(a)
    r = _as64(r)
    o = np.empty((B, H, T, d))
    lse = np.empty((B, H, T))

    def one(bh):
        b, h = bh
        o[b, h], lse[b, h] = head_fwd(q[b, h], k[b, h // g], v[b, h // g], a[h], r[h], bool(frozen[h]))

    _map(one, [(b, h) for b in range(B) for h in range(H)], threads)
    return o, lse


def gqa_bwd(q, k, v, do, a, r, frozen, threads=1):
    """Layer backward of gqa_fwd. Returns dq [B, H, T, d] (zero for frozen
    heads) and dk, dv [B, Hkv, T, d]: a shared head's gradient is the sum of
    what each query head of its group sends it (frozen heads send dV only)."""
    q = _as64(q)
    k = _as64(k)
    v = _as64(v)
    do = _as64(do)
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    assert H % Hkv == 0, "the query heads must split evenly over the key/value heads"
    g = H // Hkv
    a = _as64(a)
    r = _as64(r)
    dq = np.empty((B, H, T, d))
    parts = [[None] * H for _ in range(B)]

    def one(bh):
        b, h = bh
        dq[b, h], dkh, dvh = head_bwd(q[b, h], k[b, h // g], v[b, h // g], do[b, h], a[h], r[h], bool(frozen[h]))
        parts[b][h] = (dkh, dvh)

    _map(one, [(b, h) for b in range(B) for h in range(H)], threads)
    dk = np.zeros((B, Hkv, T, d))
    dv = np.zeros((B, Hkv, T, d))
    for b in range(B):
        for h in range(H):
            dk[b, h // g] += parts[b][h][0]
            dv[b, h // g] += parts[b][h][1]
    return dq, dk, dv
