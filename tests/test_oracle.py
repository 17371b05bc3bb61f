"""Pins for the fp64 oracle, independent of the oracle itself.

Each test checks the oracle against something the paper or the mathematics
fixes: closed forms of Eq. 3 ("When Can Attention Heads Be Statically
Defined?", §3.2), brute force in 50-digit arithmetic, a library attention
routine, finite differences, and invariants of the softmax and of Eq. 3.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from softmax_attention_hybrid_gb300.inputs import custom_workload, make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _frozen_case(T=37, d=5, seed=0, slope=0.05):
    g = _rng(seed)
    a = g.normal(size=T)
    r = -slope * np.arange(T) + 0.5 * g.normal(size=T)
    v = g.normal(size=(T, d))
    return a, r, v


# --------------------------------------------------------------------------
# Eq. 3: structure of the pattern
# --------------------------------------------------------------------------

def test_frozen_rows_stochastic_and_causal():
    a, r, _ = _frozen_case()
    W = oracle.frozen_pattern(a, r, len(a))
    assert np.all(W >= 0)
    assert np.all(np.triu(W, 1) == 0.0)          # P(i, j) = 0 for j > i, exactly
    assert np.max(np.abs(W.sum(axis=1) - 1.0)) < 1e-12


def test_uniform_pattern_is_prefix_mean():
    # a = r = 0: every causal entry of Eq. 3 is exp(0) / (i + 1).
    T, d = 29, 6
    v = _rng(1).normal(size=(T, d))
    o, lse = oracle.head_fwd(None, None, v, np.zeros(T), np.zeros(T), True)
    want = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.max(np.abs(o - want)) < 1e-13
    assert np.max(np.abs(lse - np.log(np.arange(1, T + 1)))) < 1e-13


def test_dominant_r0_gives_identity():
    a, r, v = _frozen_case(T=40, d=4, seed=2)
    r = r.copy()
    r[0] = 60.0
    o, _ = oracle.head_fwd(None, None, v, a, r, True)
    assert np.max(np.abs(o - v)) < 1e-12


@pytest.mark.parametrize("lam", [0.05, 0.7, 3.0])
def test_geometric_closed_form(lam):
    # a = 0, r[delta] = -lam*delta: W_ij = e^{-lam(i-j)} (1-e^{-lam}) / (1-e^{-lam(i+1)}).
    T = 23
    W = oracle.frozen_pattern(np.zeros(T), -lam * np.arange(T), T)
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    want = np.where(j <= i,
                    np.exp(-lam * (i - j)) * (1 - np.exp(-lam)) / (1 - np.exp(-lam * (i + 1))),
                    0.0)
    assert np.max(np.abs(W - want)) < 1e-13


def test_exact_rational_pattern():
    # a[j] = ln(j+1), r[delta] = -delta ln 2: W_ij = (j+1) 2^j / sum_{k<=i} (k+1) 2^k.
    T = 6
    a = np.log(np.arange(1, T + 1, dtype=np.float64))
    r = -np.log(2.0) * np.arange(T)
    W = oracle.frozen_pattern(a, r, T)
    for i in range(T):
        den = sum(Fraction((k + 1) * 2 ** k) for k in range(i + 1))
        for j in range(T):
            want = Fraction((j + 1) * 2 ** j) / den if j <= i else Fraction(0)
            assert abs(W[i, j] - float(want)) < 1e-14
    # row 3 is [1, 4, 12, 32] / 49
    assert np.allclose(W[3, :4], np.array([1, 4, 12, 32]) / 49.0, atol=1e-15, rtol=0)


def test_shift_invariance():
    a, r, _ = _frozen_case(T=31, seed=3)
    W0 = oracle.frozen_pattern(a, r, 31)
    W1 = oracle.frozen_pattern(a + 7.25, r - 3.5, 31)
    assert np.max(np.abs(W0 - W1)) < 1e-13


def test_log_normaliser_closed_form():
    # a = 0, r[delta] = -lam*delta: Z(i) = (1 - e^{-lam(i+1)}) / (1 - e^{-lam}).
    T, lam = 17, 0.3
    lz = oracle.log_normaliser(np.zeros(T), -lam * np.arange(T), T)
    i = np.arange(T)
    want = np.log((1 - np.exp(-lam * (i + 1))) / (1 - np.exp(-lam)))
    assert np.max(np.abs(lz - want)) < 1e-13


def test_prior_longer_than_T_uses_prefix():
    # A stored prior of length 192 used at T = 129 (App. D.2 layer test).
    g = _rng(4)
    a = g.normal(size=192)
    r = -0.05 * np.arange(192) + 0.5 * g.normal(size=192)
    v = g.normal(size=(129, 8))
    o1, l1 = oracle.head_fwd(None, None, v, a, r, True)
    o2, l2 = oracle.head_fwd(None, None, v, a[:129], r[:129], True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# --------------------------------------------------------------------------
# Brute force in 50-digit arithmetic (literal loops of Eqs. 3 and 5-7)
# --------------------------------------------------------------------------

def _mp_frozen(a, r, v):
    import mpmath as mp
    T, d = v.shape
    out = []
    lse = []
    for i in range(T):
        Z = mp.fsum(mp.exp(mp.mpf(a[k]) + mp.mpf(r[i - k])) for k in range(i + 1))
        row = [mp.mpf(0)] * d
        for j in range(i + 1):
            p = mp.exp(mp.mpf(a[j]) + mp.mpf(r[i - j])) / Z
            for c in range(d):
                row[c] += p * mp.mpf(v[j, c])
        out.append([float(x) for x in row])
        lse.append(float(mp.log(Z)))
    return np.array(out), np.array(lse)


def _mp_ordinary(q, k, v):
    import mpmath as mp
    T, d = v.shape
    sc = 1 / mp.sqrt(d)
    out = []
    lse = []
    for i in range(T):
        s = [mp.fsum(mp.mpf(q[i, c]) * mp.mpf(k[j, c]) for c in range(d)) * sc for j in range(i + 1)]
        Z = mp.fsum(mp.exp(x) for x in s)
        row = [mp.fsum(mp.exp(s[j]) / Z * mp.mpf(v[j, c]) for j in range(i + 1)) for c in range(d)]
        out.append([float(x) for x in row])
        lse.append(float(mp.log(Z)))
    return np.array(out), np.array(lse)


@pytest.mark.parametrize("T", [1, 2, 5, 6])
def test_bruteforce_frozen(T):
    import mpmath as mp
    mp.mp.dps = 50
    a, r, v = _frozen_case(T=T, d=3, seed=10 + T)
    o, lse = oracle.head_fwd(None, None, v, a, r, True)
    o_mp, lse_mp = _mp_frozen(a, r, v)
    assert np.max(np.abs(o - o_mp)) < 1e-14
    assert np.max(np.abs(lse - lse_mp)) < 1e-14


@pytest.mark.parametrize("T", [1, 3, 6])
def test_bruteforce_ordinary(T):
    import mpmath as mp
    mp.mp.dps = 50
    g = _rng(20 + T)
    q, k, v = (g.normal(size=(T, 4)) for _ in range(3))
    o, lse = oracle.head_fwd(q, k, v, None, None, False)
    o_mp, lse_mp = _mp_ordinary(q, k, v)
    assert np.max(np.abs(o - o_mp)) < 1e-14
    assert np.max(np.abs(lse - lse_mp)) < 1e-14


def test_first_row_copies_v0():
    a, r, v = _frozen_case(T=9, d=3, seed=5)
    g = _rng(6)
    q, k = g.normal(size=(9, 3)), g.normal(size=(9, 3))
    for fz in (True, False):
        o, _ = oracle.head_fwd(q, k, v, a, r, fz)
        assert np.array_equal(o[0], v[0]) or np.max(np.abs(o[0] - v[0])) < 1e-15


# --------------------------------------------------------------------------
# Ordinary head: library routine, special cases, and the cross-path identity
# --------------------------------------------------------------------------

def test_ordinary_matches_torch_sdpa():
    g = torch.Generator().manual_seed(0)
    B, H, T, d = 2, 3, 45, 16
    q, k, v = (torch.randn(B, H, T, d, generator=g, dtype=torch.float64) for _ in range(3))
    want = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True).numpy()
    o, lse = oracle.attn_fwd(q.numpy(), k.numpy(), v.numpy(), np.zeros((H, T)), np.zeros((H, T)),
                             [0] * H)
    # torch's fp64 CPU kernels are occasionally (about one process in thirty) off by
    # ~1e-9 from both the oracle and a plain einsum; 1e-8 still catches any formula error
    assert np.max(np.abs(o - want)) < 1e-8, np.max(np.abs(o - want))
    S = (q @ k.transpose(-1, -2)) / math.sqrt(d)
    S = S.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    e = np.max(np.abs(lse - torch.logsumexp(S, dim=-1).numpy()))
    assert e < 1e-8, e
    # the dense pattern itself: A V reproduces the library output, rows are stochastic
    A = oracle.ordinary_pattern(q[0, 1].numpy(), k[0, 1].numpy())
    e = np.max(np.abs(A @ v[0, 1].numpy() - want[0, 1]))
    assert e < 1e-8, e
    assert np.all(np.triu(A, 1) == 0.0) and np.max(np.abs(A.sum(1) - 1)) < 1e-13


def test_ordinary_zero_query_is_prefix_mean():
    T, d = 21, 8
    g = _rng(7)
    k, v = g.normal(size=(T, d)), g.normal(size=(T, d))
    o, _ = oracle.head_fwd(np.zeros((T, d)), k, v, None, None, False)
    want = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.max(np.abs(o - want)) < 1e-13


def test_cross_path_ordinary_equals_geometric_frozen():
    # q_i = sqrt(d) e1, k_j = (a_j + lam*j) e1 gives S_ij = a_j + lam*j; the row
    # constant -lam*i cancels in the softmax, leaving a_j + r[i-j], r[delta] = -lam*delta.
    T, d, lam = 50, 8, 0.15
    g = _rng(8)
    a = g.normal(size=T)
    q = np.zeros((T, d))
    q[:, 0] = math.sqrt(d)
    k = np.zeros((T, d))
    k[:, 0] = a + lam * np.arange(T)
    v = g.normal(size=(T, d))
    o_ord, _ = oracle.head_fwd(q, k, v, None, None, False)
    o_frz, _ = oracle.head_fwd(None, None, v, a, -lam * np.arange(T), True)
    assert np.max(np.abs(o_ord - o_frz)) < 1e-12


# --------------------------------------------------------------------------
# Gradients
# --------------------------------------------------------------------------

def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp = x.copy()
        xm = x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


@pytest.mark.parametrize("frozen", [False, True])
def test_finite_differences(frozen):
    T, d = 9, 4
    g = _rng(30 + frozen)
    q, k, v, G = (g.normal(size=(T, d)) for _ in range(4))
    a = g.normal(size=T)
    r = -0.1 * np.arange(T) + 0.5 * g.normal(size=T)

    def loss(qq, kk, vv):
        o, _ = oracle.head_fwd(qq, kk, vv, a, r, frozen)
        return float(np.sum(o * G))

    dq, dk, dv = oracle.head_bwd(q, k, v, G, a, r, frozen)
    nv = _fd_grad(lambda x: loss(q, k, x), v)
    assert np.max(np.abs(dv - nv)) / np.max(np.abs(nv)) < 1e-6
    if frozen:
        assert not np.any(dq) and not np.any(dk)
    else:
        nq = _fd_grad(lambda x: loss(x, k, v), q)
        nk = _fd_grad(lambda x: loss(q, x, v), k)
        assert np.max(np.abs(dq - nq)) / np.max(np.abs(nq)) < 1e-6
        assert np.max(np.abs(dk - nk)) / np.max(np.abs(nk)) < 1e-6


def test_gradients_match_torch_autograd():
    B, H, T, d = 1, 3, 33, 8
    frozen = [0, 1, 0]
    g = torch.Generator().manual_seed(1)
    q, k, v, do = (torch.randn(B, H, T, d, generator=g, dtype=torch.float64) for _ in range(4))
    a = torch.randn(H, T, generator=g, dtype=torch.float64)
    r = -0.05 * torch.arange(T, dtype=torch.float64) + 0.5 * torch.randn(H, T, generator=g,
                                                                        dtype=torch.float64)
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    outs = []
    for h in range(H):
        if frozen[h]:
            i = torch.arange(T)[:, None]
            j = torch.arange(T)[None, :]
            L = a[h][None, :].expand(T, T) + r[h][(i - j).clamp(min=0)]
            L = L.masked_fill(j > i, float("-inf"))
            outs.append(torch.softmax(L, dim=-1) @ vv[:, h])
        else:
            outs.append(torch.nn.functional.scaled_dot_product_attention(
                qq[:, h], kk[:, h], vv[:, h], is_causal=True))
    torch.stack(outs, dim=1).backward(do)
    dq, dk, dv = oracle.attn_bwd(q.numpy(), k.numpy(), v.numpy(), do.numpy(), a.numpy(),
                                 r.numpy(), frozen)
    assert np.max(np.abs(dv - vv.grad.numpy())) < 1e-12
    assert np.max(np.abs(dq - qq.grad.numpy())) < 1e-12
    assert np.max(np.abs(dk - kk.grad.numpy())) < 1e-12


@pytest.mark.parametrize("frozen", [False, True])
def test_gradient_invariants(frozen):
    T, d = 40, 6
    g = _rng(40 + frozen)
    q, k, v, do = (g.normal(size=(T, d)) for _ in range(4))
    a, r, _ = _frozen_case(T=T, seed=41)
    dq, dk, dv = oracle.head_bwd(q, k, v, do, a, r, frozen)
    # Rows of the pattern sum to one, so sum_j dV_j = sum_i dO_i.
    assert np.max(np.abs(dv.sum(0) - do.sum(0))) < 1e-11
    if frozen:
        assert not np.any(dq) and not np.any(dk)
    else:
        # Softmax is invariant to a per-row shift of the scores: sum_j dS_ij = 0.
        assert np.max(np.abs(dk.sum(0))) < 1e-11


# ---------------------------------------------------------------------------
# Trainable patterns (App. C.3.2): gradients of alpha and rho
# ---------------------------------------------------------------------------

def test_pattern_grad_finite_differences():
    # central differences of L = sum(O * G) through Eq. 3, with a stored prior
    # longer than T (only its first T entries may receive gradient)
    T, d, Tp = 11, 3, 15
    g = _rng(60)
    v, G = (g.normal(size=(T, d)) for _ in range(2))
    a = g.normal(size=Tp)
    r = -0.1 * np.arange(Tp) + 0.5 * g.normal(size=Tp)

    def loss(aa, rr):
        o, _ = oracle.head_fwd(None, None, v, aa, rr, True)
        return float(np.sum(o * G))

    da, dr = oracle.pattern_grad(v, G, a, r)
    assert da.shape == (T,) and dr.shape == (T,)
    na = _fd_grad(lambda x: loss(x, r), a)
    nr = _fd_grad(lambda x: loss(a, x), r)
    assert not np.any(na[T:]) and not np.any(nr[T:])
    assert np.max(np.abs(da - na[:T])) / np.max(np.abs(na)) < 1e-6
    assert np.max(np.abs(dr - nr[:T])) / np.max(np.abs(nr)) < 1e-6


def test_pattern_grad_matches_torch_autograd():
    # an independent construction of Eq. 3 in torch (masked logits, softmax), fp64
    T, d = 37, 5
    gen = torch.Generator().manual_seed(7)
    v, do = (torch.randn(T, d, generator=gen, dtype=torch.float64) for _ in range(2))
    a = torch.randn(T, generator=gen, dtype=torch.float64).requires_grad_(True)
    r = (-0.05 * torch.arange(T, dtype=torch.float64)
         + 0.5 * torch.randn(T, generator=gen, dtype=torch.float64)).requires_grad_(True)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    L = (a[None, :] + r[(i - j).clamp(min=0)]).masked_fill(j > i, float("-inf"))
    (torch.softmax(L, dim=-1) @ v).backward(do)
    da, dr = oracle.pattern_grad(v.numpy(), do.numpy(), a.detach().numpy(), r.detach().numpy())
    assert np.max(np.abs(da - a.grad.numpy())) < 1e-12
    assert np.max(np.abs(dr - r.grad.numpy())) < 1e-12


def test_pattern_grad_invariants():
    # adding one constant to every a (or to every r) shifts all logits of every row
    # alike and leaves Eq. 3 unchanged, so both gradients sum to zero; the first key
    # only ever meets offsets 0..T-1 and the last offset only the pair (T-1, 0)
    T, d = 50, 4
    g = _rng(61)
    v, do = (g.normal(size=(T, d)) for _ in range(2))
    a, r, _ = _frozen_case(T=T, seed=62)
    da, dr = oracle.pattern_grad(v, do, a, r)
    assert abs(da.sum()) < 1e-10 and abs(dr.sum()) < 1e-10
    P = oracle.frozen_pattern(a, r, T)
    G = do @ v.T
    # dr[T-1] comes from the single entry (i, j) = (T-1, 0) of the softmax Jacobian
    row = T - 1
    expect = P[row, 0] * (G[row, 0] - np.dot(P[row], G[row]))
    assert abs(dr[T - 1] - expect) < 1e-12


def _pattern_layer_case(seed):
    B, H, T, d = 2, 3, 40, 4
    g = _rng(seed)
    q, k, v, do = (g.normal(size=(B, H, T, d)) for _ in range(4))
    a = g.normal(size=(H, T))
    r = -0.1 * np.arange(T) + 0.4 * g.normal(size=(H, T))
    return q, k, v, do, a, r, [1, 0, 1]


def test_pattern_grad_at_equals_the_full_gradient_for_the_exact_output():
    # with the layer's own output (o = P V for a frozen head), D_i = dO_i . o_i is
    # the D of the softmax Jacobian, so every entry equals attn_pattern_grad's
    q, k, v, do, a, r, frozen = _pattern_layer_case(64)
    T = v.shape[2]
    o, _ = oracle.attn_fwd(q, k, v, a, r, frozen)
    da, dr = oracle.attn_pattern_grad(v, do, a, r, frozen)
    sa, sr = oracle.attn_pattern_grad_at(v, do, o, a, r, frozen, range(T), range(T))
    assert np.max(np.abs(sa - da)) < 1e-12 and np.max(np.abs(sr - dr)) < 1e-12
    # a subset in any order
    cols, dists = [T - 1, 0, 17], [3, T - 1, 0]
    sa2, sr2 = oracle.attn_pattern_grad_at(v, do, o, a, r, frozen, cols, dists)
    assert np.max(np.abs(sa2 - da[:, cols])) < 1e-12 and np.max(np.abs(sr2 - dr[:, dists])) < 1e-12


def test_pattern_grad_at_moves_with_the_given_output():
    # dL = P (G - D) is linear in D: replacing o by o + E moves da[j] by
    # -sum_b sum_i P_ij dO_i . E_i and dr[x] by the same sum along diagonal x
    q, k, v, do, a, r, frozen = _pattern_layer_case(65)
    B, H, T, _ = v.shape
    o, _ = oracle.attn_fwd(q, k, v, a, r, frozen)
    E = 1e-2 * _rng(66).normal(size=o.shape)
    base = oracle.attn_pattern_grad_at(v, do, o, a, r, frozen, range(T), range(T))
    moved = oracle.attn_pattern_grad_at(v, do, o + E, a, r, frozen, range(T), range(T))
    for h in (0, 2):
        P = oracle.frozen_pattern(a[h], r[h], T)
        ea = np.zeros(T)
        er = np.zeros(T)
        for b in range(B):
            M = P * np.sum(do[b, h] * E[b, h], axis=1)[:, None]
            ea -= M.sum(axis=0)
            er -= np.array([np.trace(M, -x) for x in range(T)])
        assert np.max(np.abs(moved[0][h] - base[0][h] - ea)) < 1e-12
        assert np.max(np.abs(moved[1][h] - base[1][h] - er)) < 1e-12
    assert not np.any(moved[0][1]) and not np.any(moved[1][1])


def test_attn_pattern_grad_sums_over_batch():
    # the pattern is shared by the batch: a layer's gradient is the sum over batch
    # entries, and ordinary heads get none
    B, H, T, d = 3, 3, 20, 4
    g = _rng(63)
    v, do = (g.normal(size=(B, H, T, d)) for _ in range(2))
    a = g.normal(size=(H, T))
    r = -0.1 * np.arange(T) + 0.3 * g.normal(size=(H, T))
    frozen = [1, 0, 1]
    da, dr = oracle.attn_pattern_grad(v, do, a, r, frozen)
    assert not np.any(da[1]) and not np.any(dr[1])
    for h in (0, 2):
        parts = [oracle.pattern_grad(v[b, h], do[b, h], a[h], r[h]) for b in range(B)]
        assert np.max(np.abs(da[h] - sum(p[0] for p in parts))) < 1e-12
        assert np.max(np.abs(dr[h] - sum(p[1] for p in parts))) < 1e-12


# ---------------------------------------------------------------------------
# Compact fitting (Eq. 4, Eq. 20, the fitting steps of the selection algorithm)
# ---------------------------------------------------------------------------

def _family_target(T, seed):
    g = _rng(seed)
    a = g.normal(size=T)
    r = -0.1 * np.arange(T) + 0.5 * g.normal(size=T)
    return a, r, oracle.frozen_pattern(a, r, T)


def test_fit_marginals_bruteforce():
    T = 7
    g = _rng(70)
    P = oracle.floor_and_normalise(g.random((T, T)))
    ea, er = oracle.target_marginals(P)
    for j in range(T):
        assert abs(ea[j] - sum(P[i, j] for i in range(j, T))) < 1e-15
    for delta in range(T):
        assert abs(er[delta] - sum(P[i, i - delta] for i in range(delta, T))) < 1e-15
    # each row is a distribution, so both marginals carry T units of mass
    assert abs(ea.sum() - T) < 1e-12 and abs(er.sum() - T) < 1e-12


def test_floor_and_normalise():
    A = np.array([[0.0, 5.0, 5.0], [2.0, 0.0, 7.0], [1.0, 1.0, 2.0]])
    P = oracle.floor_and_normalise(A)
    assert np.allclose(P.sum(axis=1), 1.0) and not np.any(np.triu(P, 1))
    assert P[0, 0] == 1.0                       # a floored lone entry becomes the whole row
    assert abs(P[1, 1] - 1e-9 / (2.0 + 1e-9)) < 1e-24
    assert np.allclose(P[2], [0.25, 0.25, 0.5])


def test_fit_grad_finite_differences():
    T = 10
    _, _, P = _family_target(T, 71)
    ea, er = oracle.target_marginals(P)
    g = _rng(72)
    a, r = g.normal(size=T), g.normal(size=T)
    ga, gr = oracle.fit_grad(a, r, ea, er)
    na = _fd_grad(lambda x: oracle.fit_loss(x, r, ea, er), a)
    nr = _fd_grad(lambda x: oracle.fit_loss(a, x, ea, er), r)
    assert np.max(np.abs(ga - na)) < 1e-8 and np.max(np.abs(gr - nr)) < 1e-8


def test_fit_loss_minus_optimum_is_kl():
    # for a target inside the family of Eq. 3, Eq. 4 is the row-averaged cross
    # entropy, so its excess over the generating parameters is exactly the kappa KL
    T = 24
    a0, r0, P = _family_target(T, 73)
    ea, er = oracle.target_marginals(P)
    g = _rng(74)
    for _ in range(3):
        a, r = g.normal(size=T), g.normal(size=T)
        excess = oracle.fit_loss(a, r, ea, er) - oracle.fit_loss(a0, r0, ea, er)
        assert abs(excess - oracle.fit_kl(P, a, r)) < 1e-12
    assert abs(oracle.fit_kl(P, a0, r0)) < 1e-14


def test_fit_loss_shift_invariant_and_convex():
    T = 16
    _, _, P = _family_target(T, 75)
    ea, er = oracle.target_marginals(P)
    g = _rng(76)
    a, r = g.normal(size=T), g.normal(size=T)
    f = oracle.fit_loss(a, r, ea, er)
    assert abs(oracle.fit_loss(a + 3.0, r, ea, er) - f) < 1e-12
    assert abs(oracle.fit_loss(a, r - 2.0, ea, er) - f) < 1e-12
    a2, r2 = g.normal(size=T), g.normal(size=T)
    mid = oracle.fit_loss((a + a2) / 2, (r + r2) / 2, ea, er)
    assert mid <= (f + oracle.fit_loss(a2, r2, ea, er)) / 2 + 1e-12


def test_fit_recovers_target_from_the_family():
    # the paper's settings (400 Adam steps at 0.05 from its initialisation) fit a
    # target generated by Eq. 3: the marginals match (Eq. 20 at the optimum) and
    # kappa is far below the 0.2-nat acceptance threshold
    T = 48
    _, _, P = _family_target(T, 77)
    ea, er = oracle.target_marginals(P)
    a, r = oracle.fit_compact(ea, er)
    fa, fr = oracle.target_marginals(oracle.frozen_pattern(a, r, T))
    assert np.max(np.abs(fa - ea)) < 1e-3 and np.max(np.abs(fr - er)) < 1e-3
    assert oracle.fit_kl(P, a, r) < 1e-6 < oracle.FIT_TOL


def test_fit_rejects_a_pattern_outside_the_family():
    # a target that attends only to key i // 2 cannot be written as Eq. 3 with a
    # small KL: neither key position nor distance alone decides the weight
    T = 32
    A = np.zeros((T, T))
    A[np.arange(T), np.arange(T) // 2] = 1.0
    P = oracle.floor_and_normalise(A)
    ea, er = oracle.target_marginals(P)
    a, r = oracle.fit_compact(ea, er)
    assert oracle.fit_kl(P, a, r) > oracle.FIT_TOL


def test_target_negentropy_closed_form_and_kappa_split():
    # uniform causal target P(i, j) = 1 / (i + 1): each row has entropy log(i + 1),
    # so (1/T) sum P log P = -(1/T) sum_i log(i + 1) = -log(T!) / T
    T = 30
    P = oracle.floor_and_normalise(np.ones((T, T)))
    assert abs(oracle.target_negentropy(P) + math.lgamma(T + 1) / T) < 1e-12
    # a one-hot row contributes 0 (0 log 0 = 0, 1 log 1 = 0)
    Pid = np.eye(T)
    assert oracle.target_negentropy(Pid) == 0.0
    # kappa = negentropy + Eq. 4 loss, for any (a, r) and any causal target
    g = _rng(79)
    Pt = oracle.floor_and_normalise(g.random((T, T)))
    ea, er = oracle.target_marginals(Pt)
    for _ in range(3):
        a, r = g.normal(size=T), g.normal(size=T)
        kl = oracle.fit_kl(Pt, a, r)
        assert abs(kl - (oracle.target_negentropy(Pt) + oracle.fit_loss(a, r, ea, er))) < 1e-12


def test_fit_start_point_closed_form():
    # App. C.1 starts the fit at a = 0 and r(delta) = log(eta_rel(delta) / (T - delta)):
    # the mean weight on diagonal delta, which holds T - delta entries. For the
    # uniform causal target P(i, j) = 1 / (i + 1), diagonal delta holds
    # 1 / (delta + 1), ..., 1 / T, so eta_rel(delta) = H_T - H_delta (harmonic
    # numbers) and column j sums to H_T - H_j as well; both are computed here in
    # exact rationals, without the oracle's marginals
    T = 20
    harm = [Fraction(0)]
    for n in range(1, T + 1):
        harm.append(harm[-1] + Fraction(1, n))
    eta = np.array([float(harm[T] - harm[t]) for t in range(T)])
    r_want = np.array([math.log(float((harm[T] - harm[t]) / (T - t))) for t in range(T)])
    a, r = oracle.fit_compact(eta, eta, steps=0)
    assert np.all(a == 0.0)
    assert np.max(np.abs(r - r_want)) < 1e-12
    # a diagonal with no mass starts at the 1e-9 floor instead of log 0
    eta0 = eta.copy()
    eta0[T - 1] = 0.0
    _, r0 = oracle.fit_compact(eta, eta0, steps=0)
    assert r0[T - 1] == math.log(1e-9) and np.array_equal(r0[:T - 1], r[:T - 1])


def test_fit_first_adam_steps():
    # Adam with bias-corrected moments (Kingma and Ba; beta = 0.9, 0.999, eps 1e-8):
    # after one step m_hat = g and v_hat = g^2, so every coordinate moves by
    # lr |g| / (|g| + eps), about lr, against the sign of its gradient; the second
    # step is lr m2 / (sqrt(v2) + eps) with m2 = (0.09 g1 + 0.1 g2) / (1 - 0.9^2) and
    # v2 = (0.000999 g1^2 + 0.001 g2^2) / (1 - 0.999^2), the moments written out by hand
    T = 12
    _, _, P = _family_target(T, 78)
    ea, er = oracle.target_marginals(P)
    lr, eps = 0.05, 1e-8
    x0 = oracle.fit_compact(ea, er, steps=0)
    x1 = oracle.fit_compact(ea, er, steps=1)
    x2 = oracle.fit_compact(ea, er, steps=2)
    g1 = oracle.fit_grad(x0[0], x0[1], ea, er)
    g2 = oracle.fit_grad(x1[0], x1[1], ea, er)
    for k in range(2):
        step1 = x1[k] - x0[k]
        assert np.max(np.abs(step1 + lr * g1[k] / (np.abs(g1[k]) + eps))) < 1e-13
        moved = np.abs(g1[k]) > 1e-5
        assert moved.sum() >= T // 2
        assert np.max(np.abs(np.abs(step1[moved]) - lr)) < 1e-3 * lr
        m2 = (0.9 * 0.1 * g1[k] + 0.1 * g2[k]) / (1 - 0.9 ** 2)
        v2 = (0.999 * 0.001 * g1[k] ** 2 + 0.001 * g2[k] ** 2) / (1 - 0.999 ** 2)
        assert np.max(np.abs((x2[k] - x1[k]) + lr * m2 / (np.sqrt(v2) + eps))) < 1e-13


# ---------------------------------------------------------------------------
# Grouped-query layout
# ---------------------------------------------------------------------------

def _gqa_case(B, H, Hkv, T, d, seed):
    g = _rng(seed)
    q = g.normal(size=(B, H, T, d))
    k, v = (g.normal(size=(B, Hkv, T, d)) for _ in range(2))
    do = g.normal(size=(B, H, T, d))
    a = g.normal(size=(H, T))
    r = -0.1 * np.arange(T) + 0.3 * g.normal(size=(H, T))
    return q, k, v, do, a, r


def test_gqa_equals_mha_on_repeated_heads():
    # grouped-query attention is multi-head attention whose key/value heads are
    # repeated over each group; shared-head gradients are the group sums
    B, H, Hkv, T, d = 2, 6, 2, 19, 4
    q, k, v, do, a, r = _gqa_case(B, H, Hkv, T, d, 80)
    frozen = [0, 1, 0, 0, 1, 1]
    rep = lambda x: np.repeat(x, H // Hkv, axis=1)   # noqa: E731
    o, lse = oracle.gqa_fwd(q, k, v, a, r, frozen)
    o_m, lse_m = oracle.attn_fwd(q, rep(k), rep(v), a, r, frozen)
    assert np.array_equal(o, o_m) and np.array_equal(lse, lse_m)
    dq, dk, dv = oracle.gqa_bwd(q, k, v, do, a, r, frozen)
    dq_m, dk_m, dv_m = oracle.attn_bwd(q, rep(k), rep(v), do, a, r, frozen)
    assert np.array_equal(dq, dq_m)
    grp = lambda x: x.reshape(B, Hkv, H // Hkv, T, d).sum(axis=2)   # noqa: E731
    assert np.max(np.abs(dk - grp(dk_m))) < 1e-12 and np.max(np.abs(dv - grp(dv_m))) < 1e-12


def test_gqa_finite_differences():
    B, H, Hkv, T, d = 1, 4, 2, 7, 3
    q, k, v, G, a, r = _gqa_case(B, H, Hkv, T, d, 81)
    frozen = [0, 1, 1, 0]

    def loss(kk, vv):
        o, _ = oracle.gqa_fwd(q, kk, vv, a, r, frozen)
        return float(np.sum(o * G))

    _, dk, dv = oracle.gqa_bwd(q, k, v, G, a, r, frozen)
    nk = _fd_grad(lambda x: loss(x, v), k)
    nv = _fd_grad(lambda x: loss(k, x), v)
    assert np.max(np.abs(dk - nk)) / np.max(np.abs(nk)) < 1e-6
    assert np.max(np.abs(dv - nv)) / np.max(np.abs(nv)) < 1e-6


def test_frozen_head_ignores_nan_qk():
    B, H, T, d = 1, 2, 12, 4
    g = _rng(50)
    q, k, v = (g.normal(size=(B, H, T, d)) for _ in range(3))
    a = g.normal(size=(H, T))
    r = g.normal(size=(H, T))
    q[:, 1] = np.nan
    k[:, 1] = np.nan
    o, lse = oracle.attn_fwd(q, k, v, a, r, [0, 1])
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    dq, dk, dv = oracle.attn_bwd(q, k, v, v, a, r, [0, 1])
    assert np.all(dq[:, 1] == 0) and np.all(dk[:, 1] == 0) and np.all(np.isfinite(dv))


# --------------------------------------------------------------------------
# Causality, layer assembly, row blocking
# --------------------------------------------------------------------------

def test_causal_prefix_truncation():
    w = custom_workload(2, 3, 70, d=8, dtype="fp32", frozen=(1,), scale=1.0)
    x = make_inputs(w, seed=3)
    args = [x[n].double().numpy() for n in ("q", "k", "v")]
    o, lse = oracle.attn_fwd(*args, x["a"].numpy(), x["r"].numpy(), x["frozen"])
    Tp = 33
    o2, lse2 = oracle.attn_fwd(*[t[:, :, :Tp] for t in args], x["a"].numpy()[:, :Tp],
                               x["r"].numpy()[:, :Tp], x["frozen"])
    assert np.max(np.abs(o[:, :, :Tp] - o2)) < 1e-13
    assert np.max(np.abs(lse[:, :, :Tp] - lse2)) < 1e-13


def test_row_blocking_does_not_change_results():
    T, d = 77, 5
    g = _rng(60)
    q, k, v, do = (g.normal(size=(T, d)) for _ in range(4))
    a, r, _ = _frozen_case(T=T, seed=61)
    for fz in (False, True):
        o1, l1 = oracle.head_fwd(q, k, v, a, r, fz, block=T)
        o2, l2 = oracle.head_fwd(q, k, v, a, r, fz, block=10)
        assert np.max(np.abs(o1 - o2)) < 1e-14 and np.max(np.abs(l1 - l2)) < 1e-14
        g1 = oracle.head_bwd(q, k, v, do, a, r, fz, block=T)
        g2 = oracle.head_bwd(q, k, v, do, a, r, fz, block=13)
        for x1, x2 in zip(g1, g2):
            assert np.max(np.abs(x1 - x2)) < 1e-13


def test_sampled_rows_match_full():
    T, d = 60, 4
    g = _rng(70)
    q, k, v = (g.normal(size=(T, d)) for _ in range(3))
    a, r, _ = _frozen_case(T=T, seed=71)
    rows = np.array([0, 7, 31, 59])
    for fz in (False, True):
        o, l = oracle.head_fwd(q, k, v, a, r, fz)
        os_, ls = oracle.head_fwd(q, k, v, a, r, fz, rows=rows)
        assert np.array_equal(o[rows], os_) or np.max(np.abs(o[rows] - os_)) < 1e-14
        assert np.max(np.abs(l[rows] - ls)) < 1e-14


def test_layer_keeps_head_order():
    w = custom_workload(2, 4, 19, d=4, dtype="fp32", frozen=(0, 3), scale=1.0)
    x = make_inputs(w, seed=9)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    o, lse = oracle.attn_fwd(q, k, v, a, r, x["frozen"], threads=3)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, a, r, x["frozen"], threads=3)
    for b in range(2):
        for h in range(4):
            fz = bool(x["frozen"][h])
            oh, lh = oracle.head_fwd(q[b, h], k[b, h], v[b, h], a[h], r[h], fz)
            assert np.array_equal(o[b, h], oh) and np.array_equal(lse[b, h], lh)
            gh = oracle.head_bwd(q[b, h], k[b, h], v[b, h], do[b, h], a[h], r[h], fz)
            assert all(np.array_equal(x1, x2) for x1, x2 in zip((dq[b, h], dk[b, h], dv[b, h]), gh))


def test_regression_fixture():
    import json
    import os
    import importlib.util
    here = os.path.join(os.path.dirname(__file__), "golden")
    spec = importlib.util.spec_from_file_location("mk", os.path.join(here, "make_oracle_small.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    with open(os.path.join(here, "oracle_small.json")) as f:
        want = json.load(f)
    got = mk.compute()
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.max(np.abs(np.array(got[key]) - np.array(want[key]))) < 1e-12
