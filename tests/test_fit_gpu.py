"""GPU parity of the compact fitter (saf_fit_compact) against the fp64 oracle.

The fitter runs 400 Adam steps in fp32. Eq. 4 is invariant to adding a
constant to all of a or to all of r, so the comparison is on what the fit is
for: the fitted pattern's KL from the target (the acceptance statistic of the
selection algorithm, threshold 0.2 nats) and, for targets from the family of
Eq. 3, its marginals. The reported loss must be Eq. 4 at the returned
parameters.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def saf():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from softmax_attention_hybrid_gb300 import saf as mod
    return mod


def _targets(T, seed):
    g = np.random.default_rng(seed)
    # two targets from the family of Eq. 3 and one outside it (each row attends to key i // 2)
    P1 = oracle.frozen_pattern(g.normal(size=T), -0.1 * np.arange(T) + 0.5 * g.normal(size=T), T)
    P2 = oracle.frozen_pattern(0.3 * g.normal(size=T), -0.02 * np.arange(T) + 0.2 * g.normal(size=T), T)
    A = np.zeros((T, T))
    A[np.arange(T), np.arange(T) // 2] = 1.0
    return [P1, P2, oracle.floor_and_normalise(A)]


def _dev(x):
    return torch.tensor(np.asarray(x), dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("T", [96, 300])
def test_fit_compact_matches_oracle(saf, T):
    Ps = _targets(T, 80 + T)
    marg = [oracle.target_marginals(P) for P in Ps]
    a, r, loss = saf.saf_fit_compact(_dev([m[0] for m in marg]), _dev([m[1] for m in marg]),
                                     steps=oracle.FIT_STEPS, lr=oracle.FIT_LR)
    torch.cuda.synchronize()
    a, r, loss = (x.double().cpu().numpy() for x in (a, r, loss))
    for h, P in enumerate(Ps):
        ea, er = marg[h]
        assert abs(loss[h] - oracle.fit_loss(a[h], r[h], ea, er)) < 1e-4
        ao, ro = oracle.fit_compact(ea, er)
        k_gpu, k_ref = oracle.fit_kl(P, a[h], r[h]), oracle.fit_kl(P, ao, ro)
        assert abs(k_gpu - k_ref) <= 1e-3 + 1e-2 * k_ref, (h, k_gpu, k_ref)
        assert (k_gpu <= oracle.FIT_TOL) == (k_ref <= oracle.FIT_TOL)
        if h < 2:
            fa, fr = oracle.target_marginals(oracle.frozen_pattern(a[h], r[h], T))
            assert np.max(np.abs(fa - ea) / np.maximum(1.0, ea)) < 2e-2
            assert np.max(np.abs(fr - er) / np.maximum(1.0, er)) < 2e-2


def test_fit_compact_zero_steps_is_the_start_point(saf):
    T = 64
    ea, er = oracle.target_marginals(_targets(T, 90)[0])
    a, r, loss = saf.saf_fit_compact(_dev(ea[None]), _dev(er[None]), steps=0)
    torch.cuda.synchronize()
    ao, ro = oracle.fit_compact(ea, er, steps=0)
    assert np.max(np.abs(a.double().cpu().numpy()[0] - ao)) == 0.0
    assert np.max(np.abs(r.double().cpu().numpy()[0] - ro)) < 1e-5
    assert abs(loss.item() - oracle.fit_loss(ao, ro, ea, er)) < 1e-4


# ---------------------------------------------------------------------------
# From a measured pattern to accept / reject on the device
# ---------------------------------------------------------------------------

def _measured(T, seed):
    """Three 'measured' mean attention matrices (dense, with values above the
    diagonal that must be ignored): a pattern from the family of Eq. 3 with
    noise, a spiky random one (uniform draws to the 4th power: neither key
    position nor distance decides its weights), and one that attends to key
    i // 2 only (zeros elsewhere, which the 1e-9 floor turns into a valid
    target)."""
    g = np.random.default_rng(seed)
    A0 = oracle.frozen_pattern(g.normal(size=T), -0.08 * np.arange(T) + 0.4 * g.normal(size=T), T)
    A0 = A0 * (1.0 + 0.01 * g.random((T, T))) + np.triu(g.random((T, T)), 1)
    A1 = g.random((T, T)) ** 4
    A2 = np.zeros((T, T))
    A2[np.arange(T), np.arange(T) // 2] = 1.0
    A2 += np.triu(np.ones((T, T)), 1)
    return np.stack([A0, A1, A2])


@pytest.mark.parametrize("T", [96, 257])
def test_target_stats_match_oracle(saf, T):
    A = _measured(T, 60 + T)
    ea, er, ng = saf.saf_fit_target_stats(_dev(A))
    ea2, er2, ng2 = saf.saf_fit_target_stats(_dev(A))
    torch.cuda.synchronize()
    # fixed summation order: the same bits on every run
    assert torch.equal(ea, ea2) and torch.equal(er, er2) and torch.equal(ng, ng2)
    ea, er, ng = (x.double().cpu().numpy() for x in (ea, er, ng))
    for h in range(A.shape[0]):
        P = oracle.floor_and_normalise(A[h].astype(np.float32).astype(np.float64))
        ea_ref, er_ref = oracle.target_marginals(P)
        assert np.max(np.abs(ea[h] - ea_ref)) <= 1e-4 * max(1.0, np.max(ea_ref)), h
        assert np.max(np.abs(er[h] - er_ref)) <= 1e-4 * max(1.0, np.max(er_ref)), h
        assert abs(ng[h] - oracle.target_negentropy(P)) <= 1e-4, (h, ng[h], oracle.target_negentropy(P))


def test_fit_from_target_accepts_and_rejects(saf):
    # the whole selection path on the device: the noisy family pattern passes the
    # 0.2-nat test, the spiky random pattern and the i // 2 pattern do not; kappa
    # equals the fp64 KL of each target from the fitted pattern the device returns
    T = 128
    A = _measured(T, 64)
    a, r, kappa, accept = saf.saf_fit_from_target(_dev(A), steps=oracle.FIT_STEPS, lr=oracle.FIT_LR,
                                                  tol=oracle.FIT_TOL)
    torch.cuda.synchronize()
    a, r, kappa = (x.double().cpu().numpy() for x in (a, r, kappa))
    accept = accept.cpu().numpy()
    for h in range(3):
        P = oracle.floor_and_normalise(A[h].astype(np.float32).astype(np.float64))
        k_ref = oracle.fit_kl(P, a[h], r[h])
        assert abs(kappa[h] - k_ref) <= 2e-4 + 1e-3 * k_ref, (h, kappa[h], k_ref)
        assert accept[h] == (1 if kappa[h] <= oracle.FIT_TOL else 0)
        # and the oracle's own fit of the same target takes the same decision
        ao, ro = oracle.fit_compact(*oracle.target_marginals(P))
        assert (oracle.fit_kl(P, ao, ro) <= oracle.FIT_TOL) == bool(accept[h]), h
    assert accept.tolist() == [1, 0, 0]
