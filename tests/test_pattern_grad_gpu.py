"""GPU parity of saf_pattern_grad (gradients of a and r for trainable patterns,
App. C.3.2) against the fp64 oracle.

The kernel takes D_i = dO_i . O_i from the forward output it is given. With
bf16 inputs that output is rounded to bf16, which moves D by up to 2^-9 of
|dO||O| per row; the bound below allows for that. fp32 inputs get a tight
bound. Rows of ordinary heads must be exact zeros.
"""
import numpy as np
import pytest
import torch

import oracle
from softmax_attention_hybrid_gb300.inputs import custom_workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def saf():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from softmax_attention_hybrid_gb300 import saf as mod
    return mod


@pytest.mark.parametrize("dtype,T,tol", [("fp32", 200, 1e-3), ("bf16", 200, 3e-2), ("bf16", 321, 3e-2)])
def test_pattern_grad_matches_oracle(saf, dtype, T, tol):
    w = custom_workload(2, 3, T, dtype=dtype, frozen=(0, 2), slope=0.05)
    x = make_inputs(w, seed=50 + T)
    g = {n: x[n].to("cuda") for n in ("q", "k", "v", "do", "a", "r")}
    o, lse = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    da, dr = saf.saf_pattern_grad(g["v"], g["do"], o, lse, g["a"], g["r"], x["frozen"])
    torch.cuda.synchronize()
    da, dr = da.double().cpu().numpy(), dr.double().cpu().numpy()
    v, do = (x[n].double().numpy() for n in ("v", "do"))
    ra, rr = oracle.attn_pattern_grad(v, do, x["a"].double().numpy(), x["r"].double().numpy(), x["frozen"])
    assert not np.any(da[1]) and not np.any(dr[1])
    for h in (0, 2):
        scale = max(1.0, np.max(np.abs(ra[h])), np.max(np.abs(rr[h])))
        assert np.max(np.abs(da[h] - ra[h])) <= tol * scale, (h, np.max(np.abs(da[h] - ra[h])), scale)
        assert np.max(np.abs(dr[h] - rr[h])) <= tol * scale, (h, np.max(np.abs(dr[h] - rr[h])), scale)
        # both gradients sum to zero (shifting all of a, or all of r, leaves Eq. 3 unchanged)
        assert abs(da[h].sum()) <= tol * scale * T ** 0.5 and abs(dr[h].sum()) <= tol * scale * T ** 0.5


@pytest.mark.parametrize("dtype,d", [("fp32", 96), ("bf16", 128)])
def test_pattern_grad_wide_heads_matches_oracle(saf, dtype, d):
    # head dimensions 96 and 128 on CUDA cores: G and D summed over 64-column chunks
    T, tol = 257, (1e-3 if dtype == "fp32" else 3e-2)
    w = custom_workload(2, 3, T, d=d, dtype=dtype, frozen=(0, 2), slope=0.05)
    x = make_inputs(w, seed=60 + d)
    g = {n: x[n].to("cuda") for n in ("q", "k", "v", "do", "a", "r")}
    o, lse = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    da, dr = saf.saf_pattern_grad(g["v"], g["do"], o, lse, g["a"], g["r"], x["frozen"])
    torch.cuda.synchronize()
    da, dr = da.double().cpu().numpy(), dr.double().cpu().numpy()
    v, do = (x[n].double().numpy() for n in ("v", "do"))
    ra, rr = oracle.attn_pattern_grad(v, do, x["a"].double().numpy(), x["r"].double().numpy(), x["frozen"])
    assert not np.any(da[1]) and not np.any(dr[1])
    for h in (0, 2):
        scale = max(1.0, np.max(np.abs(ra[h])), np.max(np.abs(rr[h])))
        assert np.max(np.abs(da[h] - ra[h])) <= tol * scale
        assert np.max(np.abs(dr[h] - rr[h])) <= tol * scale


# ---------------------------------------------------------------------------
# Tensor-core form (saf_pattern_grad_tc): bf16, d = 64, 96, 128, fixed summation order
# ---------------------------------------------------------------------------
#
# The kernel takes D_i = dO_i . o_i from the bf16 forward output o it is given,
# while the oracle uses the exact D_i = sum_j P_ij G_ij. dL is linear in D, so
# the oracle's gradients move by exactly -sum_i P_ij dD_i (da) and
# -sum_i P_{i,i-d} dD_i (dr), dD_i = dO_i . (o_i - O_i); the tests add that
# shift to the oracle and then allow fp32 rounding only: 2^-15 of
# sum_b sum_i P (|dO_i| . |V_j| + |dO_i| . |o_i|) over the same entries (the
# kernel rounds G, D, W and every partial sum to fp32), plus 1e-6 of the
# gradients' scale.

def _col_and_diag(M):
    """Column sums and diagonal sums sum_i M[i, i - d] of a T x T matrix."""
    T = M.shape[0]
    return M.sum(axis=0), np.array([np.trace(M, -d) for d in range(T)])


def _tc_expectation(x, o):
    """Oracle gradients shifted to the kernel's D, and the rounding bound."""
    v, do = (x[n].double().numpy() for n in ("v", "do"))
    q, k = (x[n].double().numpy() for n in ("q", "k"))
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    fz = x["frozen"]
    B, H, T, _ = v.shape
    O, _ = oracle.attn_fwd(q, k, v, a, r, fz)
    ra, rr = oracle.attn_pattern_grad(v, do, a, r, fz)
    o = o.double().cpu().numpy()
    ba, br = np.zeros((H, T)), np.zeros((H, T))
    for h in range(H):
        if not fz[h]:
            continue
        P = oracle.frozen_pattern(a[h], r[h], T)
        for b in range(B):
            dD = np.sum(do[b, h] * (o[b, h] - O[b, h]), axis=1)
            sa, sr = _col_and_diag(P * dD[:, None])
            ra[h] -= sa
            rr[h] -= sr
            G = np.abs(do[b, h]) @ np.abs(v[b, h]).T          # bounds |G| and its rounding
            D = np.sum(np.abs(do[b, h] * o[b, h]), axis=1)
            ma, mr = _col_and_diag(P * (G + D[:, None]))
            ba[h] += ma
            br[h] += mr
    scale = max(1.0, np.max(np.abs(ra)), np.max(np.abs(rr)))
    return ra, rr, 2.0 ** -15 * ba + 1e-6 * scale, 2.0 ** -15 * br + 1e-6 * scale


def _run_tc(saf, x):
    g = {n: x[n].to("cuda") for n in ("q", "k", "v", "do", "a", "r")}
    o, lse = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    da, dr = saf.saf_pattern_grad_tc(g["v"], g["do"], o, lse, g["a"], g["r"], x["frozen"])
    torch.cuda.synchronize()
    return o, da, dr


def _check_tc(x, o, da, dr):
    ra, rr, ta, tr = _tc_expectation(x, o)
    da, dr = da.double().cpu().numpy(), dr.double().cpu().numpy()
    for h in range(da.shape[0]):
        if not x["frozen"][h]:
            assert not np.any(da[h]) and not np.any(dr[h]), h
            continue
        ea, er = np.abs(da[h] - ra[h]), np.abs(dr[h] - rr[h])
        assert np.all(ea <= ta[h]), (h, int(np.argmax(ea - ta[h])), float(np.max(ea)), float(np.max(ta[h])))
        assert np.all(er <= tr[h]), (h, int(np.argmax(er - tr[h])), float(np.max(er)), float(np.max(tr[h])))


@pytest.mark.parametrize("B,H,T,frozen", [(2, 3, 200, (0, 2)), (2, 3, 321, (0, 2)), (1, 4, 700, (1, 2, 3)),
                                          (3, 2, 128, (1,)), (1, 2, 129, (0,)), (2, 1, 1, (0,))])
def test_pattern_grad_tc_matches_oracle(saf, B, H, T, frozen):
    # several 128 x 128 tiles and bands, a ragged last block, a single tile, T = 1
    w = custom_workload(B, H, T, frozen=frozen, slope=0.05)
    x = make_inputs(w, seed=70 + T + H)
    _check_tc(x, *_run_tc(saf, x))


@pytest.mark.parametrize("d", [96, 128])
@pytest.mark.parametrize("B,H,T,frozen", [(2, 3, 321, (0, 2)), (1, 2, 129, (0,))])
def test_pattern_grad_tc_wide_heads(saf, d, B, H, T, frozen):
    # head dimensions 96 and 128: G = dO V^T over two 64-column atoms per tile (columns
    # past 96 zero-filled), several tiles and bands and a ragged last block
    w = custom_workload(B, H, T, d=d, frozen=frozen, slope=0.05)
    x = make_inputs(w, seed=80 + T + d)
    _check_tc(x, *_run_tc(saf, x))


def test_pattern_grad_tc_exact_form_head(saf):
    # head 1: a sink of weight e^100 at key 0 and a steep distance penalty, so
    # log Z' < -64 on far rows and the kernel takes the exact form for it;
    # head 2 stays in the factorised form
    w = custom_workload(1, 4, 600, frozen=(1, 2), slope=0.02)
    x = make_inputs(w, seed=23)
    x["a"][1, 0] = 100.0
    x["r"][1] = -1.0 * torch.arange(600, dtype=torch.float32)
    x["do"] = (x["do"].float() * 0.1).to(x["do"].dtype)
    _check_tc(x, *_run_tc(saf, x))


def test_pattern_grad_tc_is_deterministic_and_agrees_with_cuda_cores(saf):
    w = custom_workload(2, 4, 1000, frozen=(0, 3), slope=0.02)
    x = make_inputs(w, seed=24)
    g = {n: x[n].to("cuda") for n in ("q", "k", "v", "do", "a", "r")}
    o, lse = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    ws = torch.empty(saf.saf_pattern_grad_tc_workspace_bytes(2, 4, 1000, 2), dtype=torch.uint8, device="cuda")
    runs = [saf.saf_pattern_grad_tc(g["v"], g["do"], o, lse, g["a"], g["r"], x["frozen"], workspace=ws)
            for _ in range(3)]
    torch.cuda.synchronize()
    for da, dr in runs[1:]:
        assert torch.equal(da, runs[0][0]) and torch.equal(dr, runs[0][1])
    # the CUDA-core kernel forms the same sums from the same o in another order
    ca, cr = saf.saf_pattern_grad(g["v"], g["do"], o, lse, g["a"], g["r"], x["frozen"])
    torch.cuda.synchronize()
    scale = max(1.0, ca.abs().max().item(), cr.abs().max().item())
    assert (runs[0][0] - ca).abs().max().item() <= 1e-4 * scale
    assert (runs[0][1] - cr).abs().max().item() <= 1e-4 * scale


def test_pattern_grad_tc_without_frozen_heads_gives_zeros(saf):
    w = custom_workload(1, 2, 300, frozen=(), slope=0.02)
    x = make_inputs(w, seed=25)
    g = {n: x[n].to("cuda") for n in ("q", "k", "v", "do", "a", "r")}
    o, lse = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    da = torch.full((2, 300), 5.0, device="cuda")
    dr = torch.full((2, 300), 5.0, device="cuda")
    saf.saf_pattern_grad_tc(g["v"], g["do"], o, lse, g["a"], g["r"], x["frozen"], da=da, dr=dr)
    torch.cuda.synchronize()
    assert not torch.any(da) and not torch.any(dr)


@pytest.mark.parametrize("name", ["gpt2_124m_25", "gpt2_124m_50", "1b_d96"])
def test_pattern_grad_tc_full_size_sampled(saf, name):
    # the bench's workloads at full size, in the launch configuration bench.py times
    # (one call on the layer's own o and lse): sampled entries of da and dr against
    # the oracle's entry-wise form with the same D = dO . o, within the fp32 rounding
    # bound of the small cases
    from softmax_attention_hybrid_gb300.inputs import WORKLOADS
    w = WORKLOADS[name]
    x = make_inputs(w, seed=1)
    g = {n: x[n].to("cuda") for n in ("q", "k", "v", "do", "a", "r")}
    o, lse = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    ws = torch.empty(saf.saf_pattern_grad_tc_workspace_bytes(w.B, w.H, w.T, sum(x["frozen"])), dtype=torch.uint8,
                     device="cuda")
    da, dr = saf.saf_pattern_grad_tc(g["v"], g["do"], o, lse, g["a"], g["r"], x["frozen"], workspace=ws)
    assert saf.saf_device_status(ws) == saf.SAF_OK
    T = w.T
    rng = np.random.default_rng(5)
    idx = sorted(set([0, 1, 127, 128, 129, T // 2, T - 129, T - 128, T - 2, T - 1] +
                     rng.integers(0, T, size=14).tolist()))
    v, do = (x[n].double().numpy() for n in ("v", "do"))
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    on = o.double().cpu().numpy()
    ra, rr = oracle.attn_pattern_grad_at(v, do, on, a, r, x["frozen"], idx, idx)
    da, dr = da.double().cpu().numpy(), dr.double().cpu().numpy()
    scale = max(1.0, np.max(np.abs(ra)), np.max(np.abs(rr)))
    for h in range(w.H):
        if not x["frozen"][h]:
            assert not np.any(da[h]) and not np.any(dr[h])
            continue
        P = oracle.frozen_pattern(a[h], r[h], T)
        ba, br = np.zeros(len(idx)), np.zeros(len(idx))
        for b in range(w.B):
            Dabs = np.sum(np.abs(do[b, h] * on[b, h]), axis=1)
            for n, j in enumerate(idx):
                gc = np.abs(do[b, h, j:]) @ np.abs(v[b, h, j])
                ba[n] += np.sum(P[j:, j] * (gc + Dabs[j:]))
                ii = np.arange(j, T)
                gd = np.sum(np.abs(do[b, h, ii]) * np.abs(v[b, h, ii - j]), axis=1)
                br[n] += np.sum(P[ii, ii - j] * (gd + Dabs[ii]))
        ta, tr = 2.0 ** -15 * ba + 1e-6 * scale, 2.0 ** -15 * br + 1e-6 * scale
        ea, er = np.abs(da[h, idx] - ra[h]), np.abs(dr[h, idx] - rr[h])
        assert np.all(ea <= ta), (name, h, float(np.max(ea)), float(np.max(ta)))
        assert np.all(er <= tr), (name, h, float(np.max(er)), float(np.max(tr)))
