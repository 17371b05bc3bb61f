"""Prepared frozen-pattern state (saf_frozen_prepare + saf_attn_*_prepared).

A frozen head's pattern depends on a and r only ("When Can Attention Heads Be
Statically Defined?", §3.2 Eq. 3), and the paper keeps its normalisers as
persistent state (§3.3, App. D.2). The prepared calls take them from a state
filled once; their forward must equal saf_attn_fwd bit for bit, and their
backward must match the fp64 oracle within the parity tolerances, with exact
zeros in dq and dk of frozen heads.
"""
import numpy as np
import pytest
import torch

import oracle
from softmax_attention_hybrid_gb300.inputs import custom_workload, make_gqa_inputs, make_inputs
from tests import _parity_log

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 2e-2), "fp32": (2e-4, 2e-4)}


@pytest.fixture(scope="module")
def saf():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from softmax_attention_hybrid_gb300 import saf as mod
    return mod


def _np(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_prepared_layer_matches_per_call_normalisers(saf, dtype):
    w = custom_workload(2, 6, 413, dtype=dtype, frozen=(1, 4, 5), scale=0.5 if dtype == "bf16" else 1.0,
                        slope=0.03)
    x = make_inputs(w, seed=90)
    dev = torch.device("cuda:0")
    g = {n: x[n].to(dev) for n in ("q", "k", "v", "do", "a", "r")}
    state = saf.saf_frozen_prepare(g["a"], g["r"], x["frozen"], w.T, w.torch_dtype)
    o1, l1 = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    o2, l2 = saf.saf_attn_fwd_prepared(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"], state)
    dq, dk, dv = saf.saf_attn_bwd_prepared(g["q"], g["k"], g["v"], o2, g["do"], l2, g["a"], g["r"], x["frozen"],
                                           state)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd(q, k, v, do, a, r, x["frozen"], threads=8)
    tol = TOL[dtype][1]
    err = {nm: float(np.max(np.abs(_np(t) - ref))) for nm, t, ref in
           (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref))}
    _parity_log.record(f"prepared state {dtype}", err, {nm: tol for nm in err})
    assert max(err.values()) <= tol, err
    fz = [h for h in range(w.H) if x["frozen"][h]]
    assert torch.all(dq[:, fz] == 0) and torch.all(dk[:, fz] == 0)


@pytest.mark.parametrize("d", [96, 128])
def test_prepared_layer_at_wide_head_dims(saf, d):
    # the d = 96 / 128 kernels with the state: the forward equals the per-call one bit
    # for bit, and so does the backward (its passes add in a fixed order); one state
    # also serves the grouped layout
    w = custom_workload(2, 8, 300, d=d, frozen=(1, 4, 5), slope=0.03)
    dev = torch.device("cuda:0")
    for Hkv in (8, 2):
        x = make_gqa_inputs(w, Hkv, seed=93 + d)
        g = {n: x[n].to(dev) for n in ("q", "k", "v", "do", "a", "r")}
        state = saf.saf_frozen_prepare(g["a"], g["r"], x["frozen"], w.T, torch.bfloat16)
        o1, l1 = saf.saf_attn_fwd_gqa(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
        o2, l2 = saf.saf_attn_fwd_prepared(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"], state)
        b1 = saf.saf_attn_bwd_gqa(g["q"], g["k"], g["v"], o1, g["do"], l1, g["a"], g["r"], x["frozen"])
        b2 = saf.saf_attn_bwd_prepared(g["q"], g["k"], g["v"], o2, g["do"], l2, g["a"], g["r"], x["frozen"], state)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        for t1, t2 in zip(b1, b2):
            assert torch.equal(t1, t2)
    # and against the oracle, for the last (grouped) layout
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    o_ref, _ = oracle.gqa_fwd(q, k, v, a, r, x["frozen"], threads=8)
    refs = oracle.gqa_bwd(q, k, v, do, a, r, x["frozen"], threads=8)
    err = {"o": float(np.max(np.abs(_np(o2) - o_ref)))}
    err.update({nm: float(np.max(np.abs(_np(t) - ref))) for nm, t, ref in zip(("dq", "dk", "dv"), b2, refs)})
    _parity_log.record(f"prepared state bf16 d{d} H8/Hkv2", err, {nm: TOL["bf16"][nm != "o"] for nm in err})
    assert err["o"] <= TOL["bf16"][0] and max(err["dq"], err["dk"], err["dv"]) <= TOL["bf16"][1], err


def test_one_state_serves_every_batch_and_the_grouped_layout(saf):
    # the state is per head and sequence length, not per batch entry: prepared once,
    # it serves a multi-head batch of 1 and a grouped-query batch of 3
    dev = torch.device("cuda:0")
    w1 = custom_workload(1, 8, 300, frozen=(2, 7), slope=0.02)
    w3 = custom_workload(3, 8, 300, frozen=(2, 7), slope=0.02)
    x1 = make_inputs(w1, seed=91)
    x3 = make_gqa_inputs(w3, 2, seed=91)   # a, r are the same draws: same seed, same H, T
    assert torch.equal(x1["a"], x3["a"]) and torch.equal(x1["r"], x3["r"])
    a, r = x1["a"].to(dev), x1["r"].to(dev)
    state = saf.saf_frozen_prepare(a, r, x1["frozen"], 300, torch.bfloat16)
    for x, gqa in ((x1, False), (x3, True)):
        g = {n: x[n].to(dev) for n in ("q", "k", "v")}
        ref = (saf.saf_attn_fwd_gqa if gqa else saf.saf_attn_fwd)(g["q"], g["k"], g["v"], a, r, x["frozen"])
        got = saf.saf_attn_fwd_prepared(g["q"], g["k"], g["v"], a, r, x["frozen"], state)
        torch.cuda.synchronize()
        assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1])


def test_prepared_state_of_a_stiff_pattern_uses_the_exact_form(saf):
    # a sink at key 0 and a steep distance penalty push Z' out of the factorised
    # form's range: the prepared state must carry the exact-form flag
    w = custom_workload(1, 3, 600, frozen=(0, 2), slope=0.0)
    x = make_inputs(w, seed=92)
    x["a"][:, 0] = 100.0
    x["r"][:] = -1.0 * torch.arange(600, dtype=torch.float32)
    x["do"] = (x["do"].float() * 0.1).to(x["do"].dtype)
    dev = torch.device("cuda:0")
    g = {n: x[n].to(dev) for n in ("q", "k", "v", "do", "a", "r")}
    state = saf.saf_frozen_prepare(g["a"], g["r"], x["frozen"], w.T, torch.bfloat16)
    o, lse = saf.saf_attn_fwd_prepared(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"], state)
    _, _, dv = saf.saf_attn_bwd_prepared(g["q"], g["k"], g["v"], o, g["do"], lse, g["a"], g["r"], x["frozen"],
                                         state)
    torch.cuda.synchronize()
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    o_ref, _ = oracle.attn_fwd(q, k, v, a, r, x["frozen"])
    _, _, dv_ref = oracle.attn_bwd(q, k, v, do, a, r, x["frozen"])
    assert np.max(np.abs(_np(o) - o_ref)) <= 1e-2
    assert np.max(np.abs(_np(dv) - dv_ref)) <= 2e-2
