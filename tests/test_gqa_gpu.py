"""GPU parity of the grouped-query layer (saf_attn_fwd_gqa / saf_attn_bwd_gqa)
against the fp64 oracle (oracle.gqa_fwd / gqa_bwd).

"When Can Attention Heads Be Statically Defined?", §3.3 and App. C.6: query
head h reads key/value head h // (H / Hkv); a frozen query head applies its
own fixed pattern to the shared values and has no query slot. The gradient of
a shared key/value head is the sum over its group; frozen query heads add to
dV only, so a group without an ordinary query head has dK = 0 exactly, and a
frozen query head has dQ = 0 exactly. Tolerances as in the multi-head parity
tests: bf16 o, lse 1e-2 and dq, dk, dv 2e-2; fp32 2e-4.
"""
import numpy as np
import pytest
import torch

import oracle
from softmax_attention_hybrid_gb300.inputs import custom_workload, make_gqa_inputs
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


def _run(saf, x, with_qk=True):
    dev = torch.device("cuda:0")
    g = {n: x[n].to(dev) for n in ("q", "k", "v", "do", "a", "r")}
    q = g["q"] if with_qk else None
    k = g["k"] if with_qk else None
    o, lse = saf.saf_attn_fwd_gqa(q, k, g["v"], g["a"], g["r"], x["frozen"])
    dq = torch.full_like(g["q"], 7.0)   # frozen rows must come back as exact zeros
    dq, dk, dv = saf.saf_attn_bwd_gqa(q, k, g["v"], o, g["do"], lse, g["a"], g["r"], x["frozen"], dq=dq)
    torch.cuda.synchronize()
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def _check(saf, w, Hkv, seed, with_qk=True, case=None):
    x = make_gqa_inputs(w, Hkv, seed=seed)
    out = _run(saf, x, with_qk)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    o_ref, lse_ref = oracle.gqa_fwd(q, k, v, a, r, x["frozen"], threads=8)
    dq, dk, dv = oracle.gqa_bwd(q, k, v, do, a, r, x["frozen"], threads=8)
    tol_o, tol_g = TOL[w.dtype]
    err = {}
    for nm, ref in (("o", o_ref), ("lse", lse_ref), ("dq", dq), ("dk", dk), ("dv", dv)):
        got = _np(out[nm])
        assert np.all(np.isfinite(got)), nm
        err[nm] = float(np.max(np.abs(got - ref)))
    if case:
        _parity_log.record(case, err, {nm: (tol_o if nm in ("o", "lse") else tol_g) for nm in err})
    assert err["o"] <= tol_o and err["lse"] <= tol_o, err
    assert max(err["dq"], err["dk"], err["dv"]) <= tol_g, err
    G = w.H // Hkv
    for h in range(w.H):
        if x["frozen"][h]:
            assert torch.all(out["dq"][:, h] == 0), h
    for hk in range(Hkv):
        if all(x["frozen"][hk * G + gi] for gi in range(G)):
            assert torch.all(out["dk"][:, hk] == 0), hk
    return out, x


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_groups_with_mixed_heads(saf, dtype):
    # 8 query heads over 2 key/value heads: group 0 (heads 0-3) has heads 1 and 3
    # frozen, group 1 (heads 4-7) has head 6 frozen
    w = custom_workload(2, 8, 300, dtype=dtype, frozen=(1, 3, 6), scale=0.5 if dtype == "bf16" else 1.0,
                        slope=0.03)
    _check(saf, w, 2, seed=70, case=f"gqa H8/Hkv2 T300 {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_group_with_every_head_frozen(saf, dtype):
    # group 1 (query heads 2 and 3) is fully frozen: its key gradient is exactly zero
    w = custom_workload(2, 8, 257, dtype=dtype, frozen=(2, 3, 5), scale=0.5 if dtype == "bf16" else 1.0,
                        slope=0.03)
    _check(saf, w, 4, seed=71, case=f"gqa H8/Hkv4 T257 {dtype}")


def test_single_shared_head(saf):
    # multi-query layout: every query head reads one key/value head
    w = custom_workload(1, 4, 129, frozen=(0, 2), slope=0.05)
    _check(saf, w, 1, seed=72, case="gqa H4/Hkv1 T129 bf16")


def test_every_head_frozen_without_qk(saf):
    w = custom_workload(2, 4, 200, frozen=(0, 1, 2, 3), slope=0.05)
    _check(saf, w, 2, seed=73, with_qk=False, case="gqa all frozen, q = k = NULL")


def test_qwen_shaped_group_layout(saf):
    # 32 query heads over 8 key/value heads (the layout of App. C.6), a quarter of
    # the query heads frozen, one sequence of 1024 tokens, head dimension 64
    fz = tuple(h for h in range(32) if h % 4 == 3)
    w = custom_workload(2, 32, 1024, frozen=fz, slope=0.01)
    _check(saf, w, 8, seed=74, case="gqa H32/Hkv8 T1024 bf16")


@pytest.mark.parametrize("d", [96, 128])
def test_groups_at_wide_head_dims(saf, d):
    # the d = 96 / 128 kernels in the grouped layout: 8 query heads over 4 key/value
    # heads, groups {0, 1} and {2, 3} mixed, {4, 5} every head frozen (dK exactly zero),
    # {6, 7} ordinary; T not a multiple of 128
    w = custom_workload(2, 8, 300, d=d, frozen=(1, 3, 4, 5), slope=0.03)
    _check(saf, w, 4, seed=76 + d, case=f"gqa H8/Hkv4 T300 d{d} bf16")


def test_qwen_shaped_groups_at_head_dim_128(saf):
    # Qwen3-4B's layout at its own head dimension (App. C.6): 32 query heads over 8
    # key/value heads, d 128, one frozen query head per group, plus q = k = NULL when
    # every head is frozen
    fz = tuple(h for h in range(32) if h % 4 == 3)
    w = custom_workload(1, 32, 640, d=128, frozen=fz, slope=0.01)
    _check(saf, w, 8, seed=78, case="gqa H32/Hkv8 T640 d128 bf16")
    w = custom_workload(1, 8, 200, d=128, frozen=tuple(range(8)), slope=0.05)
    _check(saf, w, 2, seed=79, with_qk=False, case="gqa d128 all frozen, q = k = NULL")


@pytest.mark.parametrize("d", [64, 128])
def test_maximum_head_count_grouped(saf, d):
    # 256 query heads over 64 key/value heads: one frozen query head in every group,
    # and the last group frozen throughout (its dK exactly zero)
    fz = tuple(h for h in range(256) if h % 4 == 3 or h >= 252)
    w = custom_workload(1, 256, 65, d=d, frozen=fz, slope=0.05)
    _check(saf, w, 64, seed=95 + d, case=f"gqa H256/Hkv64 T65 d{d} bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_one_query_head_per_group_is_the_multi_head_layer(saf, dtype):
    # Hkv = H: the grouped-query entry points compute exactly what saf_attn_fwd /
    # saf_attn_bwd compute (the same kernels on the same inputs)
    w = custom_workload(2, 4, 300, dtype=dtype, frozen=(1,), slope=0.05)
    x = make_gqa_inputs(w, 4, seed=75)
    dev = torch.device("cuda:0")
    g = {n: x[n].to(dev) for n in ("q", "k", "v", "do", "a", "r")}
    o1, l1 = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    o2, l2 = saf.saf_attn_fwd_gqa(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
    b1 = saf.saf_attn_bwd(g["q"], g["k"], g["v"], o1, g["do"], l1, g["a"], g["r"], x["frozen"])
    b2 = saf.saf_attn_bwd_gqa(g["q"], g["k"], g["v"], o2, g["do"], l2, g["a"], g["r"], x["frozen"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(b1[1], b2[1]) and torch.equal(b1[2], b2[2])
    # dQ sums its key-block contributions with floating-point reduce-adds, whose order
    # may differ between runs: one unit in the last place at most
    assert (b1[0].float() - b2[0].float()).abs().max().item() <= TOL[dtype][1]


@pytest.mark.parametrize("name", ["gqa_32q8kv_4k", "gqa_32q8kv_d128"])
def test_full_size_grouped_layer_sampled(saf, name):
    # the grouped-query bench workload (B4, 32 query heads over 8 key/value heads,
    # T 4096, one frozen query head per group) in the launch configuration the
    # benchmark times; two whole groups are compared element by element (every query
    # head of the group, and the group sums dK, dV), the rest of the output is checked
    # for finiteness and exact zeros
    import concurrent.futures as cf
    from softmax_attention_hybrid_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    x = make_inputs(w, seed=0)
    out = _run(saf, x)
    G = w.H // w.Hkv
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    tol_o, tol_g = TOL[w.dtype]
    err = {}
    for b, hk in ((0, 0), (w.B - 1, w.Hkv - 1)):
        k, v = (x[n][b, hk].double().numpy() for n in ("k", "v"))

        def one(h):
            q, do = (x[n][b, h].double().numpy() for n in ("q", "do"))
            fz = bool(x["frozen"][h])
            return h, oracle.head_fwd(q, k, v, a[h], r[h], fz), oracle.head_bwd(q, k, v, do, a[h], r[h], fz)

        dk_ref = np.zeros_like(k)
        dv_ref = np.zeros_like(v)
        with cf.ThreadPoolExecutor(G) as ex:
            for h, (o_ref, lse_ref), (dq_ref, dkh, dvh) in ex.map(one, range(hk * G, hk * G + G)):
                for nm, ref in (("o", o_ref), ("lse", lse_ref), ("dq", dq_ref)):
                    err[nm] = max(err.get(nm, 0.0), float(np.max(np.abs(_np(out[nm][b, h]) - ref))))
                dk_ref += dkh
                dv_ref += dvh
        for nm, ref in (("dk", dk_ref), ("dv", dv_ref)):
            err[nm] = max(err.get(nm, 0.0), float(np.max(np.abs(_np(out[nm][b, hk]) - ref))))
    _parity_log.record(f"{name} (2 groups)", err,
                       {nm: (tol_o if nm in ("o", "lse") else tol_g) for nm in err})
    assert err["o"] <= tol_o and err["lse"] <= tol_o, err
    assert max(err["dq"], err["dk"], err["dv"]) <= tol_g, err
    for nm, t in out.items():
        assert torch.isfinite(t).all(), nm
    fzh = [h for h in range(w.H) if x["frozen"][h]]
    assert torch.all(out["dq"][:, fzh] == 0)
