"""The allocation-free forward entry point, saf_attn_fwd_noalloc.

Callers that cannot allocate device memory (no cudaMalloc allowed where they
run, or a host framework that hands them only input and output buffers) use
this entry point instead of saf_attn_fwd: the library supplies the workspace
from a fixed device array. This file checks, through the C ABI, that two
calls in a row give bit-for-bit the outputs of saf_attn_fwd with a
caller-owned workspace (the same kernels run on the same inputs), that those
outputs match the fp64 oracle within the parity tolerances, and that a
problem too large for the fixed array is refused.

Collected last on purpose (file name), and independent of the other tests:
it passes alone in a fresh process and after the rest of the suite.
"""
import ctypes

import pytest
import torch

import numpy as np

import oracle
from softmax_attention_hybrid_gb300.inputs import custom_workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp32": 2e-4}   # the output tolerances of the parity tests


@pytest.fixture(scope="module")
def saf():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from softmax_attention_hybrid_gb300 import saf as mod
    return mod


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc_call(saf, g, frozen, o, lse):
    B, H, T, d = g["v"].shape
    fz = (ctypes.c_uint8 * H)(*frozen)
    dt = saf.SAF_BF16 if g["v"].dtype == torch.bfloat16 else saf.SAF_FP32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return saf.library().saf_attn_fwd_noalloc(_p(g["q"]), _p(g["k"]), _p(g["v"]), _p(g["a"]), _p(g["r"]),
                                              g["a"].shape[1], fz, B, H, T, d, dt, _p(o), _p(lse), stream)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noalloc_forward_matches_workspace_forward(saf, dtype):
    dev = torch.device("cuda:0")
    # two calls in a row with different shapes and head sets: the second one
    # finds the scratch holding the first call's contents
    cases = [custom_workload(2, 6, 513, dtype=dtype, frozen=(1, 4, 5), scale=0.5, slope=0.03),
             custom_workload(3, 4, 200, dtype=dtype, frozen=(0,), scale=0.5, slope=0.05)]
    for i, w in enumerate(cases):
        x = make_inputs(w, seed=40 + i)
        g = {n: x[n].to(dev) for n in ("q", "k", "v", "a", "r")}
        o_ref, lse_ref = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"])
        o = torch.full_like(g["v"], float("nan"))
        lse = torch.full((w.B, w.H, w.T), float("nan"), device=dev)
        st = _noalloc_call(saf, g, x["frozen"], o, lse)
        assert st == saf.SAF_OK, saf.saf_error_string(st)
        torch.cuda.synchronize()
        assert torch.isfinite(o).all() and torch.isfinite(lse).all()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
        if i == 0:
            q, k, v = (x[n].double().numpy() for n in ("q", "k", "v"))
            o_or, lse_or = oracle.attn_fwd(q, k, v, x["a"].double().numpy(), x["r"].double().numpy(), x["frozen"])
            err_o = np.max(np.abs(o.double().cpu().numpy() - o_or))
            err_l = np.max(np.abs(lse.double().cpu().numpy() - lse_or))
            print(f"noalloc {dtype} vs oracle: o {err_o:.2e} lse {err_l:.2e}")
            assert err_o <= TOL[dtype] and err_l <= TOL[dtype]


def test_noalloc_rejects_problems_beyond_its_scratch(saf):
    dev = torch.device("cuda:0")
    # H * T = 4 * 600000 floats of normalisers alone exceed the 8 MiB scratch;
    # the call must fail before touching any buffer, so tiny tensors suffice
    w = custom_workload(1, 4, 8, frozen=(1,))
    x = make_inputs(w, seed=1)
    g = {n: x[n].to(dev) for n in ("q", "k", "v", "a", "r")}
    o = torch.empty_like(g["v"])
    lse = torch.empty((1, 4, 8), device=dev)
    B, H, T, d = 1, 4, 600000, 64
    fz = (ctypes.c_uint8 * H)(0, 1, 0, 0)
    st = saf.library().saf_attn_fwd_noalloc(_p(g["q"]), _p(g["k"]), _p(g["v"]), _p(g["a"]), _p(g["r"]),
                                            T, fz, B, H, T, d, saf.SAF_BF16, _p(o), _p(lse), None)
    assert st == saf.SAF_ESCRATCH
    assert "scratch" in saf.saf_error_string(st)
