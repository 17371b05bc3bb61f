"""Failure detection of the tensor-core kernels, made to happen without a GPU fault.

Every wait inside the kernels is bounded. When one expires, the kernel records
a timeout in the workspace's error word, its other warps give up, it frees its
tensor memory and returns, so the CUDA context stays usable and
saf_device_status reports SAF_ETIMEOUT. saf_attn_fwd_diag makes a wait run out
on purpose: its producer publishes no work item, so the first wait of every
other role has nothing to wait for, with a limit of 1 ms instead of 2 s.
"""
import time

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


def test_expired_wait_is_reported_and_the_context_recovers(saf):
    w = custom_workload(2, 4, 300, frozen=(1,), slope=0.05)
    x = make_inputs(w, seed=50)
    dev = torch.device("cuda:0")
    g = {n: x[n].to(dev) for n in ("q", "k", "v", "a", "r")}
    ws = saf.alloc_workspace(w.B, w.H, w.T, w.d, torch.bfloat16, False)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    saf.saf_attn_fwd_diag(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"], withhold=1, wait_limit_us=1000,
                          workspace=ws)
    st = saf.saf_device_status(ws)   # waits for the stream
    elapsed = time.perf_counter() - t0
    assert st == saf.SAF_ETIMEOUT, saf.saf_error_string(st)
    assert elapsed < 1.0, elapsed   # the shortened limit, not the 2 s default, ended the waits

    # the context and the workspace are still usable: a normal call passes parity
    o, lse = saf.saf_attn_fwd(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"], workspace=ws)
    assert saf.saf_device_status(ws) == saf.SAF_OK
    q, k, v = (x[n].double().numpy() for n in ("q", "k", "v"))
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, x["a"].double().numpy(), x["r"].double().numpy(), x["frozen"])
    assert np.max(np.abs(o.double().cpu().numpy() - o_ref)) <= 1e-2
    assert np.max(np.abs(lse.double().cpu().numpy() - lse_ref)) <= 1e-2

    # the diagnostic entry point with nothing withheld is the normal forward
    o2, lse2, _ = saf.saf_attn_fwd_diag(g["q"], g["k"], g["v"], g["a"], g["r"], x["frozen"], withhold=0,
                                        wait_limit_us=0, workspace=ws)
    torch.cuda.synchronize()
    assert saf.saf_device_status(ws) == saf.SAF_OK
    assert torch.equal(o2, o) and torch.equal(lse2, lse)
