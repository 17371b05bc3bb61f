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
