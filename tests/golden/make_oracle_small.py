"""Write oracle_small.json: oracle outputs for one small seeded layer.

Calls only oracle/ and the shared input generator. The fixture pins the
oracle against later edits of its arithmetic (a regression pin); the
independent pins are in tests/test_oracle.py.

    python tests/golden/make_oracle_small.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from softmax_attention_hybrid_gb300.inputs import custom_workload, make_inputs  # noqa: E402

W = custom_workload(1, 2, 9, d=4, dtype="fp32", frozen=(1,), scale=1.0, slope=0.1, name="golden")


def compute():
    x = make_inputs(W, seed=0)
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    a, r = x["a"].double().numpy(), x["r"].double().numpy()
    o, lse = oracle.attn_fwd(q, k, v, a, r, x["frozen"])
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, a, r, x["frozen"])
    return {"workload": "B=1 H=2 T=9 d=4 fp32, head 1 frozen, slope 0.1, seed 0",
            "o": o.tolist(), "lse": lse.tolist(), "dq": dq.tolist(), "dk": dk.tolist(),
            "dv": dv.tolist()}


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(compute(), f, indent=1)
