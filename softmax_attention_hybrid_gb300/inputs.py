"""Seeded synthetic inputs for the hybrid attention layer.

This module is shared by the fp64 oracle tests and the CUDA path. It holds
workload shapes and random draws only; none of the layer's arithmetic lives
here.

Workloads (shapes from "When Can Attention Heads Be Statically Defined?",
§4 "Model pretraining" and App. C.5: a 124M GPT layer has 12 heads of
dimension 64 at T=4096, the systems runs use B=8; the 1B study runs T=8192):

    tiny          B=1  H=4  F=1 (head 3) T=256   d=64 fp32, q,k,v,dO ~ N(0,1)
    gpt2_124m_25  B=8  H=12 F=3  T=4096  d=64 bf16, q,k,v,dO ~ 0.5 N(0,1)
    gpt2_124m_50  B=8  H=12 F=6  T=4096  d=64 bf16
    1b_25         B=2  H=32 F=8  T=8192  d=64 bf16
    prefill_16k   B=1  H=12 F=3  T=16384 d=64 bf16, forward only
    prefill_b64_4k, prefill_b64_4k_50  B=64 H=12 F=3 / 6 T=4096 d=64 bf16, forward only
    gqa_32q8kv_4k B=4  H=32 (over Hkv=8 key/value heads) F=8 T=4096 d=64 bf16
    gqa_32q8kv_d128 the same at head dimension 128
    1b_d96        B=2  H=16 F=4  T=8192  d=96 bf16

In every workload a[j] ~ N(0,1) (absolute key preference) and
r[δ] = -slope*δ + 0.5 N(0,1) (relative distance preference), one row per
head, fp32, shape [H, T]. The structured-random control of §3.2 draws α, ρ
iid N(0,1) and plugs them into Eq. 3; the slope adds the recency bias that
fitted means show, and keeps the pattern's mass spread over a few hundred
keys.

Which heads are frozen: with F frozen heads out of H, head h is frozen when
h mod (H/F) == H/F - 1. This gives {3} for the tiny layer (its stated frozen
head), {3, 7, 11} for 3 of 12, and every second head for 6 of 12.
"""
from __future__ import annotations

import dataclasses

import torch

__all__ = ["Workload", "WORKLOADS", "frozen_mask", "make_inputs", "make_gqa_inputs", "custom_workload"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    F: int
    T: int
    d: int
    dtype: str          # "fp32" or "bf16": storage and I/O type of q, k, v, o, dO, grads
    scale: float        # std of q, k, v, dO
    slope: float        # r[δ] = -slope*δ + 0.5*N(0,1)
    fwd_only: bool = False
    frozen: tuple | None = None   # explicit frozen head list (overrides the F rule)
    Hkv: int | None = None        # shared key/value heads (grouped-query layout); None: H

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 1, 256, 64, "fp32", 1.0, 0.05),
    "gpt2_124m_25": Workload("gpt2_124m_25", 8, 12, 3, 4096, 64, "bf16", 0.5, 0.02),
    "gpt2_124m_50": Workload("gpt2_124m_50", 8, 12, 6, 4096, 64, "bf16", 0.5, 0.02),
    "1b_25": Workload("1b_25", 2, 32, 8, 8192, 64, "bf16", 0.5, 0.01),
    "prefill_16k": Workload("prefill_16k", 1, 12, 3, 16384, 64, "bf16", 0.5, 0.005, fwd_only=True),
    # batched causal prefill (App. D.3, Table 29: B 64 at 4K, a quarter and a half of the
    # 12 heads replaced), one layer, forward only
    "prefill_b64_4k": Workload("prefill_b64_4k", 64, 12, 3, 4096, 64, "bf16", 0.5, 0.02, fwd_only=True),
    "prefill_b64_4k_50": Workload("prefill_b64_4k_50", 64, 12, 6, 4096, 64, "bf16", 0.5, 0.02, fwd_only=True),
    # 32 query heads over 8 key/value heads (the grouped-query layout of the paper's
    # Qwen3-4B study, App. C.6) at head dimension 64, one frozen query head per group
    "gqa_32q8kv_4k": Workload("gqa_32q8kv_4k", 4, 32, 8, 4096, 64, "bf16", 0.5, 0.02, Hkv=8),
    # the same layout at Qwen3-4B's own head dimension, 128 (App. C.6)
    "gqa_32q8kv_d128": Workload("gqa_32q8kv_d128", 4, 32, 8, 4096, 128, "bf16", 0.5, 0.02, Hkv=8),
    # the paper's 1B layer at its own head dimension (App. C.5: 16 heads of d 96),
    # a quarter of them frozen, at the 8K context of the long-sequence runs
    "1b_d96": Workload("1b_d96", 2, 16, 4, 8192, 96, "bf16", 0.5, 0.01),
}


def custom_workload(B, H, T, d=64, dtype="bf16", frozen=(), scale=0.5, slope=0.02,
                    name="custom", fwd_only=False) -> Workload:
    """A workload with an explicit frozen head list (edge and parity cases)."""
    return Workload(name, B, H, len(frozen), T, d, dtype, scale, slope, fwd_only,
                    tuple(int(h) for h in frozen))


def frozen_mask(w: Workload) -> list[int]:
    """Per-head 0/1 flags, length H."""
    if w.frozen is not None:
        s = set(w.frozen)
        return [1 if h in s else 0 for h in range(w.H)]
    if w.F == 0:
        return [0] * w.H
    if w.H % w.F != 0:
        raise ValueError("F must divide H for the spacing rule")
    g = w.H // w.F
    return [1 if h % g == g - 1 else 0 for h in range(w.H)]


def _normal(shape, seed, stream):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1000003 + stream)
    return torch.randn(shape, generator=g, dtype=torch.float32)


def make_inputs(w: Workload, seed: int = 0, T_prior: int | None = None):
    """Draw every input of workload `w` on the CPU.

    Each tensor comes from its own generator stream, in the fixed order
    q, k, v, dO, a, r-noise, drawn in fp32 and then cast to the workload's
    dtype. a and r stay fp32 and have `T_prior` >= T columns (default T);
    only the first T are used by the layer.

    Returns a dict of CPU tensors: q, k, v, do ([B,H,T,d], workload dtype),
    a, r ([H, T_prior] fp32) and frozen (list of H ints).
    """
    B, H, T, d = w.B, w.H, w.T, w.d
    Tp = T if T_prior is None else int(T_prior)
    if Tp < T:
        raise ValueError("T_prior must be >= T")
    shp = (B, H, T, d)
    q = (_normal(shp, seed, 0) * w.scale).to(w.torch_dtype)
    k = (_normal(shp, seed, 1) * w.scale).to(w.torch_dtype)
    v = (_normal(shp, seed, 2) * w.scale).to(w.torch_dtype)
    do = (_normal(shp, seed, 3) * w.scale).to(w.torch_dtype)
    a = _normal((H, Tp), seed, 4)
    delta = torch.arange(Tp, dtype=torch.float32)
    r = -w.slope * delta[None, :] + 0.5 * _normal((H, Tp), seed, 5)
    if w.Hkv is not None and w.Hkv != H:
        # grouped-query layout: the same draws, k and v cut to their first Hkv heads
        k = k[:, :w.Hkv].contiguous()
        v = v[:, :w.Hkv].contiguous()
    return {"q": q, "k": k, "v": v, "do": do, "a": a.contiguous(), "r": r.contiguous(),
            "frozen": frozen_mask(w)}


def make_gqa_inputs(w: Workload, Hkv: int, seed: int = 0, T_prior: int | None = None):
    """Inputs of a grouped-query layer with w.H query heads over Hkv shared
    key/value heads (w.H a multiple of Hkv): the draws of make_inputs, with k
    and v cut to their first Hkv heads ([B, Hkv, T, d]). q, dO, a, r and the
    frozen flags stay per query head."""
    if Hkv <= 0 or w.H % Hkv != 0:
        raise ValueError("H must be a multiple of Hkv")
    x = make_inputs(w, seed=seed, T_prior=T_prior)
    x["k"] = x["k"][:, :Hkv].contiguous()
    x["v"] = x["v"][:, :Hkv].contiguous()
    return x
