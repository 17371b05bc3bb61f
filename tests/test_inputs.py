"""The synthetic input recipe (softmax_attention_hybrid_gb300/inputs.py): the
stand-in for trained layers' activations that every parity test and the bench
draw from. Shapes, dtypes, distributions, seeding and the frozen-head rule."""
import numpy as np
import pytest
import torch

from softmax_attention_hybrid_gb300.inputs import (WORKLOADS, custom_workload, frozen_mask, make_gqa_inputs,
                                                   make_inputs)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_frozen_heads_are_spread_evenly(name):
    # F of H heads frozen, one in every H / F: heads H/F - 1, 2 H/F - 1, ...
    w = WORKLOADS[name]
    m = frozen_mask(w)
    assert len(m) == w.H and sum(m) == w.F
    if w.F:
        g = w.H // w.F
        assert [h for h in range(w.H) if m[h]] == list(range(g - 1, w.H, g))


def test_explicit_head_lists_win():
    assert frozen_mask(custom_workload(1, 6, 8, frozen=(0, 5))) == [1, 0, 0, 0, 0, 1]
    assert frozen_mask(custom_workload(1, 6, 8)) == [0] * 6


def test_shapes_dtypes_and_prior_length():
    w = custom_workload(2, 3, 40, d=96, frozen=(1,))
    x = make_inputs(w, seed=3, T_prior=64)
    for n in ("q", "k", "v", "do"):
        assert x[n].shape == (2, 3, 40, 96) and x[n].dtype == torch.bfloat16
    for n in ("a", "r"):
        assert x[n].shape == (3, 64) and x[n].dtype == torch.float32
    assert x["frozen"] == [0, 1, 0]
    with pytest.raises(ValueError):
        make_inputs(w, T_prior=39)


def test_draws_are_seeded_and_independent_per_tensor():
    w = custom_workload(1, 2, 64, dtype="fp32", frozen=(1,), scale=1.0)
    x0, x1, y = make_inputs(w, seed=7), make_inputs(w, seed=7), make_inputs(w, seed=8)
    for n in ("q", "k", "v", "do", "a", "r"):
        assert torch.equal(x0[n], x1[n]), n
        assert not torch.equal(x0[n], y[n]), n
    # each tensor has its own stream: no two of them repeat each other's values
    flat = {n: x0[n].flatten()[:64] for n in ("q", "k", "v", "do")}
    for a in flat:
        for b in flat:
            if a < b:
                assert not torch.allclose(flat[a], flat[b]), (a, b)


def test_value_distributions():
    # q, k, v, dO ~ scale * N(0, 1); a ~ N(0, 1); r[h, d] = -slope * d + 0.5 * N(0, 1)
    w = custom_workload(2, 4, 4096, dtype="fp32", frozen=(3,), scale=0.5, slope=0.02)
    x = make_inputs(w, seed=0)
    for n in ("q", "k", "v", "do"):
        t = x[n].double().numpy()
        assert abs(t.mean()) < 0.01 and abs(t.std() - 0.5) < 0.01, n
    a = x["a"].double().numpy()
    assert abs(a.mean()) < 0.05 and abs(a.std() - 1.0) < 0.05
    noise = x["r"].double().numpy() + 0.02 * np.arange(w.T)[None, :]
    assert abs(noise.mean()) < 0.03 and abs(noise.std() - 0.5) < 0.03


def test_grouped_inputs_keep_the_first_key_value_heads():
    w = custom_workload(2, 8, 50, frozen=(1, 5))
    x, xg = make_inputs(w, seed=4), make_gqa_inputs(w, 2, seed=4)
    assert xg["k"].shape == (2, 2, 50, 64) and xg["v"].shape == (2, 2, 50, 64)
    assert torch.equal(xg["k"], x["k"][:, :2]) and torch.equal(xg["v"], x["v"][:, :2])
    for n in ("q", "do", "a", "r"):
        assert torch.equal(xg[n], x[n]), n
    with pytest.raises(ValueError):
        make_gqa_inputs(w, 3)
