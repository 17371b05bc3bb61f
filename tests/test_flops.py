"""The counted-work model behind every TFLOP/s and roofline figure
(softmax_attention_hybrid_gb300/flops.py), pinned by brute force.

Convention: a head's causal pairs (i, j), j <= i; one contraction over the head
dimension costs one multiply-add (2 FLOP) per pair and coordinate. Ordinary
heads run 2 contractions forward (Q K^T, P V) and 5 backward (S again, dV, dP,
dQ, dK); frozen heads run 1 each way (W V; W^T dO). The counts here come from
loops that perform those contractions element by element on tiny shapes and
tally their multiply-adds, not from the formula under test.
"""
import itertools

import numpy as np
import pytest

from softmax_attention_hybrid_gb300 import flops as F


def _causal_contraction_madds(T, d):
    """Multiply-adds of one causal contraction, counted while computing it."""
    rng = np.random.default_rng(0)
    x, y = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    out = np.zeros((T, T))
    n = 0
    for i in range(T):
        for j in range(i + 1):          # causal pairs only
            s = 0.0
            for c in range(d):
                s += x[i, c] * y[j, c]
                n += 1
            out[i, j] = s
    assert np.allclose(np.tril(x @ y.T), out)   # the loop is the contraction it claims to be
    return n


def test_causal_pairs_by_enumeration():
    for T in (1, 2, 5, 17, 128, 129):
        assert F.pairs(T) == sum(1 for i, j in itertools.product(range(T), repeat=2) if j <= i)


@pytest.mark.parametrize("B,H,Fz,T,d", [(1, 1, 0, 5, 3), (2, 3, 1, 7, 4), (1, 4, 4, 6, 2), (3, 2, 1, 1, 8)])
def test_layer_flops_by_counting(B, H, Fz, T, d):
    madds = _causal_contraction_madds(T, d)
    per_slice_fwd = [1 if h < Fz else 2 for h in range(H)]   # frozen heads first: W V; else Q K^T, P V
    per_slice_bwd = [1 if h < Fz else 5 for h in range(H)]
    fwd = B * sum(per_slice_fwd) * 2 * madds
    bwd = B * sum(per_slice_bwd) * 2 * madds
    assert F.layer_flops(B, H, Fz, T, d, backward=False) == fwd
    assert F.layer_flops(B, H, Fz, T, d, backward=True, fwd=False) == bwd
    assert F.layer_flops(B, H, Fz, T, d) == fwd + bwd


def test_ideal_speedups_of_the_quarter_and_half_frozen_layers():
    # 12 heads, T 4096, d 64: all-ordinary work over hybrid work, forward + backward
    full = F.layer_flops(8, 12, 0, 4096, 64)
    assert full / F.layer_flops(8, 12, 3, 4096, 64) == pytest.approx(84 / 69)
    assert full / F.layer_flops(8, 12, 6, 4096, 64) == pytest.approx(84 / 54)
    # the forward-only prefill: 2 contractions per ordinary head, 1 per frozen one
    assert F.layer_flops(1, 12, 0, 16384, 64, backward=False) / F.layer_flops(1, 12, 3, 16384, 64, backward=False) \
        == pytest.approx(24 / 21)


def test_algorithmic_bytes_by_tensor_inventory():
    # forward: q, k of ordinary heads, v, o of every head (elem bytes each value),
    # lse (fp32) of every row, a and r (fp32) of frozen heads
    B, H, Fz, T, d, e = 2, 5, 2, 33, 16, 2
    od = H - Fz
    fwd = (B * od * T * d * e) * 2 + (B * H * T * d * e) * 2 + B * H * T * 4 + Fz * T * 4 * 2
    assert F.fwd_bytes(B, H, Fz, T, d, e) == fwd
    # backward: q, k, o of ordinary heads, v and dO of every head, lse, the three
    # gradients of every head, a and r of frozen heads
    bwd = (B * od * T * d * e) * 3 + (B * H * T * d * e) * 2 + B * H * T * 4 + (B * H * T * d * e) * 3 + Fz * T * 4 * 2
    assert F.bwd_bytes(B, H, Fz, T, d, e) == bwd
