"""Counted work of the hybrid attention layer (for throughput and roofline).

Convention: causal pairs P = T(T+1)/2 per (batch, head); one contraction over
the head dimension costs 2*P*d FLOP.
  ordinary head: forward 2 contractions (Q K^T, P V);
                 backward 5 (S recompute, dV, dP, dQ, dK).
  frozen head:   forward 1 (W V); backward 1 (W^T dO).
Exponentials, normaliser prep and the D_i prep are not counted.

Algorithmic bytes: every tensor the pass must read or write once.
  forward : q, k (ordinary heads), v, o; lse; a, r (frozen heads).
  backward: q, k (ordinary), v, o (ordinary), dO, lse, dq, dk, dv; a, r (frozen).
"""
from __future__ import annotations


def pairs(T: int) -> int:
    return T * (T + 1) // 2


def layer_flops(B, H, F, T, d, backward=True, fwd=True):
    """Counted FLOP of one forward (+ backward) pass with F frozen heads."""
    c = 2 * pairs(T) * d
    ordinary = H - F
    total = 0
    if fwd:
        total += B * (ordinary * 2 + F * 1) * c
    if backward:
        total += B * (ordinary * 5 + F * 1) * c
    return total


def fwd_bytes(B, H, F, T, d, elem):
    od = H - F
    per = T * d * elem
    return B * (od * 2 * per + H * 2 * per + H * T * 4) + F * 2 * T * 4


def bwd_bytes(B, H, F, T, d, elem):
    od = H - F
    per = T * d * elem
    reads = B * (od * 3 * per + H * 2 * per + H * T * 4)      # q, k, o (ordinary); v, dO (all); lse
    writes = B * H * 3 * per                                  # dq, dk, dv
    return reads + writes + F * 2 * T * 4
