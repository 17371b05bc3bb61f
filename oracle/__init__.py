"""fp64 CPU oracle for the hybrid (ordinary + frozen) causal attention layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package:
only the tests, the smoke check in ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` may call it. It shares no code with the CUDA library.

See ``oracle/saf_oracle.py`` for the definitions and their citations.
"""
from .saf_oracle import (  # noqa: F401
    frozen_logits,
    frozen_pattern,
    log_normaliser,
    ordinary_pattern,
    head_fwd,
    head_bwd,
    attn_fwd,
    attn_bwd,
    pattern_grad,
    attn_pattern_grad,
    attn_pattern_grad_at,
    FIT_STEPS,
    FIT_LR,
    FIT_TOL,
    floor_and_normalise,
    target_marginals,
    target_negentropy,
    fit_loss,
    fit_grad,
    fit_compact,
    fit_kl,
    gqa_fwd,
    gqa_bwd,
)
