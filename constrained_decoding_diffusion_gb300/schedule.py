"""Remasking schedules driven from the host: every step is one fa_constrained_step call and
one fa_apply_commits call, with no host synchronisation inside the loop.

Block-wise decoding (paperfeed.app summary, "Arbitrary schedules and NFAs"; papernotes.org
notes, key design 3): the sequence is split into blocks of `block` positions decoded left
to right, `steps_per_block` steps each, every step committing the `k` masked positions of
the current block with the highest constrained marginal of their sampled token.  The whole
sequence stays inside the constraint at every step.  With block = L it is plain parallel
decoding.
"""
from __future__ import annotations

from typing import Callable, Optional

from . import native


def blockwise_schedule(aut, probs_fn: Callable[[int], "object"], committed, k: int, block: int,
                       steps_per_block: int, seed: int, stream=None, step: Optional[native.ConstrainedStep] = None):
    """Run the schedule in place on `committed` ([B, L] int32 device tensor, -1 = masked).

    probs_fn(i) returns the [B, L, V] fp32 device probabilities of step i (the denoiser's
    prediction).  Returns the ConstrainedStep holding the last step's outputs; the per-step
    Philox offset is the step index."""
    B, L = committed.shape
    if step is None:
        step = native.ConstrainedStep(aut, B, L, k)
    n_blocks = (L + block - 1) // block
    i = 0
    for blk in range(n_blocks):
        lo, hi = blk * block, min(L, (blk + 1) * block)
        for _ in range(steps_per_block):
            step(probs_fn(i), committed, seed, i, lo, hi, stream)
            native.fa_apply_commits(step.commit_idx, step.tokens, committed, stream)
            i += 1
    return step
