"""Remasking schedules on the GPU: block-wise decoding with top-k commits by constrained
marginal, checked step by step against the oracle, and the full-size block-wise workload
(|S|=512, |V|=151936, L=512, B=16, 64 steps of k=8)."""
import numpy as np
import pytest

import oracle
from constrained_decoding_diffusion_gb300 import synth

from gpu_util import check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    from constrained_decoding_diffusion_gb300 import native as nat
    nat.load()
    return nat


def test_blockwise_schedule_small(native):
    import torch
    rng = np.random.default_rng(0)
    fa = synth.random_dfa(32, 500, 0.6, 5, seed=3)
    o = oracle.OracleFA(fa)
    aut = native.fa_compile(fa)
    B, L, k, block, spb = 3, 32, 2, 8, 4
    committed = torch.full((B, L), -1, dtype=torch.int32, device="cuda")
    step = native.ConstrainedStep(aut, B, L, k)
    i = 0
    for blk in range(L // block):
        lo, hi = blk * block, (blk + 1) * block
        for _ in range(spb):
            probs = synth.gaussian_probs(rng, B, L, 500, 3.0)
            com_before = committed.cpu().numpy()
            step(torch.from_numpy(probs).cuda(), committed, 11, i, lo, hi)
            torch.cuda.synchronize()
            res = dict(tokens=step.tokens.cpu().numpy(), logZ=step.logZ.cpu().numpy(), marg=step.marg.cpu().numpy(),
                       commit=step.commit_idx.cpu().numpy(), status=step.row_status.cpu().numpy())
            check_against_oracle(fa, o, probs, com_before, res, k, lo, hi)
            native.fa_apply_commits(step.commit_idx, step.tokens, committed)
            i += 1
    final = committed.cpu().numpy()
    assert (final >= 0).all()
    assert all(o.accepts(final[b]) for b in range(B))


@pytest.mark.slow
def test_blockwise_workload_full_size(native):
    """The 64-step block-wise schedule at full size; step 0 of sequence 0 against the oracle,
    every final string accepted."""
    import torch
    from constrained_decoding_diffusion_gb300 import schedule
    w = synth.workload("blockwise_dfa_S512_L512")
    aut = native.fa_compile(w.fa)
    committed = torch.from_numpy(w.committed).cuda()
    first = {}

    def probs_fn(i):
        p = synth.gaussian_probs_torch(w.seed * 1000 + i, w.B, w.L, w.V, w.sigma)
        if i == 0:
            first["probs"] = p[0].cpu().numpy()
        return p

    step = native.ConstrainedStep(aut, w.B, w.L, w.k)
    # step 0 alone, checked on sequence 0
    p0 = probs_fn(0)
    com0 = committed.cpu().numpy()
    step(p0, committed, 5, 0, 0, w.window)
    torch.cuda.synchronize()
    assert (step.row_status.cpu().numpy() == 0).all()
    o = oracle.OracleFA(w.fa)
    res = dict(tokens=step.tokens.cpu().numpy()[:1], logZ=step.logZ.cpu().numpy()[:1], marg=step.marg.cpu().numpy()[:1],
               commit=step.commit_idx.cpu().numpy()[:1], status=step.row_status.cpu().numpy()[:1])
    check_against_oracle(w.fa, o, first["probs"][None], com0[:1], res, w.k, 0, w.window)
    # the whole schedule from the start
    committed = torch.from_numpy(w.committed).cuda()
    schedule.blockwise_schedule(aut, probs_fn, committed, w.k, w.window, 8, seed=5, step=step)
    torch.cuda.synchronize()
    final = committed.cpu().numpy()
    assert (final >= 0).all()
    assert all(o.accepts(final[b]) for b in range(w.B))
