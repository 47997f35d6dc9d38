"""Sampling statistics on the NFA workload's automaton (|S| = 2048, |V| = 151936; the
tensor-core span products), at L = 16 so that many draws fit one GPU: 64 sequences x 313
calls = 20032 draws.  Every draw is accepted by the oracle's acceptor, and each masked
position's token frequencies pass a chi-square test against the oracle's exact marginals
(Bonferroni over the positions)."""
import numpy as np
import pytest
from scipy import stats

import oracle
from constrained_decoding_diffusion_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from constrained_decoding_diffusion_gb300 import native as nat
    nat.load()
    return nat


def chisq_p(counts, p):
    n = counts.sum()
    exp = p * n
    big = exp >= 5
    obs = np.concatenate([counts[big], [counts[~big].sum()]])
    ex = np.concatenate([exp[big], [exp[~big].sum()]])
    keep = ex > 0
    chi = ((obs[keep] - ex[keep]) ** 2 / ex[keep]).sum()
    return stats.chi2.sf(chi, max(int(keep.sum()) - 1, 1))


def test_nfa_S2048_acceptance_and_marginals(native):
    import torch
    w = synth.workload("random_nfa_S2048_L256")
    L, n_batch, n_calls = 16, 64, 313
    rng = np.random.default_rng(44)
    probs = synth.gaussian_probs(rng, 1, L, w.V, w.sigma)[0]
    committed = np.full(L, -1, np.int32)
    x = synth.random_accepted_string(w.fa, L, rng)
    committed[[3, 11]] = x[[3, 11]]
    step = native.ConstrainedStep(native.fa_compile(w.fa), n_batch, L, 0)
    p = torch.from_numpy(probs).cuda().expand(n_batch, L, w.V).contiguous()
    c = torch.from_numpy(committed).cuda().expand(n_batch, L).contiguous()
    draws = []
    for call in range(n_calls):
        step(p, c, 77, call)
        draws.append(step.tokens.cpu().numpy().copy())
        assert (step.row_status.cpu().numpy() == 0).all()
    draws = np.concatenate(draws)
    assert draws.shape[0] == n_batch * n_calls
    assert (draws[:, committed >= 0] == committed[committed >= 0]).all()
    o = oracle.OracleFA(w.fa)
    assert all(o.accepts(d) for d in draws)
    ref = o.posterior(probs, committed, want_all=True)["marg_all"]
    masked = np.nonzero(committed < 0)[0]
    pvals = [chisq_p(np.bincount(draws[:, t], minlength=w.V), ref[t]) for t in masked]
    assert min(pvals) > 1e-3 / len(pvals), pvals
