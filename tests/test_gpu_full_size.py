"""GPU parity at the workloads' full sizes, called through the C ABI.

- The SQL-like NFA (|S| = 2048, |V| = 151936, L = 256, all masked): logZ, every position's
  marginal and the commit set against the oracle (the tensor-core span products at their
  largest |S|).
- The same automaton at L = 16: 10^5 draws, every one accepted by the oracle's acceptor,
  and each masked position's token frequencies against the oracle's exact marginals.
- The real-number DFA at its own length L = 6: 10^5 draws, all accepted, and their
  distribution over the 12^6 strings against brute force (chi-square, cells with expected
  count below 5 pooled).
- The block-wise workload's first step (B = 16, L = 512, |S| = 512): every sequence against
  the oracle, in a pool of spawned oracle processes.

The tree is an exact method for the constrained posterior (paperfeed.app summary, "The scan
trick"), so each bar is the oracle's float64 chain result within the stated tolerances."""
import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import brute
from constrained_decoding_diffusion_gb300 import synth

from gpu_util import (check_against_oracle, check_rows_against_refs, oracle_rows_parallel, run_step)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from constrained_decoding_diffusion_gb300 import native as nat
    nat.load()
    return nat


def chisq_p(counts, p):
    """Chi-square p-value of counts against probabilities p, cells with expected count
    below 5 pooled into one."""
    n = counts.sum()
    exp = p * n
    big = exp >= 5
    obs = np.concatenate([counts[big], [counts[~big].sum()]])
    ex = np.concatenate([exp[big], [exp[~big].sum()]])
    keep = ex > 0
    chi = ((obs[keep] - ex[keep]) ** 2 / ex[keep]).sum()
    return stats.chi2.sf(chi, max(int(keep.sum()) - 1, 1))


def draws_of(native, fa, probs_row, committed_row, n_batch, n_calls, seed):
    import torch
    L, V = probs_row.shape
    step = native.ConstrainedStep(native.fa_compile(fa), n_batch, L, 0)
    p = torch.from_numpy(np.ascontiguousarray(probs_row)).cuda().expand(n_batch, L, V).contiguous()
    c = torch.from_numpy(np.ascontiguousarray(committed_row, np.int32)).cuda().expand(n_batch, L).contiguous()
    out = []
    for call in range(n_calls):
        step(p, c, seed, call)
        out.append(step.tokens.cpu().numpy().copy())
        assert (step.row_status.cpu().numpy() == 0).all()
    return np.concatenate(out)


@pytest.mark.slow
def test_nfa_S2048_full_size_parity(native):
    w = synth.workload("random_nfa_S2048_L256")
    probs = w.probs()
    o = oracle.OracleFA(w.fa)
    res = run_step(native.fa_compile(w.fa), probs, w.committed, seed=21, offset=0, k=w.k)
    assert (res["status"] == 0).all()
    check_against_oracle(w.fa, o, probs, w.committed, res, w.k)


@pytest.mark.slow
def test_nfa_S2048_acceptance_and_marginals_1e5_draws(native):
    w = synth.workload("random_nfa_S2048_L256")
    L, n_batch, n_calls = 16, 128, 782
    rng = np.random.default_rng(45)
    probs = synth.gaussian_probs(rng, 1, L, w.V, w.sigma)[0]
    committed = np.full(L, -1, np.int32)
    x = synth.random_accepted_string(w.fa, L, rng)
    committed[[2, 9]] = x[[2, 9]]
    draws = draws_of(native, w.fa, probs, committed, n_batch, n_calls, seed=78)
    assert draws.shape[0] >= 100000
    assert (draws[:, committed >= 0] == committed[committed >= 0]).all()
    o = oracle.OracleFA(w.fa)
    assert all(o.accepts(d) for d in draws)
    ref = o.posterior(probs, committed, want_all=True)["marg_all"]
    masked = np.nonzero(committed < 0)[0]
    pvals = [chisq_p(np.bincount(draws[:, t], minlength=w.V), ref[t]) for t in masked]
    assert min(pvals) > 1e-3 / len(pvals), pvals


@pytest.mark.slow
def test_real_number_L6_1e5_draws_against_brute_force(native):
    w = synth.workload("real_number_L6")
    probs = w.probs()[0]
    com = w.committed[0]
    draws = draws_of(native, w.fa, probs, com, 1000, 100, seed=12)
    assert draws.shape[0] == 100000
    o = oracle.OracleFA(w.fa)
    assert all(o.accepts(d) for d in draws)
    bf = brute.posterior(w.fa, probs)
    idx = brute.string_index(draws, w.V)
    assert (bf["p"][idx] > 0).all()
    counts = np.bincount(idx, minlength=bf["p"].shape[0])
    sup = bf["p"] > 0
    assert chisq_p(counts[sup], bf["p"][sup]) > 1e-3


@pytest.mark.slow
def test_blockwise_first_step_every_sequence(native):
    """The block-wise workload's first step on the device-drawn probabilities of the
    schedule: all 16 sequences' logZ, marginals, acceptance and commit sets (window of the
    first block) against the oracle."""
    import torch
    w = synth.workload("blockwise_dfa_S512_L512")
    aut = native.fa_compile(w.fa)
    probs = synth.gaussian_probs_torch(w.seed * 1000, w.B, w.L, w.V, w.sigma)
    committed = torch.from_numpy(w.committed).cuda()
    step = native.ConstrainedStep(aut, w.B, w.L, w.k)
    step(probs, committed, 5, 0, 0, w.window)
    torch.cuda.synchronize()
    res = dict(tokens=step.tokens.cpu().numpy(), logZ=step.logZ.cpu().numpy(), marg=step.marg.cpu().numpy(),
               commit=step.commit_idx.cpu().numpy(), status=step.row_status.cpu().numpy())
    assert (res["status"] == 0).all()
    host = probs.cpu().numpy()
    del step, probs
    refs = oracle_rows_parallel(w.fa, host, w.committed, res["tokens"], workers=8)
    check_rows_against_refs(refs, res, w.committed, w.k, 0, w.window)
