"""GPU parity of the chain form of the step (fa_constrained_step_chain): the same
distribution as the tree, reached through O(L)-depth forward messages and
forward-filtering backward-sampling.  Bars as for the tree path: every sampled string
accepted, logZ within 1e-5 * max(1, |logZ|), marginals of the sampled tokens within 1e-5,
commit sets equal outside 1e-5 gaps, chi-square against brute force on tiny cases."""
import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import brute
from constrained_decoding_diffusion_gb300 import synth

from gpu_util import LOGZ_RTOL, check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from constrained_decoding_diffusion_gb300 import native as nat
    nat.load()
    return nat


def run(native, fa, probs, committed, seed, k, method="chain", confidence="marginal"):
    import torch
    B, L, V = probs.shape
    step = native.ConstrainedStep(native.fa_compile(fa), B, L, k, method=method, confidence=confidence)
    p = torch.from_numpy(np.ascontiguousarray(probs)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(committed, np.int32)).cuda()
    step(p, c, seed, 0)
    torch.cuda.synchronize()
    return dict(tokens=step.tokens.cpu().numpy(), logZ=step.logZ.cpu().numpy(), marg=step.marg.cpu().numpy(),
                commit=step.commit_idx.cpu().numpy(), status=step.row_status.cpu().numpy())


def chisq_p(counts, p):
    n = counts.sum()
    exp = p * n
    big = exp >= 5
    obs = np.concatenate([counts[big], [counts[~big].sum()]])
    ex = np.concatenate([exp[big], [exp[~big].sum()]])
    keep = ex > 0
    chi = ((obs[keep] - ex[keep]) ** 2 / ex[keep]).sum()
    return stats.chi2.sf(chi, max(int(keep.sum()) - 1, 1))


@pytest.mark.parametrize("case", ["real", "tiny_nfa", "dup_dfa", "random_dfa", "random_nfa", "S128", "unconstrained"])
def test_chain_matches_oracle(native, case):
    rng = np.random.default_rng(7)
    if case == "real":
        fa, B, L, sigma = synth.real_number_dfa(), 4, 6, 2.0
    elif case == "tiny_nfa":
        fa, B, L, sigma = synth.tiny_random_fa(rng, 5, 7, 14, 4, 2), 4, 9, 1.5
    elif case == "dup_dfa":
        fa, B, L, sigma = synth.random_dfa(12, 40, 0.5, 3, seed=4).duplicated_edges(), 3, 17, 2.0
    elif case == "random_dfa":
        fa, B, L, sigma = synth.random_dfa(64, 3000, 0.7, 8, seed=1), 2, 77, 3.0
    elif case == "random_nfa":
        fa, B, L, sigma = synth.random_nfa(100, 2000, 8, 60, 6, seed=3), 2, 40, 3.0
    elif case == "S128":
        fa, B, L, sigma = synth.random_dfa(128, 1500, 0.8, 8, seed=2), 1, 33, 3.0
    else:
        fa, B, L, sigma = synth.single_state_fa(300), 2, 5, 2.0
    probs = synth.gaussian_probs(rng, B, L, fa.vocab, sigma)
    committed = np.full((B, L), -1, np.int32)
    if case in ("random_dfa", "dup_dfa", "random_nfa"):
        for b in range(B):
            x = synth.random_accepted_string(fa, L, rng)
            pos = rng.choice(L, size=L // 3, replace=False)
            committed[b, pos] = x[pos]
    res = run(native, fa, probs, committed, 13, 4)
    check_against_oracle(fa, oracle.OracleFA(fa), probs, committed, res, 4)
    tree = run(native, fa, probs, committed, 13, 4, method="tree")
    ok = res["status"] == 0
    np.testing.assert_allclose(res["logZ"][ok], tree["logZ"][ok], rtol=2 * LOGZ_RTOL, atol=2 * LOGZ_RTOL)


def test_chain_empty_language(native):
    fa = synth.real_number_dfa()
    probs = np.full((2, 4, 12), 1.0 / 12, np.float32)
    committed = np.full((2, 4), -1, np.int32)
    committed[1, 0] = synth.DOT
    res = run(native, fa, probs, committed, 0, 2)
    assert res["status"].tolist() == [0, 1]
    assert res["logZ"][1] == -np.inf and (res["commit"][1] == -1).all()
    assert (res["tokens"][1, 1:] == -1).all() and res["tokens"][1, 0] == synth.DOT


def test_chain_distribution_matches_brute_force(native):
    import torch
    rng = np.random.default_rng(20)
    fa = synth.tiny_random_fa(rng, 4, 4, 10, 3, 2)
    L, n_batch = 5, 4096
    probs = synth.gaussian_probs(rng, 1, L, 4, 1.0)[0]
    bf = brute.posterior(fa, probs)
    step = native.ConstrainedStep(native.fa_compile(fa), n_batch, L, 0, method="chain")
    p = torch.from_numpy(probs).cuda().expand(n_batch, L, 4).contiguous()
    c = torch.full((n_batch, L), -1, dtype=torch.int32, device="cuda")
    draws = []
    for call in range(10):
        step(p, c, 5, call)
        draws.append(step.tokens.cpu().numpy().copy())
        assert (step.row_status.cpu().numpy() == 0).all()
    idx = brute.string_index(np.concatenate(draws), 4)
    assert (bf["p"][idx] > 0).all()
    counts = np.bincount(idx, minlength=bf["p"].shape[0])
    sup = bf["p"] > 0
    assert chisq_p(counts[sup], bf["p"][sup]) > 1e-3


def test_chain_uniform_over_language(native):
    import torch
    fa = synth.real_number_dfa()
    L, n_batch = 3, 4096
    step = native.ConstrainedStep(native.fa_compile(fa), n_batch, L, 0, method="chain")
    p = torch.full((n_batch, L, 12), 1.0 / 12, dtype=torch.float32, device="cuda")
    c = torch.full((n_batch, L), -1, dtype=torch.int32, device="cuda")
    draws = []
    for call in range(12):
        step(p, c, 9, call)
        draws.append(step.tokens.cpu().numpy().copy())
    draws = np.concatenate(draws)
    strings = brute.all_strings(12, L)
    acc = brute.path_counts(fa, strings) > 0
    idx = brute.string_index(draws, 12)
    assert acc[idx].all()
    counts = np.bincount(idx, minlength=strings.shape[0])[acc]
    assert chisq_p(counts, np.full(1200, 1 / 1200)) > 1e-3


def test_chain_full_workload_rows(native):
    """The block-wise automaton (S=512) at L=64: every row's logZ, sample and marginals."""
    w = synth.workload("blockwise_dfa_S512_L512")
    rng = np.random.default_rng(1)
    B, L = 2, 64
    probs = synth.gaussian_probs(rng, B, L, w.V, 3.0)
    committed = np.full((B, L), -1, np.int32)
    res = run(native, w.fa, probs, committed, 3, 8)
    check_against_oracle(w.fa, oracle.OracleFA(w.fa), probs, committed, res, 8)
