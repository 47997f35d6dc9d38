"""GPU parity of the full constrained marginals and of the three remasking confidences.

The all-token marginal p(x_t = v) and its entropy come from the prefix/suffix messages
of the step (fa_token_marginals, fa_constrained_step_ex).  Bars: every token's marginal
within 1e-5 absolute of the float64 oracle and each masked row summing to 1 within 1e-5;
entropies within ENT_ATOL * max(1, H) of the oracle's; commit sets equal wherever the
confidence gap exceeds the confidence's tolerance (1e-5 for the constrained marginal,
ENT_ATOL for minus the entropy, exact for the mean-field probability, which the GPU
reads unchanged from probs)."""
import math

import numpy as np
import pytest

import oracle
from constrained_decoding_diffusion_gb300 import synth

from gpu_util import MARG_ATOL, check_against_oracle

pytestmark = pytest.mark.gpu

# Entropy tolerance.  The marginals carry relative errors of about 1e-6 (fp32 span products
# and messages; the normaliser is the sum of the same terms), and H = -sum p ln p moves by at
# most sum_v |dp_v| (|ln p_v| + 1) <= 1e-6 (H + 1), a few 1e-5 for H <= 10.
ENT_ATOL = 1e-4


@pytest.fixture(scope="module")
def native():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from constrained_decoding_diffusion_gb300 import native as nat
    nat.load()
    return nat


def run(native, fa, probs, committed, seed, k, confidence="marginal", lo=0, hi=None):
    import torch
    B, L, V = probs.shape
    step = native.ConstrainedStep(native.fa_compile(fa), B, L, k, confidence=confidence, want_entropy=True)
    p = torch.from_numpy(np.ascontiguousarray(probs)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(committed, np.int32)).cuda()
    step(p, c, seed, 0, lo, L if hi is None else hi)
    marg_all, ent = step.token_marginals(p, c)
    torch.cuda.synchronize()
    return dict(tokens=step.tokens.cpu().numpy(), logZ=step.logZ.cpu().numpy(), marg=step.marg.cpu().numpy(),
                commit=step.commit_idx.cpu().numpy(), status=step.row_status.cpu().numpy(),
                entropy_step=step.entropy.cpu().numpy(), marg_all=marg_all.cpu().numpy(), entropy=ent.cpu().numpy())


def check_commit_by(commit, conf, committed, k, lo, hi, gap):
    elig = [t for t in range(lo, hi) if committed[t] < 0]
    n = min(k, len(elig))
    got = [int(x) for x in commit[:n]]
    assert all(x == -1 for x in commit[n:]), commit
    assert len(set(got)) == n and all(t in elig for t in got), (got, elig)
    for a, b in zip(got, got[1:]):
        assert conf[a] >= conf[b] - gap, (a, b, conf[a], conf[b])
    rest = [t for t in elig if t not in got]
    if rest and got:
        assert min(conf[t] for t in got) >= max(conf[t] for t in rest) - gap


def check_full(fa, probs, committed, res, rows=None):
    o = oracle.OracleFA(fa)
    B, L, V = probs.shape
    for b in (range(B) if rows is None else rows):
        ref = o.posterior(probs[b], committed[b], want_all=True)
        if ref["empty"]:
            assert res["status"][b] == 1
            masked = committed[b] < 0
            assert (res["marg_all"][b][masked] == 0).all() and (res["entropy"][b] == 0).all()
            for t in np.nonzero(~masked)[0]:
                assert res["marg_all"][b, t, committed[b, t]] == 1.0 and res["marg_all"][b, t].sum() == 1.0
            continue
        assert res["status"][b] == 0
        ma = res["marg_all"][b]
        np.testing.assert_allclose(ma, ref["marg_all"], rtol=0, atol=MARG_ATOL)
        masked = committed[b] < 0
        np.testing.assert_allclose(ma[masked].sum(axis=1), 1.0, rtol=0, atol=MARG_ATOL)
        for t in np.nonzero(~masked)[0]:
            assert ma[t, committed[b, t]] == 1.0 and ma[t].sum() == 1.0
        h_ref = oracle.entropy(ref["marg_all"])
        h = res["entropy"][b]
        assert (np.abs(h - h_ref) <= ENT_ATOL * np.maximum(1.0, h_ref)).all(), np.abs(h - h_ref).max()
        assert (h[~masked] == 0).all()
        # the step's own entropy output is the same computation
        np.testing.assert_array_equal(res["entropy_step"][b], h)
        # the marginal of the sampled token is the full marginal at that token
        tok = res["tokens"][b]
        np.testing.assert_allclose(res["marg"][b][masked], ma[masked, tok[masked]], rtol=0, atol=MARG_ATOL)


def test_entropy_closed_form_real_number(native):
    """Uniform probabilities, L=2: position 0 uniform over '-' and the digits (ln 11),
    position 1 over the digits (ln 10)."""
    probs = np.full((1, 2, 12), 1.0 / 12, np.float32)
    res = run(native, synth.real_number_dfa(), probs, np.full((1, 2), -1, np.int32), 5, 1)
    np.testing.assert_allclose(res["entropy"][0], [math.log(11), math.log(10)], rtol=0, atol=1e-5)


@pytest.mark.parametrize("case", ["real", "tiny_nfa", "dup_dfa", "random_dfa", "tensor_core", "unconstrained",
                                  "rare_start_rare_end"])
def test_full_marginals_match_oracle(native, case):
    """rare_start_rare_end (a rare first and a rare last token carry the only two accepting
    paths) puts the normaliser about 2^-100 below the largest message products, so the
    all-token pass takes its exact form there."""
    rng = np.random.default_rng(11)
    if case == "rare_start_rare_end":
        from test_gpu_parity import rare_start_rare_end_fa
        fa, B, L, V = rare_start_rare_end_fa(4), 2, 12, 8
        probs = synth.gaussian_probs(rng, B, L, V, 1.0)
        probs[:, 0, 0] = 1e-30
        probs[:, L - 1, 7] = 1e-30
        committed = np.full((B, L), -1, np.int32)
        res = run(native, fa, probs, committed, 17, 3)
        check_full(fa, probs, committed, res)
        return
    if case == "real":
        fa, B, L, sigma = synth.real_number_dfa(), 3, 6, 2.0
    elif case == "tiny_nfa":
        fa, B, L, sigma = synth.tiny_random_fa(rng, 5, 7, 14, 4, 2), 4, 7, 1.5
    elif case == "dup_dfa":
        fa, B, L, sigma = synth.random_dfa(12, 40, 0.5, 3, seed=4).duplicated_edges(), 2, 9, 2.0
    elif case == "random_dfa":
        fa, B, L, sigma = synth.random_dfa(64, 3000, 0.7, 8, seed=1), 2, 21, 3.0
    elif case == "tensor_core":
        fa, B, L, sigma = synth.random_dfa(128, 1500, 0.8, 8, seed=2), 1, 10, 3.0
    else:
        fa, B, L, sigma = synth.single_state_fa(300), 2, 5, 2.0
    V = fa.vocab
    probs = synth.gaussian_probs(rng, B, L, V, sigma)
    committed = np.full((B, L), -1, np.int32)
    if case in ("random_dfa", "dup_dfa"):
        for b in range(B):
            x = synth.random_accepted_string(fa, L, rng)
            pos = rng.choice(L, size=L // 3, replace=False)
            committed[b, pos] = x[pos]
    res = run(native, fa, probs, committed, 17, 3)
    check_full(fa, probs, committed, res)


def test_empty_language_gives_zero_marginals(native):
    fa = synth.real_number_dfa()
    probs = np.full((2, 3, 12), 1.0 / 12, np.float32)
    committed = np.full((2, 3), -1, np.int32)
    committed[1, 0] = synth.DOT   # no accepted string starts with '.'
    res = run(native, fa, probs, committed, 3, 2)
    assert res["status"].tolist() == [0, 1]
    check_full(fa, probs, committed, res)


@pytest.mark.parametrize("confidence", ["marginal", "neg_entropy", "unconstrained"])
def test_commit_by_confidence(native, confidence):
    """The commit ranks masked positions of the window by the chosen confidence, computed
    by the oracle from the GPU's own sampled tokens."""
    rng = np.random.default_rng(23)
    fa = synth.random_dfa(32, 500, 0.6, 4, seed=5)
    B, L, k, lo, hi = 3, 24, 5, 2, 20
    probs = synth.gaussian_probs(rng, B, L, fa.vocab, 3.0)
    committed = np.full((B, L), -1, np.int32)
    for b in range(B):
        x = synth.random_accepted_string(fa, L, rng)
        pos = rng.choice(L, size=6, replace=False)
        committed[b, pos] = x[pos]
    res = run(native, fa, probs, committed, 29, k, confidence=confidence, lo=lo, hi=hi)
    o = oracle.OracleFA(fa)
    gap = {"marginal": MARG_ATOL, "neg_entropy": ENT_ATOL, "unconstrained": 0.0}[confidence]
    for b in range(B):
        assert res["status"][b] == 0
        tok = res["tokens"][b]
        assert o.accepts(tok)
        ref = o.posterior(probs[b], committed[b], tokens=tok, want_all=True)
        conf = oracle.confidence(confidence, probs[b], tok, ref["marg_tokens"], ref["marg_all"])
        check_commit_by(res["commit"][b], conf, committed[b], k, lo, hi, gap)
    if confidence == "unconstrained":
        # exact: the same fp32 probabilities, ties to the lower position
        for b in range(B):
            elig = [t for t in range(lo, hi) if committed[b, t] < 0]
            want = sorted(elig, key=lambda t: (-float(probs[b, t, res["tokens"][b, t]]), t))[:k]
            assert res["commit"][b].tolist() == want


def test_confidence_does_not_change_the_sample(native):
    """The confidence only reorders the commit: tokens, logZ and marginals are identical."""
    rng = np.random.default_rng(31)
    fa = synth.random_dfa(16, 200, 0.5, 3, seed=6)
    probs = synth.gaussian_probs(rng, 2, 12, fa.vocab, 2.0)
    committed = np.full((2, 12), -1, np.int32)
    outs = [run(native, fa, probs, committed, 41, 4, confidence=c) for c in ("marginal", "neg_entropy", "unconstrained")]
    for r in outs[1:]:
        for key in ("tokens", "logZ", "marg", "status", "entropy"):
            np.testing.assert_array_equal(r[key], outs[0][key])
    check_against_oracle(fa, oracle.OracleFA(fa), probs, committed, outs[0], 4)


def test_full_marginals_wide_vocabulary_blocks(native):
    """4096 positions: the all-token pass takes its widest vocabulary blocks (4096 tokens;
    the small cases above run 1024-token blocks).  Two sequences against the oracle."""
    rng = np.random.default_rng(52)
    fa = synth.random_dfa(16, 5000, 0.6, 4, seed=52)
    B, L = 16, 256
    probs = synth.gaussian_probs(rng, B, L, fa.vocab, 3.0)
    committed = np.full((B, L), -1, np.int32)
    for b in (0, 9):
        x = synth.random_accepted_string(fa, L, rng)
        pos = rng.choice(L, size=40, replace=False)
        committed[b, pos] = x[pos]
    res = run(native, fa, probs, committed, 61, 4)
    check_full(fa, probs, committed, res, rows=[0, 9])
