"""GPU parity of greedy (T = 0) constrained decoding (fa_map_step) against the oracle's
max-product chain.  What is unique is compared exactly: the best score within
1e-5 * max(1, |score|); the returned string must be accepted, echo the committed tokens and
attain that score (several strings may share the maximum)."""
import numpy as np
import pytest

import oracle
from constrained_decoding_diffusion_gb300 import synth

pytestmark = pytest.mark.gpu

SCORE_RTOL = 1e-5


@pytest.fixture(scope="module")
def native():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from constrained_decoding_diffusion_gb300 import native as nat
    nat.load()
    return nat


def run(native, fa, probs, committed):
    import torch
    B, L, V = probs.shape
    step = native.GreedyStep(native.fa_compile(fa), B, L)
    p = torch.from_numpy(np.ascontiguousarray(probs)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(committed, np.int32)).cuda()
    step(p, c)
    torch.cuda.synchronize()
    return step.tokens.cpu().numpy(), step.score.cpu().numpy(), step.row_status.cpu().numpy()


def check(fa, probs, committed, tokens, score, status):
    o = oracle.OracleFA(fa)
    for b in range(probs.shape[0]):
        ref, x = oracle.viterbi(fa, probs[b], committed[b])
        if x is None:
            assert status[b] != 0 and score[b] == -np.inf
            assert (tokens[b][committed[b] < 0] == -1).all()
            continue
        assert status[b] == 0, status[b]
        tol = SCORE_RTOL * max(1.0, abs(ref))
        assert abs(score[b] - ref) <= tol, (b, score[b], ref)
        tok = tokens[b]
        assert np.array_equal(tok[committed[b] >= 0], committed[b][committed[b] >= 0])
        assert o.accepts(tok)
        assert abs(oracle.string_log_weight(probs[b], tok, committed[b]) - ref) <= tol


@pytest.mark.parametrize("case", ["real", "dotdot", "tiny_nfa", "dup_dfa", "random_dfa", "random_nfa",
                                  "simt_S100", "S256", "unconstrained", "length1"])
def test_greedy_matches_oracle(native, case):
    rng = np.random.default_rng(3)
    if case == "real":
        fa, B, L, sigma = synth.real_number_dfa(), 4, 6, 2.0
    elif case == "dotdot":
        fa, B, L, sigma = synth.dotted_real_dfa(), 3, 2, 2.0
    elif case == "tiny_nfa":
        fa, B, L, sigma = synth.tiny_random_fa(rng, 5, 7, 14, 4, 2), 4, 9, 1.5
    elif case == "dup_dfa":
        fa, B, L, sigma = synth.random_dfa(12, 40, 0.5, 3, seed=4).duplicated_edges(), 3, 17, 2.0
    elif case == "random_dfa":
        fa, B, L, sigma = synth.random_dfa(64, 3000, 0.7, 8, seed=1), 2, 100, 3.0
    elif case == "random_nfa":
        fa, B, L, sigma = synth.random_nfa(100, 2000, 8, 60, 6, seed=3), 2, 40, 3.0
    elif case == "simt_S100":
        fa, B, L, sigma = synth.random_dfa(100, 1000, 0.7, 6, seed=5), 2, 23, 3.0
    elif case == "S256":
        fa, B, L, sigma = synth.layered_chain(256, 4000, seed=2, size_lo=5, size_hi=200), 1, 300, 4.0
    elif case == "unconstrained":
        fa, B, L, sigma = synth.single_state_fa(300), 2, 5, 2.0
    else:
        fa, B, L, sigma = synth.real_number_dfa(), 3, 1, 2.0
    probs = synth.gaussian_probs(rng, B, L, fa.vocab, sigma)
    committed = np.full((B, L), -1, np.int32)
    if case in ("random_dfa", "dup_dfa", "random_nfa", "S256"):
        for b in range(B):
            x = synth.random_accepted_string(fa, L, rng)
            pos = rng.choice(L, size=L // 4, replace=False)
            committed[b, pos] = x[pos]
    tokens, score, status = run(native, fa, probs, committed)
    check(fa, probs, committed, tokens, score, status)
    if case == "unconstrained":
        np.testing.assert_array_equal(tokens, probs.argmax(axis=2))


def test_greedy_avoids_dotdot(native):
    probs = np.full((1, 2, 12), 0.01, np.float32)
    probs[0, :, synth.DOT] = 0.5
    probs[0, :, 1] = 0.4
    tokens, score, status = run(native, synth.real_number_dfa(), probs, np.full((1, 2), -1, np.int32))
    assert tokens[0].tolist() == [1, 1] and status[0] == 0


def test_greedy_empty_language(native):
    fa = synth.real_number_dfa()
    probs = np.full((2, 3, 12), 1.0 / 12, np.float32)
    committed = np.full((2, 3), -1, np.int32)
    committed[1, 0] = synth.DOT
    tokens, score, status = run(native, fa, probs, committed)
    assert status.tolist() == [0, 1]
    check(fa, probs, committed, tokens, score, status)


def test_greedy_is_deterministic(native):
    rng = np.random.default_rng(9)
    fa = synth.random_dfa(64, 3000, 0.7, 8, seed=1)
    probs = synth.gaussian_probs(rng, 3, 50, fa.vocab, 3.0)
    committed = np.full((3, 50), -1, np.int32)
    a = run(native, fa, probs, committed)
    b = run(native, fa, probs, committed)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
