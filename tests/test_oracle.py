"""Pins for the float64 oracle: every check here compares it with something other than
itself (closed forms, Python's regex engine, brute-force enumeration, textbook special
cases and the generator's published test vectors)."""
import math
import os
import re

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import brute
from constrained_decoding_diffusion_gb300 import synth


def chisq_pvalue(observed: np.ndarray, expected_p: np.ndarray) -> float:
    """Pearson chi-square with categories of expected count < 5 pooled together."""
    n = observed.sum()
    exp = expected_p * n
    big = exp >= 5
    obs_b, exp_b = list(observed[big]), list(exp[big])
    if (~big).any():
        obs_b.append(observed[~big].sum())
        exp_b.append(exp[~big].sum())
    obs_b, exp_b = np.array(obs_b, float), np.array(exp_b, float)
    keep = exp_b > 0
    chi = ((obs_b[keep] - exp_b[keep]) ** 2 / exp_b[keep]).sum()
    dof = max(int(keep.sum()) - 1, 1)
    return float(stats.chi2.sf(chi, dof))


def load_language(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "real_number_language.txt")):
        if line.startswith("#") or not line.strip():
            continue
        L, c, lz = line.split()
        rows.append((int(L), int(c), float(lz)))
    return rows


# --------------------------------------------------------------------------- language pins

def test_language_size_by_regex(golden_dir):
    """Python's regex engine counts the real-number language; it must agree with the fixture."""
    pat = re.compile(r"-?[0-9]+(\.[0-9]+)?")
    alphabet = "0123456789.-"
    for L, count, _ in load_language(golden_dir):
        if L > 4:
            continue
        strings = brute.all_strings(12, L)
        n = sum(1 for row in strings if pat.fullmatch("".join(alphabet[i] for i in row)))
        assert n == count


def test_brute_force_path_counts_match_language(golden_dir):
    fa = synth.real_number_dfa()
    for L, count, _ in load_language(golden_dir):
        strings = brute.all_strings(12, L)
        n = brute.path_counts(fa, strings)
        assert set(np.unique(n)) <= {0.0, 1.0}
        assert int(n.sum()) == count


def test_logz_uniform_equals_language_size(golden_dir):
    """DFA with uniform weights: Z * V^L = |C_L| (page 1: p_M is uniform over C for a DFA)."""
    o = oracle.OracleFA(synth.real_number_dfa())
    for L, count, lz_exact in load_language(golden_dir):
        p = synth.uniform_probs(1, L, 12)[0]
        w = float(np.float32(1.0 / 12.0))
        expect = math.log(count) + L * math.log(w)
        got = o.posterior(p)["logZ"]
        assert abs(got - expect) <= 1e-12 * max(1.0, abs(expect))
        # and the fixture's exactly-uniform value differs only by the fp32 rounding of 1/12
        assert abs(got - lz_exact - L * math.log(12.0 * w)) <= 1e-12


def test_uniform_sampling_over_language():
    """Uniform weights + DFA: exact samples are uniform over the 1200 strings of length 3."""
    fa = synth.real_number_dfa()
    o = oracle.OracleFA(fa)
    L = 3
    p = synth.uniform_probs(1, L, 12)[0]
    draws = o.sample(p, None, 60000, seed=11)
    strings = brute.all_strings(12, L)
    acc = brute.path_counts(fa, strings) > 0
    idx = brute.string_index(draws, 12)
    assert acc[idx].all()
    counts = np.bincount(idx, minlength=strings.shape[0])[acc]
    assert counts.shape[0] == 1200
    assert chisq_pvalue(counts, np.full(1200, 1.0 / 1200)) > 1e-3


def test_dotdot_never_sampled_under_constraint():
    """Page 1's example: both "1." and ".1" are valid, ".." is not.  Position-wise
    independent sampling produces ".."; the constrained sampler never does."""
    fa = synth.dotted_real_dfa()
    o = oracle.OracleFA(fa)
    probs = np.full((2, 12), 0.05 / 11, np.float32)
    probs[:, synth.DOT] = 0.5
    probs[0, 1] += 0.45          # position 1 likes '1' or '.', position 2 too
    probs[1, 1] += 0.45
    probs /= probs.sum(axis=1, keepdims=True)
    draws = o.sample(probs, None, 20000, seed=3)
    assert not np.any((draws[:, 0] == synth.DOT) & (draws[:, 1] == synth.DOT))
    assert all(o.accepts(d) for d in draws[:2000])
    rng = np.random.default_rng(5)
    indep = np.stack([rng.choice(12, size=20000, p=probs[t].astype(np.float64) / probs[t].astype(np.float64).sum())
                      for t in range(2)], axis=1)
    rate = np.mean((indep[:, 0] == synth.DOT) & (indep[:, 1] == synth.DOT))
    assert abs(rate - probs[0, synth.DOT] * probs[1, synth.DOT]) < 0.02
    assert rate > 0.2


# --------------------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed", range(8))
def test_matches_brute_force(seed):
    """logZ and every token marginal equal exhaustive enumeration on tiny DFAs and NFAs,
    with parallel edges and committed positions."""
    rng = np.random.default_rng(seed)
    S, V, L = int(rng.integers(2, 6)), int(rng.integers(2, 6)), int(rng.integers(1, 6))
    fa = synth.tiny_random_fa(rng, S, V, n_edges=int(rng.integers(S, 3 * S + 1)), max_label=V,
                              n_accept=int(rng.integers(1, S + 1)))
    o = oracle.OracleFA(fa)
    for trial in range(3):
        probs = synth.gaussian_probs(rng, 1, L, V, 1.5)[0]
        committed = np.full(L, -1, np.int32)
        if trial == 2:
            committed[rng.choice(L, size=(L + 1) // 2, replace=False)] = rng.integers(0, V, size=(L + 1) // 2)
        bf = brute.posterior(fa, probs, committed)
        r = o.posterior(probs, committed, want_all=True)
        if bf["Z"] == 0:
            assert r["empty"] and r["logZ"] == -np.inf
            continue
        assert abs(r["logZ"] - bf["logZ"]) <= 1e-12 * max(1, abs(bf["logZ"]))
        np.testing.assert_allclose(r["marg_all"], bf["marg"], rtol=0, atol=1e-12)


def test_sampler_matches_brute_force_distribution():
    rng = np.random.default_rng(123)
    fa = synth.tiny_random_fa(rng, 4, 3, n_edges=9, max_label=3, n_accept=2)
    o = oracle.OracleFA(fa)
    assert not o.is_dfa
    L = 4
    probs = synth.gaussian_probs(rng, 1, L, 3, 1.0)[0]
    bf = brute.posterior(fa, probs)
    draws = o.sample(probs, None, 50000, seed=9)
    idx = brute.string_index(draws, 3)
    assert (bf["p"][idx] > 0).all()
    counts = np.bincount(idx, minlength=bf["p"].shape[0])
    sup = bf["p"] > 0
    assert chisq_pvalue(counts[sup], bf["p"][sup]) > 1e-3


# --------------------------------------------------------------------------- special cases

def test_single_state_is_unconstrained():
    """One accepting state with a self-loop over V: Z = prod_t sum_v p_t(v) and the
    constrained marginals are the model's own (page 1, the mean-field prediction)."""
    rng = np.random.default_rng(0)
    V, L = 50, 9
    o = oracle.OracleFA(synth.single_state_fa(V))
    probs = synth.gaussian_probs(rng, 1, L, V, 2.0)[0]
    r = o.posterior(probs, want_all=True)
    p64 = probs.astype(np.float64)
    assert abs(r["logZ"] - np.log(p64.sum(axis=1)).sum()) < 1e-12
    np.testing.assert_allclose(r["marg_all"], p64 / p64.sum(axis=1, keepdims=True), atol=1e-14)


def test_entropy_closed_forms_real_number_language():
    """Uniform probabilities over the real-number DFA: at L=1 the accepted strings are the
    ten digits (entropy ln 10); at L=2 they are "-d" and "dd'" (110 strings), so position
    0 is uniform over '-' and the ten digits (ln 11) and position 1 over the ten digits
    (each digit ends 1 + 10 strings: ln 10)."""
    o = oracle.OracleFA(synth.real_number_dfa())
    for L, want in ((1, [math.log(10)]), (2, [math.log(11), math.log(10)])):
        probs = np.full((L, 12), 1.0 / 12, np.float32)
        r = o.posterior(probs, want_all=True)
        np.testing.assert_allclose(oracle.entropy(r["marg_all"]), want, rtol=0, atol=1e-12)
        bf = brute.posterior(synth.real_number_dfa(), probs)
        np.testing.assert_allclose(oracle.entropy(bf["marg"]), want, rtol=0, atol=1e-12)


def test_entropy_unconstrained_is_row_entropy():
    """Single state, self-loop over V: the constrained marginal is p_t itself, so the
    entropy is each row's entropy (scipy.stats.entropy, natural log)."""
    rng = np.random.default_rng(4)
    V, L = 40, 7
    o = oracle.OracleFA(synth.single_state_fa(V))
    probs = synth.gaussian_probs(rng, 1, L, V, 2.0)[0]
    r = o.posterior(probs, want_all=True)
    want = [stats.entropy(probs[t].astype(np.float64)) for t in range(L)]
    np.testing.assert_allclose(oracle.entropy(r["marg_all"]), want, rtol=1e-12, atol=1e-12)


def test_confidence_modes():
    """The three remasking scores: constrained marginal of the sample ("Mar"), minus the
    constrained entropy (Dream), the mean-field probability of the sample ("Mf")."""
    rng = np.random.default_rng(6)
    fa = synth.real_number_dfa()
    o = oracle.OracleFA(fa)
    probs = synth.gaussian_probs(rng, 1, 5, 12, 2.0)[0]
    x = o.sample(probs, None, 1, seed=1)[0]
    r = o.posterior(probs, tokens=x, want_all=True)
    np.testing.assert_array_equal(oracle.confidence("marginal", probs, x, r["marg_tokens"]), r["marg_tokens"])
    np.testing.assert_array_equal(oracle.confidence("unconstrained", probs, x, r["marg_tokens"]),
                                  probs[np.arange(5), x].astype(np.float64))
    h = oracle.confidence("neg_entropy", probs, x, r["marg_tokens"], r["marg_all"])
    assert (h <= 0).all() and (-h <= math.log(12) + 1e-12).all()
    assert (r["marg_tokens"] <= 1 + 1e-12).all()


@pytest.mark.parametrize("seed", range(6))
def test_viterbi_matches_brute_force(seed):
    """The greedy score is the largest mean-field product over the accepted strings, found
    by enumerating V^L; the returned string is accepted and attains it."""
    rng = np.random.default_rng(100 + seed)
    S, V, L = int(rng.integers(2, 6)), int(rng.integers(2, 6)), int(rng.integers(1, 6))
    fa = synth.tiny_random_fa(rng, S, V, n_edges=int(rng.integers(S, 3 * S + 1)), max_label=V,
                              n_accept=int(rng.integers(1, S + 1)))
    probs = synth.gaussian_probs(rng, 1, L, V, 1.5)[0]
    committed = np.full(L, -1, np.int32)
    if seed % 2:
        committed[rng.choice(L, size=(L + 1) // 2, replace=False)] = rng.integers(0, V, size=(L + 1) // 2)
    strings = brute.all_strings(V, L)
    ok = brute.path_counts(fa, strings) > 0
    for t in range(L):
        if committed[t] >= 0:
            ok &= strings[:, t] == committed[t]
    lw = np.array([oracle.string_log_weight(probs, x, committed) for x in strings])
    score, x = oracle.viterbi(fa, probs, committed)
    if not ok.any() or not np.isfinite(lw[ok]).any():
        assert score == -np.inf and x is None
        return
    best = lw[ok].max()
    assert abs(score - best) <= 1e-12 * max(1.0, abs(best))
    assert oracle.OracleFA(fa).accepts(x)
    assert abs(oracle.string_log_weight(probs, x, committed) - best) <= 1e-12 * max(1.0, abs(best))


def test_viterbi_unconstrained_is_per_position_argmax():
    rng = np.random.default_rng(8)
    V, L = 30, 6
    probs = synth.gaussian_probs(rng, 1, L, V, 2.0)[0]
    score, x = oracle.viterbi(synth.single_state_fa(V), probs)
    np.testing.assert_array_equal(x, probs.argmax(axis=1))
    assert abs(score - np.log(probs.max(axis=1).astype(np.float64)).sum()) < 1e-12


def test_viterbi_avoids_dotdot():
    """Real-number DFA, L=2, both positions preferring '.' then '1': "1." and ".." are not
    numbers, so the greedy constrained string is "11"."""
    probs = np.full((2, 12), 0.01, np.float32)
    probs[:, synth.DOT] = 0.5
    probs[:, 1] = 0.4
    score, x = oracle.viterbi(synth.real_number_dfa(), probs)
    assert x.tolist() == [1, 1]
    assert abs(score - 2 * math.log(np.float32(0.4))) < 1e-12


def test_duplicated_edges_double_every_path():
    """NFA path counting (page 1, "Arbitrary schedules and NFAs"): duplicating every edge
    multiplies each accepted string's path count by 2^L, so logZ grows by L ln 2 and
    every marginal is unchanged."""
    rng = np.random.default_rng(1)
    fa = synth.random_dfa(12, 40, 0.6, 3, seed=5)
    o, o2 = oracle.OracleFA(fa), oracle.OracleFA(fa.duplicated_edges())
    assert o.is_dfa and not o2.is_dfa
    L = 7
    probs = synth.gaussian_probs(rng, 1, L, 40, 2.0)[0]
    r, r2 = o.posterior(probs, want_all=True), o2.posterior(probs, want_all=True)
    assert abs(r2["logZ"] - r["logZ"] - L * math.log(2)) < 1e-10
    np.testing.assert_allclose(r2["marg_all"], r["marg_all"], atol=1e-12)


def test_marginals_are_distributions():
    rng = np.random.default_rng(2)
    fa = synth.random_nfa(30, 200, 5, 40, 4, seed=2)
    o = oracle.OracleFA(fa)
    L = 16
    probs = synth.gaussian_probs(rng, 1, L, 200, 3.0)[0]
    r = o.posterior(probs, want_all=True, want_states=True)
    np.testing.assert_allclose(r["marg_all"].sum(axis=1), 1.0, atol=1e-12)
    np.testing.assert_allclose(r["state_post"].sum(axis=1), 1.0, atol=1e-12)
    assert r["state_post"][0, fa.start] == pytest.approx(1.0)
    assert r["state_post"][L, ~np.isin(np.arange(30), fa.accept)].max() == 0.0


def test_all_committed_gives_path_count():
    rng = np.random.default_rng(4)
    fa = synth.random_nfa(20, 100, 4, 30, 3, seed=4)
    o = oracle.OracleFA(fa)
    L = 10
    x = synth.random_accepted_string(fa, L, rng)
    probs = synth.gaussian_probs(rng, 1, L, 100, 2.0)[0]
    r = o.posterior(probs, committed=x, tokens=x)
    assert abs(r["logZ"] - math.log(o.path_count(x))) < 1e-12
    np.testing.assert_allclose(r["marg_tokens"], 1.0, atol=1e-12)


def test_committed_token_outside_language_is_empty():
    fa = synth.real_number_dfa()
    o = oracle.OracleFA(fa)
    probs = synth.uniform_probs(1, 3, 12)[0]
    r = o.posterior(probs, committed=np.array([synth.DOT, -1, -1], np.int32))
    assert r["empty"] and r["logZ"] == -np.inf


# --------------------------------------------------------------------------- compile

def test_canonical_compile_invariants():
    rng = np.random.default_rng(7)
    fa = synth.tiny_random_fa(rng, 6, 9, n_edges=15, max_label=5, n_accept=2)
    # add repeated tokens inside a label set: they must be removed
    fa.label_tokens[fa.label_offsets[1] - 1] = fa.label_tokens[fa.label_offsets[0]]
    o = oracle.OracleFA(fa)
    c = o.canonical()
    for e in range(fa.n_edges):
        lab = c["lab_tok"][c["lab_off"][e]:c["lab_off"][e + 1]]
        assert np.array_equal(lab, np.unique(fa.labels(e)))
    keys = [(fa.edge_src[e], fa.edge_dst[e], e) for e in c["src_edges"]]
    assert keys == sorted(keys) and len(set(c["src_edges"])) == fa.n_edges
    keys = [(fa.edge_dst[e], fa.edge_src[e], e) for e in c["dst_edges"]]
    assert keys == sorted(keys)
    inc = sorted((int(v), int(fa.edge_src[e]), int(fa.edge_dst[e]), e)
                 for e in range(fa.n_edges) for v in np.unique(fa.labels(e)))
    got = [(v, int(fa.edge_src[e]), int(fa.edge_dst[e]), int(e))
           for v in range(fa.vocab) for e in c["tok_edges"][c["tok_off"][v]:c["tok_off"][v + 1]]]
    assert got == inc


def test_dfa_flag():
    assert oracle.OracleFA(synth.real_number_dfa()).is_dfa
    assert oracle.OracleFA(synth.random_dfa(16, 64, 0.5, 2, seed=1)).is_dfa
    assert not oracle.OracleFA(synth.random_nfa(16, 64, 4, 20, 2, seed=1)).is_dfa


def test_invalid_automata_rejected():
    fa = synth.real_number_dfa()
    bad = synth.Automaton(fa.n_states, 7, fa.accept, fa.edge_src, fa.edge_dst, fa.label_offsets,
                          fa.label_tokens, fa.vocab)
    with pytest.raises(ValueError):
        oracle.OracleFA(bad)
    offs = fa.label_offsets.copy()
    offs[1] = offs[0]          # empty label set on edge 0
    bad = synth.Automaton(fa.n_states, 0, fa.accept, fa.edge_src, fa.edge_dst, offs, fa.label_tokens, fa.vocab)
    with pytest.raises(ValueError):
        oracle.OracleFA(bad)


# --------------------------------------------------------------------------- commit rule

def test_topk_rule_by_sorting():
    rng = np.random.default_rng(8)
    for _ in range(50):
        L = int(rng.integers(1, 40))
        marg = rng.choice([0.1, 0.5, 0.9, 0.3], size=L)            # many ties
        committed = np.where(rng.random(L) < 0.3, 5, -1).astype(np.int32)
        k = int(rng.integers(0, 10))
        lo = int(rng.integers(0, L))
        hi = int(rng.integers(lo, L + 1))
        got = oracle.topk(marg, committed, k, lo, hi)
        elig = [t for t in range(lo, hi) if committed[t] < 0]
        want = sorted(elig, key=lambda t: (-marg[t], t))[:k]
        want = want + [-1] * (k - len(want))
        assert got.tolist() == want


# --------------------------------------------------------------------------- Philox

def test_philox_known_answers(golden_dir):
    n = 0
    for line in open(os.path.join(golden_dir, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = [int(x, 16) for x in line.split()]
        assert oracle.philox4x32_10(f[0:4], f[4:6]).tolist() == f[6:10]
        n += 1
    assert n == 3


# --------------------------------------------------------------------------- generators

def test_generators_shapes_and_acceptance():
    rng = np.random.default_rng(0)
    fa = synth.layered_chain(40, 2000, seed=1, size_lo=5, size_hi=50)
    o = oracle.OracleFA(fa)
    assert o.is_dfa
    for _ in range(5):
        x = synth.random_accepted_string(fa, 40, rng)
        assert o.accepts(x)
    w = synth.workload("real_number_L6")
    assert w.fa.n_states == 5 and w.fa.n_edges == 7 and w.fa.n_incidences == 52
    p = w.probs()
    assert p.shape == (1, 6, 12) and p.dtype == np.float32
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, atol=1e-6)
