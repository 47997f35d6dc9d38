"""GPU parity: the CUDA path, called through the C ABI, against the float64 oracle.

Bars: compile arrays bit-exact; every sampled string accepted; logZ within
1e-5 * max(1, |logZ|); marginals of the sampled tokens within 1e-5 absolute;
commit sets equal wherever the marginal gap exceeds 1e-5; sample distributions
pass chi-square (p > 0.001) against brute force on tiny cases."""
import math

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import brute
from constrained_decoding_diffusion_gb300 import synth

from gpu_util import check_against_oracle, run_step

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


# --------------------------------------------------------------------------- compile

@pytest.mark.parametrize("which", ["real", "dotted", "tiny_nfa", "dup", "random_dfa_S64", "random_nfa"])
def test_compile_export_bit_exact(native, which):
    rng = np.random.default_rng(0)
    fa = {"real": synth.real_number_dfa, "dotted": synth.dotted_real_dfa,
          "tiny_nfa": lambda: synth.tiny_random_fa(rng, 6, 9, 20, 5, 2),
          "dup": lambda: synth.random_dfa(10, 30, 0.5, 2, seed=3).duplicated_edges(),
          "random_dfa_S64": lambda: synth.random_dfa(64, 32000, 0.7, 8, seed=1),
          "random_nfa": lambda: synth.random_nfa(256, 20000, 16, 200, 8, seed=2)}[which]()
    aut = native.fa_compile(fa)
    got = native.fa_export_csr(aut)
    want = oracle.OracleFA(fa).canonical()
    assert aut.is_dfa == oracle.OracleFA(fa).is_dfa
    for key in want:
        assert np.array_equal(got[key], want[key]), key


def test_compile_rejects_bad_input(native):
    fa = synth.real_number_dfa()
    bad = synth.Automaton(fa.n_states, 9, fa.accept, fa.edge_src, fa.edge_dst, fa.label_offsets, fa.label_tokens,
                          fa.vocab)
    with pytest.raises(native.FaError) as ei:
        native.fa_compile(bad)
    assert ei.value.code == native.FA_ERR_INVALID_ARG
    toks = fa.label_tokens.copy()
    toks[0] = 12
    bad = synth.Automaton(fa.n_states, 0, fa.accept, fa.edge_src, fa.edge_dst, fa.label_offsets, toks, fa.vocab)
    with pytest.raises(native.FaError):
        native.fa_compile(bad)


# --------------------------------------------------------------------------- reweight

@pytest.mark.parametrize("which", ["real", "tiny_nfa", "random_dfa_S64"])
def test_transition_matrices(native, which):
    import torch
    rng = np.random.default_rng(1)
    fa = {"real": synth.real_number_dfa, "tiny_nfa": lambda: synth.tiny_random_fa(rng, 7, 11, 25, 6, 2),
          "random_dfa_S64": lambda: synth.random_dfa(64, 32000, 0.7, 8, seed=1)}[which]()
    B, L = 2, 9
    probs = synth.gaussian_probs(rng, B, L, fa.vocab, 3.0)
    committed = np.full((B, L), -1, np.int32)
    committed[0, 2] = int(fa.label_tokens[0])
    committed[1, 5] = int(fa.label_tokens[-1])
    committed[1, 7] = fa.vocab - 1
    aut = native.fa_compile(fa)
    S = fa.n_states
    mant = torch.empty((B, L, S, S), dtype=torch.float32, device="cuda")
    rexp = torch.empty((B, L, S), dtype=torch.int32, device="cuda")
    native.fa_transition_matrices(aut, torch.from_numpy(probs).cuda(), torch.from_numpy(committed).cuda(), mant, rexp)
    M = mant.double().cpu().numpy() * np.exp2(rexp.cpu().numpy().astype(np.float64))[..., None]
    o = oracle.OracleFA(fa)
    for b in range(B):
        for t in range(L):
            ref = o.transition_matrix(probs[b, t], committed[b, t])
            np.testing.assert_allclose(M[b, t], ref, rtol=2e-6, atol=1e-37)


# --------------------------------------------------------------------------- step parity

@pytest.mark.parametrize("seed", range(6))
def test_step_tiny_random(native, seed):
    rng = np.random.default_rng(100 + seed)
    S, V = int(rng.integers(2, 9)), int(rng.integers(3, 12))
    fa = synth.tiny_random_fa(rng, S, V, int(rng.integers(S, 4 * S)), V, int(rng.integers(1, S + 1)))
    o = oracle.OracleFA(fa)
    aut = native.fa_compile(fa)
    for L in (1, 2, 3, 5, 8, 13):
        B = 3
        probs = synth.gaussian_probs(rng, B, L, V, 2.0)
        committed = np.full((B, L), -1, np.int32)
        committed[1, rng.choice(L, (L + 1) // 2, replace=False)] = rng.integers(0, V, (L + 1) // 2)
        k = int(rng.integers(0, L + 1))
        res = run_step(aut, probs, committed, seed=7 + L, offset=seed, k=k)
        check_against_oracle(fa, o, probs, committed, res, k)


def test_step_real_number_workload(native):
    w = synth.workload("real_number_L6")
    o = oracle.OracleFA(w.fa)
    aut = native.fa_compile(w.fa)
    probs = w.probs()
    res = run_step(aut, probs, w.committed, seed=0, offset=0, k=w.k)
    check_against_oracle(w.fa, o, probs, w.committed, res, w.k)


def test_step_random_dfa_S64_workload(native):
    w = synth.workload("random_dfa_S64_L128")
    o = oracle.OracleFA(w.fa)
    aut = native.fa_compile(w.fa)
    probs = w.probs()
    res = run_step(aut, probs, w.committed, seed=1, offset=0, k=w.k)
    check_against_oracle(w.fa, o, probs, w.committed, res, w.k)


def test_step_window_and_ragged_lengths(native):
    """Non-power-of-two lengths (identity padding of the tree) and a commit window."""
    rng = np.random.default_rng(5)
    fa = synth.random_dfa(24, 300, 0.6, 4, seed=9)
    o = oracle.OracleFA(fa)
    aut = native.fa_compile(fa)
    for L in (7, 31, 33, 100):
        probs = synth.gaussian_probs(rng, 2, L, 300, 3.0)
        committed = np.full((2, L), -1, np.int32)
        x = synth.random_accepted_string(fa, L, rng)
        idx = rng.choice(L, L // 3, replace=False)
        committed[0, idx] = x[idx]
        lo, hi = L // 4, L // 4 + max(1, L // 2)
        res = run_step(aut, probs, committed, seed=3, offset=L, k=5, lo=lo, hi=hi)
        check_against_oracle(fa, o, probs, committed, res, 5, lo, hi)


def test_step_nfa_path_counting(native):
    """Duplicated edges: logZ grows by L ln 2 on the GPU too (NFA path counting)."""
    rng = np.random.default_rng(6)
    fa = synth.random_dfa(16, 80, 0.5, 3, seed=2)
    fa2 = fa.duplicated_edges()
    L = 20
    probs = synth.gaussian_probs(rng, 1, L, 80, 2.0)
    committed = np.full((1, L), -1, np.int32)
    r1 = run_step(native.fa_compile(fa), probs, committed, 1, 0, 4)
    r2 = run_step(native.fa_compile(fa2), probs, committed, 1, 0, 4)
    assert abs(r2["logZ"][0] - r1["logZ"][0] - L * math.log(2)) < 1e-5 * abs(r1["logZ"][0])
    check_against_oracle(fa2, oracle.OracleFA(fa2), probs, committed, r2, 4)


# --------------------------------------------------------------------------- distributions

def _many_draws(native, fa, probs_row, committed_row, n_batch, n_calls, seed):
    import torch
    L, V = probs_row.shape
    aut = native.fa_compile(fa)
    step = native.ConstrainedStep(aut, n_batch, L, 0)
    p = torch.from_numpy(np.ascontiguousarray(probs_row)).cuda().expand(n_batch, L, V).contiguous()
    c = torch.from_numpy(np.ascontiguousarray(committed_row, np.int32)).cuda().expand(n_batch, L).contiguous()
    out = []
    for call in range(n_calls):
        step(p, c, seed, call)
        out.append(step.tokens.cpu().numpy().copy())
        assert (step.row_status.cpu().numpy() == 0).all()
    return np.concatenate(out)


def test_sample_distribution_matches_brute_force(native):
    rng = np.random.default_rng(20)
    fa = synth.tiny_random_fa(rng, 4, 4, 10, 3, 2)
    L = 5
    probs = synth.gaussian_probs(rng, 1, L, 4, 1.0)[0]
    committed = np.full(L, -1, np.int32)
    bf = brute.posterior(fa, probs)
    assert bf["Z"] > 0 and (bf["p"] > 0).sum() > 400
    draws = _many_draws(native, fa, probs, committed, 4096, 10, seed=5)
    idx = brute.string_index(draws, 4)
    assert (bf["p"][idx] > 0).all()
    counts = np.bincount(idx, minlength=bf["p"].shape[0])
    sup = bf["p"] > 0
    assert chisq_p(counts[sup], bf["p"][sup]) > 1e-3


def test_uniform_dfa_is_uniform_over_language(native):
    fa = synth.real_number_dfa()
    L = 3
    probs = synth.uniform_probs(1, L, 12)[0]
    draws = _many_draws(native, fa, probs, np.full(L, -1, np.int32), 4096, 12, seed=9)
    strings = brute.all_strings(12, L)
    acc = brute.path_counts(fa, strings) > 0
    idx = brute.string_index(draws, 12)
    assert acc[idx].all()
    counts = np.bincount(idx, minlength=strings.shape[0])[acc]
    assert chisq_p(counts, np.full(1200, 1 / 1200)) > 1e-3


def test_dotdot_never_sampled(native):
    fa = synth.dotted_real_dfa()
    probs = np.full((2, 12), 0.05 / 11, np.float32)
    probs[:, synth.DOT] = 0.5
    probs[:, 1] += 0.45
    draws = _many_draws(native, fa, probs, np.full(2, -1, np.int32), 4096, 5, seed=2)
    assert not np.any((draws[:, 0] == synth.DOT) & (draws[:, 1] == synth.DOT))
    bf = brute.posterior(fa, probs)
    counts = np.bincount(brute.string_index(draws, 12), minlength=144)
    sup = bf["p"] > 0
    assert chisq_p(counts[sup], bf["p"][sup]) > 1e-3


def test_per_position_marginals_random_dfa(native):
    """Large case: each position's sampled-token frequencies against the oracle's marginals."""
    w = synth.workload("random_dfa_S64_L128")
    probs = w.probs()[0]
    com = w.committed[0]
    draws = _many_draws(native, w.fa, probs, com, 1024, 8, seed=4)
    o = oracle.OracleFA(w.fa)
    ref = o.posterior(probs, com, want_all=True)["marg_all"]
    masked = np.nonzero(com < 0)[0]
    pvals = []
    for t in masked[:16]:
        counts = np.bincount(draws[:, t], minlength=w.V)
        pvals.append(chisq_p(counts, ref[t]))
    # a Bonferroni bound over the positions checked
    assert min(pvals) > 1e-3 / len(pvals), pvals


def test_acceptance_1e5_draws(native):
    w = synth.workload("random_dfa_S64_L128")
    probs = w.probs()[0]
    com = np.full(w.L, -1, np.int32)
    draws = _many_draws(native, w.fa, probs, com, 1000, 100, seed=11)
    assert draws.shape[0] == 100000
    o = oracle.OracleFA(w.fa)
    assert all(o.accepts(x) for x in draws)


# --------------------------------------------------------------------------- edge cases

def test_empty_language_row(native):
    fa = synth.real_number_dfa()
    rng = np.random.default_rng(0)
    probs = synth.gaussian_probs(rng, 2, 4, 12, 1.0)
    committed = np.full((2, 4), -1, np.int32)
    committed[1, 0] = synth.DOT           # no valid string starts with '.'
    res = run_step(native.fa_compile(fa), probs, committed, 0, 0, 2)
    assert res["status"].tolist() == [0, 1]
    assert res["logZ"][1] == -np.inf
    assert (res["commit"][1] == -1).all()
    assert (res["tokens"][1, 1:] == -1).all() and res["tokens"][1, 0] == synth.DOT


def test_all_committed(native):
    rng = np.random.default_rng(3)
    fa = synth.random_nfa(20, 100, 4, 30, 3, seed=4)
    o = oracle.OracleFA(fa)
    L = 10
    x = synth.random_accepted_string(fa, L, rng)
    probs = synth.gaussian_probs(rng, 1, L, 100, 2.0)
    res = run_step(native.fa_compile(fa), probs, x[None], 0, 0, 3)
    assert res["tokens"][0].tolist() == x.tolist()
    assert np.all(res["marg"][0] == 1.0)
    assert abs(res["logZ"][0] - math.log(o.path_count(x))) < 1e-6
    assert (res["commit"][0] == -1).all()


def test_length_zero_and_one(native):
    import torch
    fa = synth.real_number_dfa()
    aut = native.fa_compile(fa)
    step = native.ConstrainedStep(aut, 2, 0, 3)
    step(torch.zeros((2, 0, 12), device="cuda"), torch.zeros((2, 0), dtype=torch.int32, device="cuda"), 0)
    assert step.row_status.tolist() == [1, 1]       # s0 is not accepting
    assert (step.commit_idx.cpu().numpy() == -1).all()
    rng = np.random.default_rng(2)
    probs = synth.gaussian_probs(rng, 3, 1, 12, 2.0)
    res = run_step(aut, probs, np.full((3, 1), -1, np.int32), 0, 0, 1)
    check_against_oracle(fa, oracle.OracleFA(fa), probs, np.full((3, 1), -1, np.int32), res, 1)
    assert all(0 <= t <= 9 for t in res["tokens"][:, 0])


def test_workspace_and_argument_errors(native):
    import torch
    fa = synth.real_number_dfa()
    aut = native.fa_compile(fa)
    B, L = 1, 6
    p = torch.full((B, L, 12), 1 / 12, device="cuda")
    c = torch.full((B, L), -1, dtype=torch.int32, device="cuda")
    step = native.ConstrainedStep(aut, B, L, 2)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(native.FaError) as ei:
        native.fa_constrained_step(aut, p, c, 0, 0, 2, 0, L, small, step.tokens, step.logZ, step.marg,
                                   step.commit_idx, step.row_status)
    assert ei.value.code == native.FA_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(native.FaError) as ei:
        native.fa_constrained_step(aut, p, c, 0, 0, 2, 4, 2, step.workspace, step.tokens, step.logZ, step.marg,
                                   step.commit_idx, step.row_status)
    assert ei.value.code == native.FA_ERR_INVALID_ARG


def test_determinism_and_offsets(native):
    w = synth.workload("random_dfa_S64_L128")
    aut = native.fa_compile(w.fa)
    probs = w.probs()
    a = run_step(aut, probs, w.committed, seed=5, offset=3, k=8)
    b = run_step(aut, probs, w.committed, seed=5, offset=3, k=8)
    c = run_step(aut, probs, w.committed, seed=5, offset=4, k=8)
    for key in a:
        assert np.array_equal(a[key], b[key]), key
    assert not np.array_equal(a["tokens"], c["tokens"])
    assert a["logZ"][0] == c["logZ"][0]


# --------------------------------------------------------------------------- larger shapes

def test_step_tiled_span_products(native):
    """|S| = 100: tiled span products with a ragged last tile, and the row shift kernel."""
    rng = np.random.default_rng(8)
    fa = synth.random_dfa(100, 2000, 0.6, 10, seed=8)
    o = oracle.OracleFA(fa)
    aut = native.fa_compile(fa)
    L = 40
    probs = synth.gaussian_probs(rng, 2, L, 2000, 3.0)
    committed = np.full((2, L), -1, np.int32)
    x = synth.random_accepted_string(fa, L, rng)
    idx = rng.choice(L, 10, replace=False)
    committed[1, idx] = x[idx]
    res = run_step(aut, probs, committed, seed=2, offset=0, k=6)
    check_against_oracle(fa, o, probs, committed, res, 6)


def test_step_layered_chain_full_size(native):
    """JSON-schema-like layered chain at full size (B=4, L=256, |S|=256, |V|=151936); the
    oracle checks two of the rows."""
    w = synth.workload("layered_chain_S256_L256")
    o = oracle.OracleFA(w.fa)
    aut = native.fa_compile(w.fa)
    probs = w.probs()
    res = run_step(aut, probs, w.committed, seed=3, offset=0, k=w.k)
    assert (res["status"] == 0).all()
    check_against_oracle(w.fa, o, probs, w.committed, res, w.k, rows=[0, 3])
    for b in (1, 2):
        assert o.accepts(res["tokens"][b])


def test_step_long_sequence_global_topk(native):
    """L = 30000 > the shared-memory top-k window: keys go through the workspace."""
    rng = np.random.default_rng(9)
    fa = synth.random_dfa(3, 5, 0.2, 2, seed=1)
    o = oracle.OracleFA(fa)
    L = 30000
    probs = synth.gaussian_probs(rng, 1, L, 5, 1.0)
    committed = np.full((1, L), -1, np.int32)
    res = run_step(native.fa_compile(fa), probs, committed, seed=4, offset=0, k=40)
    check_against_oracle(fa, o, probs, committed, res, 40)


@pytest.mark.parametrize("S", [128, 200, 300, 400, 512])
def test_step_tensor_core_span_products(native, S):
    """|S| >= 128 takes the tcgen05 span products (three bf16 parts per operand, six MMAs per
    16 K-columns) in 128x256 output tiles, walked by the persistent product kernel; 200, 300
    and 400 leave ragged tiles in both directions and a ragged last K step."""
    rng = np.random.default_rng(S)
    fa = synth.random_dfa(S, 3000, 0.8, 12, seed=S)
    o = oracle.OracleFA(fa)
    aut = native.fa_compile(fa)
    L = 24
    probs = synth.gaussian_probs(rng, 2, L, 3000, 3.0)
    committed = np.full((2, L), -1, np.int32)
    x = synth.random_accepted_string(fa, L, rng)
    idx = rng.choice(L, 8, replace=False)
    committed[0, idx] = x[idx]
    res = run_step(aut, probs, committed, seed=5, offset=1, k=4)
    check_against_oracle(fa, o, probs, committed, res, 4)


def test_sequence_results_do_not_depend_on_the_batch(native):
    """Sequence b's draws depend only on the seed, the offset, b and its own inputs: the first
    16 sequences of a batch of 17 and the same 16 run alone give the same midpoints, tokens,
    logZ and marginals; both checked against the oracle."""
    rng = np.random.default_rng(40)
    fa = synth.random_dfa(48, 500, 0.6, 6, seed=40)
    aut = native.fa_compile(fa)
    B, L = 17, 37
    probs = synth.gaussian_probs(rng, B, L, 500, 2.5)
    committed = np.full((B, L), -1, np.int32)
    for b in range(B):
        x = synth.random_accepted_string(fa, L, rng)
        pos = rng.choice(L, size=8, replace=False)
        committed[b, pos] = x[pos]
    whole = run_step(aut, probs, committed, seed=6, offset=2, k=5)
    part = run_step(aut, probs[:16], committed[:16], seed=6, offset=2, k=5)
    np.testing.assert_array_equal(part["status"], whole["status"][:16])
    np.testing.assert_array_equal(part["tokens"], whole["tokens"][:16])
    np.testing.assert_array_equal(part["logZ"], whole["logZ"][:16])
    np.testing.assert_allclose(part["marg"], whole["marg"][:16], rtol=0, atol=1e-6)
    o = oracle.OracleFA(fa)
    check_against_oracle(fa, o, probs[:16], committed[:16], part, 5, rows=[0, 7, 15])
    check_against_oracle(fa, o, probs, committed, whole, 5, rows=[16])


def rare_start_rare_end_fa(n_states: int):
    """State 0 starts; token 0 leads to state 1 and tokens 1-6 to state 2; states 1 and 2 loop
    on every token; state 1 accepts, and state 2 reaches the accepting state 3 only by token 7.
    States 4.. have no edges (they only widen the matrices to the SIMT and tensor-core
    span paths)."""
    from constrained_decoding_diffusion_gb300.synth import _from_edge_lists
    V = 8
    edges = [(0, 1, np.array([0])), (0, 2, np.arange(1, 7)), (1, 1, np.arange(V)), (2, 2, np.arange(V)),
             (2, 3, np.array([7]))]
    return _from_edge_lists(n_states, 0, [1, 3], edges, V)


@pytest.mark.parametrize("S", [4, 100, 200])
def test_messages_keep_states_far_below_the_largest(native, S):
    """p(token 0) = 1e-30 at the first position and p(token 7) = 1e-30 at the last: the two
    accepting paths (a rare start into state 1, a rare end out of state 2) weigh about the
    same, while state 1's forward message and state 2's backward message lie about 2^-100
    below the largest entries of theirs, and state 2's forward weight is the dead end's only
    rival.  Such entries need the exact form of the message products: the step matches the
    oracle on logZ and the marginals, and 64 draws take the rare start at the oracle's rate."""
    fa = rare_start_rare_end_fa(S)
    o = oracle.OracleFA(fa)
    aut = native.fa_compile(fa)
    B, L, V = 64, 24, 8
    rng = np.random.default_rng(S)
    row = synth.gaussian_probs(rng, 1, L, V, 1.0)[0]
    row[0, 0] = 1e-30
    row[L - 1, 7] = 1e-30
    probs = np.ascontiguousarray(np.broadcast_to(row, (B, L, V)), dtype=np.float32)
    committed = np.full((B, L), -1, np.int32)
    res = run_step(aut, probs, committed, seed=11, offset=0, k=4)
    assert (res["status"] == 0).all()
    check_against_oracle(fa, o, probs, committed, res, 4, rows=range(8))
    tok0 = np.zeros(L, np.int32)
    p_a = float(o.posterior(row, committed[0], tokens=tok0)["marg_tokens"][0])  # P(x_0 = token 0)
    assert 0.2 < p_a < 0.8, p_a
    n_a = int((res["tokens"][:, 0] == 0).sum())
    assert abs(n_a - B * p_a) <= 4.5 * math.sqrt(B * p_a * (1 - p_a)), (n_a, B * p_a)


@pytest.mark.parametrize("S", [128, 256])
def test_committed_ranges_functional_spans(native, S):
    """A DFA on the tensor-core path with long committed ranges, as in the later steps of a
    block-wise schedule: spans over committed positions are 0/1 partial functions, composed
    instead of multiplied (level 1 up to the root for an all-committed sequence).  Every row
    matches the oracle: all masked, a committed prefix, a committed suffix with a few holes,
    committed except one position, and all committed."""
    rng = np.random.default_rng(40 + S)
    fa = synth.random_dfa(S, 2000, 0.8, 16, seed=S + 3)
    o = oracle.OracleFA(fa)
    aut = native.fa_compile(fa)
    B, L = 5, 64
    probs = synth.gaussian_probs(rng, B, L, 2000, 3.0)
    committed = np.full((B, L), -1, np.int32)
    for b in range(1, B):
        x = synth.random_accepted_string(fa, L, rng)
        if b == 1:
            committed[b, :40] = x[:40]
        elif b == 2:
            committed[b, 8:] = x[8:]
            committed[b, [20, 33, 50]] = -1
        elif b == 3:
            committed[b] = x
            committed[b, 31] = -1
        else:
            committed[b] = x
    res = run_step(aut, probs, committed, seed=6, offset=2, k=4)
    check_against_oracle(fa, o, probs, committed, res, 4)
