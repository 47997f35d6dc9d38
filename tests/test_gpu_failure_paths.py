"""Failure paths of the step on the GPU, none of which faults or hangs the device.

- Range loss: span matrices keep one power-of-two exponent per row, so an entry more than
  about 2^126 below its row's largest cannot be held.  A step whose span products would drop
  such mass reports FA_ROW_UNDERFLOW (logZ NaN, no tokens, no commits) instead of sampling
  from spans that lost it: the sequence either matches the oracle or says UNDERFLOW, never
  OK with wrong numbers (and never EMPTY for a language with mass).
- Poisoned workspace: with the workspace filled with 0xFF bytes (NaN floats, -1 integers)
  before the step, every output is bit-identical to a run on a zeroed workspace, so no
  scratch word is read before the step writes it.
- Bounded waits: the failure-injection hook makes a tensor-core launch's wait run out (a
  barrier nothing completes, a half-millisecond limit); the step reports FA_ROW_TIMEOUT for
  every sequence and the next ordinary step matches the oracle.
"""
import math

import numpy as np
import pytest

import oracle
from constrained_decoding_diffusion_gb300 import synth
from constrained_decoding_diffusion_gb300.synth import _from_edge_lists

from gpu_util import check_against_oracle, run_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from constrained_decoding_diffusion_gb300 import native as nat
    nat.load()
    return nat


def check_underflow_or_match(fa, o, probs, committed, res, k):
    """Per row: FA_ROW_UNDERFLOW with its documented outputs, or OK and within the oracle's
    tolerances.  Returns the list of statuses."""
    statuses = []
    for b in range(probs.shape[0]):
        st = int(res["status"][b])
        statuses.append(st)
        assert st in (0, 2), (b, st)
        if st == 2:
            assert math.isnan(res["logZ"][b])
            masked = committed[b] < 0
            assert (res["tokens"][b][masked] == -1).all()
            assert (res["marg"][b][masked] == 0).all()
            assert (res["commit"][b] == -1).all()
        else:
            one = {key: v[b:b + 1] for key, v in res.items()}
            check_against_oracle(fa, o, probs[b:b + 1], committed[b:b + 1], one, k)
    return statuses


# --------------------------------------------------------------------------- range loss

def two_speed_fa(n_states: int):
    """State 0 loops on token 0 and moves to state 1 on token 1, which loops on token 1; only
    state 0 accepts, so the one accepted string is all 0s.  States 2.. have no edges (they
    only widen the matrices to the SIMT and tensor-core span paths)."""
    edges = [(0, 0, np.array([0])), (0, 1, np.array([1])), (1, 1, np.array([1]))]
    return _from_edge_lists(n_states, 0, [0], edges, 4)


@pytest.mark.parametrize("S", [2, 100, 128])
def test_range_loss_is_reported_not_sampled(native, S):
    """p(token 0) = 1e-3 and p(token 1) ~ 1: after 16 steps the entry for staying in state 0
    is (1e-3)^16 ~ 2^-159 of its row's largest, below what an fp32 row can hold, and the
    product producing it underflows even though each factor (2^-80) is representable.  The
    exact answer is logZ = 64 ln 1e-3 (about -442); the step must give that or UNDERFLOW,
    never EMPTY."""
    fa = two_speed_fa(S)
    L = 64
    probs = np.zeros((1, L, 4), np.float32)
    probs[0, :, 0] = 1e-3
    probs[0, :, 1] = 1 - 1e-3 - 2e-6
    probs[0, :, 2:] = 1e-6
    committed = np.full((1, L), -1, np.int32)
    o = oracle.OracleFA(fa)
    assert abs(o.posterior(probs[0], committed[0])["logZ"] - L * math.log(probs[0, 0, 0])) < 1e-6
    res = run_step(native.fa_compile(fa), probs, committed, seed=3, offset=0, k=2)
    statuses = check_underflow_or_match(fa, o, probs, committed, res, 2)
    assert statuses == [2], "the dropped mass must be reported"


@pytest.mark.slow
def test_layered_chain_all_masked_reports_range_loss(native):
    """The layered chain with no committed position: span rows spread far beyond 2^126
    (a float64 replay of the span format finds prescaled entries near 2^-1062), so the
    sequence reports UNDERFLOW.  The same automaton with a quarter of the positions committed
    stays inside the range (2^-74 at worst for a prescaled entry times its right row's
    smallest) and reports OK with oracle parity in test_step_layered_chain_full_size."""
    w = synth.workload("layered_chain_S256_L256", B=1)
    probs = w.probs(n_rows=1)
    committed = np.full((1, w.L), -1, np.int32)
    o = oracle.OracleFA(w.fa)
    res = run_step(native.fa_compile(w.fa), probs, committed, seed=7, offset=0, k=w.k)
    check_underflow_or_match(w.fa, o, probs, committed, res, w.k)


# --------------------------------------------------------------------------- poisoned workspace

def _outputs(step):
    return {k: v.cpu().numpy().copy() for k, v in
            dict(tokens=step.tokens, logZ=step.logZ, marg=step.marg, commit=step.commit_idx,
                 status=step.row_status).items()}


def _poison_case(native, fa, probs_np, committed_np, k, method="tree", confidence="marginal", greedy=False):
    import torch
    aut = native.fa_compile(fa)
    B, L, V = probs_np.shape
    probs = torch.from_numpy(probs_np).cuda()
    com = torch.from_numpy(committed_np).cuda()
    runs = []
    for fill in (0x00, 0xFF):
        if greedy:
            step = native.GreedyStep(aut, B, L)
            step.workspace.fill_(fill)
            step(probs, com)
            torch.cuda.synchronize()
            runs.append({k2: v.cpu().numpy().copy() for k2, v in
                         dict(tokens=step.tokens, score=step.score, status=step.row_status).items()})
        else:
            step = native.ConstrainedStep(aut, B, L, k, method=method, confidence=confidence,
                                          want_entropy=confidence == "neg_entropy")
            step.workspace.fill_(fill)
            step(probs, com, 31, 2)
            torch.cuda.synchronize()
            out = _outputs(step)
            if step.entropy is not None:
                out["entropy"] = step.entropy.cpu().numpy().copy()
            runs.append(out)
    clean, poisoned = runs
    for key in clean:
        np.testing.assert_array_equal(poisoned[key], clean[key], err_msg=key)
    return poisoned


POISON_CASES = {
    "real_number_small_span": lambda: synth.workload("real_number_L6", B=3),
    "random_dfa_S64": lambda: synth.workload("random_dfa_S64_L128"),
}


@pytest.mark.parametrize("name", list(POISON_CASES))
def test_poisoned_workspace_tree(native, name):
    w = POISON_CASES[name]()
    probs = w.probs()
    out = _poison_case(native, w.fa, probs, w.committed, w.k)
    check_against_oracle(w.fa, oracle.OracleFA(w.fa), probs, w.committed, out, w.k)


@pytest.mark.parametrize("S", [100, 200])
def test_poisoned_workspace_tiled_and_tensor_core_spans(native, S):
    rng = np.random.default_rng(S + 1)
    fa = synth.random_dfa(S, 3000, 0.8, 12, seed=S + 1)
    L = 24
    probs = synth.gaussian_probs(rng, 2, L, 3000, 3.0)
    committed = np.full((2, L), -1, np.int32)
    x = synth.random_accepted_string(fa, L, rng)
    idx = rng.choice(L, 8, replace=False)
    committed[1, idx] = x[idx]
    out = _poison_case(native, fa, probs, committed, 4)
    check_against_oracle(fa, oracle.OracleFA(fa), probs, committed, out, 4)


def test_poisoned_workspace_chain_entropy_and_greedy(native):
    w = synth.workload("random_dfa_S64_L128")
    probs = w.probs()
    _poison_case(native, w.fa, probs, w.committed, w.k, method="chain")
    _poison_case(native, w.fa, probs, w.committed, w.k, confidence="neg_entropy")
    _poison_case(native, w.fa, probs, w.committed, w.k, greedy=True)


# --------------------------------------------------------------------------- bounded waits

def test_injected_wait_timeout_is_reported_and_recovered(native):
    rng = np.random.default_rng(70)
    fa = synth.random_dfa(128, 3000, 0.8, 12, seed=70)
    o = oracle.OracleFA(fa)
    aut = native.fa_compile(fa)
    L = 16
    probs = synth.gaussian_probs(rng, 2, L, 3000, 3.0)
    committed = np.full((2, L), -1, np.int32)
    x = synth.random_accepted_string(fa, L, rng)
    committed[0, [1, 5]] = x[[1, 5]]
    native.fa_debug_inject_wait_timeouts(1)
    try:
        bad = run_step(aut, probs, committed, seed=4, offset=0, k=3)
    finally:
        native.fa_debug_inject_wait_timeouts(0)
    assert (bad["status"] == 3).all(), bad["status"]
    assert np.all(bad["logZ"] == -np.inf)
    assert (bad["commit"] == -1).all()
    assert (bad["tokens"][committed < 0] == -1).all()
    assert (bad["tokens"][committed >= 0] == committed[committed >= 0]).all()
    # the next ordinary step on the same workspace shape is unaffected
    good = run_step(aut, probs, committed, seed=4, offset=0, k=3)
    assert (good["status"] == 0).all()
    check_against_oracle(fa, o, probs, committed, good, 3)
