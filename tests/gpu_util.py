"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and check its
results against the float64 oracle."""
from __future__ import annotations

import numpy as np

import oracle

LOGZ_RTOL = 1e-5      # |dlogZ| <= 1e-5 * max(1, |logZ|)
MARG_ATOL = 1e-5      # constrained marginals, absolute
COMMIT_GAP = 1e-5     # commit sets must agree wherever marginals differ by more than this


def run_step(aut, probs: np.ndarray, committed: np.ndarray, seed: int, offset: int, k: int,
             lo: int = 0, hi=None):
    import torch
    from constrained_decoding_diffusion_gb300 import native
    B, L, V = probs.shape
    step = native.ConstrainedStep(aut, B, L, k)
    p = torch.from_numpy(np.ascontiguousarray(probs)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(committed, np.int32)).cuda()
    step(p, c, seed, offset, lo, L if hi is None else hi)
    torch.cuda.synchronize()
    return dict(tokens=step.tokens.cpu().numpy(), logZ=step.logZ.cpu().numpy(), marg=step.marg.cpu().numpy(),
                commit=step.commit_idx.cpu().numpy(), status=step.row_status.cpu().numpy())


def check_commit(commit: np.ndarray, marg_ref: np.ndarray, committed: np.ndarray, k: int, lo: int, hi: int):
    """commit: the GPU's ranked list for one sequence; marg_ref: the oracle's marginals of the
    GPU's own tokens.  The list must be the top k of the eligible positions wherever the
    marginal gap exceeds COMMIT_GAP."""
    elig = [t for t in range(lo, hi) if committed[t] < 0]
    n = min(k, len(elig))
    got = [int(x) for x in commit[:n]]
    assert all(x == -1 for x in commit[n:]), commit
    assert len(set(got)) == n and all(t in elig for t in got), (got, elig)
    for a, b in zip(got, got[1:]):
        assert marg_ref[a] >= marg_ref[b] - COMMIT_GAP, (a, b, marg_ref[a], marg_ref[b])
    out = [t for t in elig if t not in got]
    if out and got:
        assert min(marg_ref[t] for t in got) >= max(marg_ref[t] for t in out) - COMMIT_GAP


def check_against_oracle(fa, o: "oracle.OracleFA", probs, committed, res, k, lo=0, hi=None, rows=None):
    B, L, V = probs.shape
    hi = L if hi is None else hi
    for b in (range(B) if rows is None else rows):
        ref = o.posterior(probs[b], committed[b], tokens=np.where(res["tokens"][b] >= 0, res["tokens"][b], 0))
        if ref["empty"]:
            assert res["status"][b] == 1 and res["logZ"][b] == -np.inf
            assert (res["commit"][b] == -1).all()
            continue
        assert res["status"][b] == 0, res["status"][b]
        lz, lz_ref = res["logZ"][b], ref["logZ"]
        assert abs(lz - lz_ref) <= LOGZ_RTOL * max(1.0, abs(lz_ref)), (b, lz, lz_ref)
        tok = res["tokens"][b]
        com = committed[b]
        assert np.array_equal(tok[com >= 0], com[com >= 0])
        assert o.accepts(tok), "sampled string rejected"
        np.testing.assert_allclose(res["marg"][b], ref["marg_tokens"], rtol=0, atol=MARG_ATOL)
        if k > 0:
            check_commit(res["commit"][b], ref["marg_tokens"], com, k, lo, hi)


# --------------------------------------------------------------------------- parallel oracle

_WORKER_ORACLE = None


def _worker_init(fa):
    global _WORKER_ORACLE
    _WORKER_ORACLE = oracle.OracleFA(fa)


def _worker_posterior(args):
    probs, committed, tokens = args
    ref = _WORKER_ORACLE.posterior(probs, committed, tokens=np.where(tokens >= 0, tokens, 0))
    return dict(logZ=ref["logZ"], empty=ref["empty"], marg_tokens=ref["marg_tokens"],
                accepts=bool(_WORKER_ORACLE.accepts(tokens)) if (tokens >= 0).all() else False)


def oracle_rows_parallel(fa, probs_rows, committed_rows, token_rows, workers: int = 8):
    """The oracle's posterior (logZ, marginals of the given tokens) and acceptance of each row,
    in a pool of spawned worker processes (spawn: the parent already holds a CUDA context)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    n = len(probs_rows)
    with ctx.Pool(processes=max(1, min(workers, n, mp.cpu_count())), initializer=_worker_init,
                  initargs=(fa,)) as pool:
        return pool.map(_worker_posterior, [(np.ascontiguousarray(probs_rows[i], np.float32),
                                             np.ascontiguousarray(committed_rows[i], np.int32),
                                             np.ascontiguousarray(token_rows[i], np.int32)) for i in range(n)],
                        chunksize=1)


def check_rows_against_refs(refs, res, committed, k, lo, hi):
    """check_against_oracle with the oracle's results computed beforehand (one per row)."""
    for b, ref in enumerate(refs):
        if ref["empty"]:
            assert res["status"][b] == 1 and res["logZ"][b] == -np.inf
            assert (res["commit"][b] == -1).all()
            continue
        assert res["status"][b] == 0, (b, res["status"][b])
        lz, lz_ref = res["logZ"][b], ref["logZ"]
        assert abs(lz - lz_ref) <= LOGZ_RTOL * max(1.0, abs(lz_ref)), (b, lz, lz_ref)
        tok = res["tokens"][b]
        com = committed[b]
        assert np.array_equal(tok[com >= 0], com[com >= 0])
        assert ref["accepts"], "sampled string rejected (row %d)" % b
        np.testing.assert_allclose(res["marg"][b], ref["marg_tokens"], rtol=0, atol=MARG_ATOL)
        if k > 0:
            check_commit(res["commit"][b], ref["marg_tokens"], com, k, lo, hi)
