"""Brute-force enumeration of the constrained posterior for tiny cases.

TEST INFRASTRUCTURE ONLY.  Independent of the chain recursion in oracle.c: it
lists every string x in V^L, counts its accepting paths N(x) by stepping a
vector of per-state path counts through the tokens, and forms
q(x) = prod_t w_t(x_t) * N(x) directly (paperfeed.app summary of
"Constrained Decoding for Diffusion Language Models via Efficient Inference
over Finite Automata", section "The insight: the constraint is a hidden Markov
model": the constrained posterior is the mean-field product times the
automaton's path-count distribution).
"""
from __future__ import annotations

import numpy as np


def all_strings(V: int, L: int) -> np.ndarray:
    """Every string of V^L as rows (lexicographic, position 0 most significant)."""
    n = V ** L
    idx = np.arange(n, dtype=np.int64)
    out = np.empty((n, L), dtype=np.int32)
    for t in range(L - 1, -1, -1):
        out[:, t] = idx % V
        idx //= V
    return out


def path_counts(fa, strings: np.ndarray) -> np.ndarray:
    """N(x) for every row of strings."""
    n, L = strings.shape
    cnt = np.zeros((n, fa.n_states), dtype=np.float64)
    cnt[:, fa.start] = 1.0
    member = []
    for e in range(fa.n_edges):
        m = np.zeros(fa.vocab, dtype=bool)
        m[fa.labels(e)] = True
        member.append(m)
    for t in range(L):
        nxt = np.zeros_like(cnt)
        x = strings[:, t]
        for e in range(fa.n_edges):
            hit = member[e][x]
            nxt[:, fa.edge_dst[e]] += cnt[:, fa.edge_src[e]] * hit
        cnt = nxt
    return cnt[:, fa.accept].sum(axis=1)


def posterior(fa, probs: np.ndarray, committed=None) -> dict:
    """Exact Z, the full distribution over V^L and the per-position token marginals."""
    L, V = probs.shape
    strings = all_strings(V, L)
    w = probs.astype(np.float64).copy()
    if committed is not None:
        for t in range(L):
            if committed[t] >= 0:
                w[t] = 0.0
                w[t, committed[t]] = 1.0
    q = np.ones(strings.shape[0], dtype=np.float64)
    for t in range(L):
        q *= w[t, strings[:, t]]
    q *= path_counts(fa, strings)
    Z = q.sum()
    p = q / Z if Z > 0 else q
    marg = np.zeros((L, V), dtype=np.float64)
    for t in range(L):
        marg[t] = np.bincount(strings[:, t], weights=p, minlength=V)
    return dict(Z=Z, logZ=np.log(Z) if Z > 0 else -np.inf, p=p, strings=strings, marg=marg)


def string_index(strings_rows: np.ndarray, V: int) -> np.ndarray:
    """Row index in all_strings(V, L) of each given string."""
    idx = np.zeros(strings_rows.shape[0], dtype=np.int64)
    for t in range(strings_rows.shape[1]):
        idx = idx * V + strings_rows[:, t]
    return idx
