"""Seeded synthetic inputs for the finite-automaton constrained denoising step.

This module feeds both the CUDA path and the float64 oracle, so it holds none
of the method's arithmetic.  Automata are built from random choices,
per-position token distributions are a softmax of Gaussian logits (the
stand-in for a diffusion LM's mean-field prediction), and committed positions
are copied from an accepted string found by a random walk that is steered by
plain boolean reachability ("can this state still reach an accepting state in
the steps that remain").  Nothing here weights paths or computes a partition
function.

The five workloads follow the shapes the pages report for this method:
function-call JSON at L=256 (page 2, ablation table), an SQL automaton of
~10k states / ~100k edges (page 1, "Arbitrary schedules and NFAs"), and the
real-number example of page 1, "Why constrained decoding breaks".  The
benchmark datasets and task automata themselves are not available, so these
generators stand in for them.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

DIGITS = list(range(10))
DOT = 10
MINUS = 11
REAL_VOCAB = 12


@dataclasses.dataclass
class Automaton:
    """A DFA or NFA M = (S, V, delta, s0, F) whose edges carry token label sets.

    edge e goes edge_src[e] -> edge_dst[e] and accepts the tokens
    label_tokens[label_offsets[e]:label_offsets[e+1]].
    """

    n_states: int
    start: int
    accept: np.ndarray          # int32 [n_accept]
    edge_src: np.ndarray        # int32 [E]
    edge_dst: np.ndarray        # int32 [E]
    label_offsets: np.ndarray   # int64 [E+1]
    label_tokens: np.ndarray    # int32 [I]
    vocab: int

    @property
    def n_edges(self) -> int:
        return int(self.edge_src.shape[0])

    @property
    def n_incidences(self) -> int:
        return int(self.label_tokens.shape[0])

    def labels(self, e: int) -> np.ndarray:
        return self.label_tokens[self.label_offsets[e]:self.label_offsets[e + 1]]

    def duplicated_edges(self) -> "Automaton":
        """Every edge twice: each accepting path of the original becomes 2^L paths."""
        E = self.n_edges
        lens = np.diff(self.label_offsets)
        offs = np.concatenate([[0], np.cumsum(np.concatenate([lens, lens]))]).astype(np.int64)
        return Automaton(self.n_states, self.start, self.accept.copy(),
                         np.concatenate([self.edge_src, self.edge_src]).astype(np.int32),
                         np.concatenate([self.edge_dst, self.edge_dst]).astype(np.int32),
                         offs, np.concatenate([self.label_tokens, self.label_tokens]).astype(np.int32),
                         self.vocab)


def _from_edge_lists(n_states, start, accept, edges, vocab) -> Automaton:
    """edges: list of (src, dst, token array)."""
    src = np.array([e[0] for e in edges], dtype=np.int32)
    dst = np.array([e[1] for e in edges], dtype=np.int32)
    lens = np.array([len(e[2]) for e in edges], dtype=np.int64)
    offs = np.zeros(len(edges) + 1, dtype=np.int64)
    np.cumsum(lens, out=offs[1:])
    toks = (np.concatenate([np.asarray(e[2], dtype=np.int32) for e in edges])
            if edges else np.zeros(0, np.int32))
    return Automaton(int(n_states), int(start), np.asarray(sorted(accept), dtype=np.int32),
                     src, dst, offs, toks.astype(np.int32), int(vocab))


# --------------------------------------------------------------------------- automata

def real_number_dfa() -> Automaton:
    """-?[0-9]+(\\.[0-9]+)? over the 12-token vocabulary 0-9, '.', '-' (5 states, 7 edges).

    States: 0 start, 1 after '-', 2 integer digits (accepting), 3 after '.',
    4 fraction digits (accepting).
    """
    edges = [
        (0, 2, DIGITS), (0, 1, [MINUS]), (1, 2, DIGITS), (2, 2, DIGITS),
        (2, 3, [DOT]), (3, 4, DIGITS), (4, 4, DIGITS),
    ]
    return _from_edge_lists(5, 0, [2, 4], edges, REAL_VOCAB)


def dotted_real_dfa() -> Automaton:
    """-?([0-9]+\\.?[0-9]*|\\.[0-9]+): both "1." and ".1" are valid length-2 strings, ".." is not.

    This is the real-number example of page 1 ("Why constrained decoding
    breaks") and page 2 (research background).
    States: 0 start, 1 after '-', 2 integer digits (acc), 3 after "d." and its
    digits (acc), 4 after a leading '.', 5 digits after a leading '.' (acc).
    """
    edges = [
        (0, 2, DIGITS), (0, 1, [MINUS]), (0, 4, [DOT]),
        (1, 2, DIGITS), (1, 4, [DOT]),
        (2, 2, DIGITS), (2, 3, [DOT]),
        (3, 3, DIGITS),
        (4, 5, DIGITS), (5, 5, DIGITS),
    ]
    return _from_edge_lists(6, 0, [2, 3, 5], edges, REAL_VOCAB)


def single_state_fa(vocab: int) -> Automaton:
    """One accepting state with a self-loop over the whole vocabulary (no constraint)."""
    return _from_edge_lists(1, 0, [0], [(0, 0, np.arange(vocab))], vocab)


def random_dfa(n_states: int, vocab: int, p_dead: float, n_accept: int, seed: int) -> Automaton:
    """Each (state, token) is dead with probability p_dead, else goes to a uniform random state.

    Edges are the live tokens of one source grouped by destination, so there is
    at most one edge per (src, dst) pair and the automaton is deterministic.
    """
    rng = np.random.default_rng(seed)
    accept = np.sort(rng.choice(n_states, size=n_accept, replace=False))
    srcs, dsts, lens, toks = [], [], [], []
    for s in range(n_states):
        live = np.nonzero(rng.random(vocab) >= p_dead)[0].astype(np.int32)
        d = rng.integers(0, n_states, size=live.shape[0]).astype(np.int32)
        order = np.argsort(d, kind="stable")
        d, live = d[order], live[order]
        u, first, cnt = np.unique(d, return_index=True, return_counts=True)
        srcs.append(np.full(u.shape[0], s, np.int32))
        dsts.append(u.astype(np.int32))
        lens.append(cnt.astype(np.int64))
        toks.append(live)
    lens = np.concatenate(lens)
    offs = np.zeros(lens.shape[0] + 1, np.int64)
    np.cumsum(lens, out=offs[1:])
    return Automaton(n_states, 0, accept.astype(np.int32), np.concatenate(srcs), np.concatenate(dsts),
                     offs, np.concatenate(toks).astype(np.int32), vocab)


def layered_chain(n_states: int, vocab: int, seed: int,
                  size_lo: int = 50, size_hi: int = 5000) -> Automaton:
    """JSON-schema-like layered chain: i->i+1 always, a self-loop ("runs") with p=0.5,
    a skip i->i+j (j in 2..4, "optional fields") with p=0.25, and a padding self-loop on
    the last (only accepting) state.  Label sets are disjoint within a source, with
    log-uniform sizes in [size_lo, size_hi].
    """
    rng = np.random.default_rng(seed)
    last = n_states - 1
    edges = []
    for i in range(n_states):
        outs = []
        if i < last:
            outs.append(i + 1)
            if rng.random() < 0.5:
                outs.append(i)
            if rng.random() < 0.25:
                j = int(rng.integers(2, 5))
                if i + j <= last:
                    outs.append(i + j)
        else:
            outs.append(i)
        sizes = np.exp(rng.uniform(np.log(size_lo), np.log(size_hi), size=len(outs))).astype(np.int64)
        sizes = np.maximum(sizes, 1)
        pool = rng.choice(vocab, size=int(sizes.sum()), replace=False).astype(np.int32)
        pos = 0
        for d, n in zip(outs, sizes):
            edges.append((i, d, np.sort(pool[pos:pos + n])))
            pos += n
    return _from_edge_lists(n_states, 0, [last], edges, vocab)


def random_nfa(n_states: int, vocab: int, out_degree: int, live_tokens: int,
               n_accept: int, seed: int) -> Automaton:
    """SQL-like NFA: each source has out_degree distinct random destinations; it has
    live_tokens random tokens and each is placed in 1-3 of that source's edges, so
    a (state, token) pair can lead to several states.
    """
    rng = np.random.default_rng(seed)
    accept = np.sort(rng.choice(n_states, size=n_accept, replace=False))
    edges = []
    for s in range(n_states):
        dsts = rng.choice(n_states, size=out_degree, replace=False)
        toks = np.sort(rng.choice(vocab, size=live_tokens, replace=False)).astype(np.int32)
        copies = rng.integers(1, 4, size=live_tokens)
        ranks = np.argsort(np.argsort(rng.random((live_tokens, out_degree)), axis=1), axis=1)
        member = ranks < copies[:, None]
        for j in range(out_degree):
            lab = toks[member[:, j]]
            if lab.shape[0] == 0:
                lab = toks[:1]
            edges.append((s, int(dsts[j]), lab))
    return _from_edge_lists(n_states, 0, accept.tolist(), edges, vocab)


def tiny_random_fa(rng: np.random.Generator, n_states: int, vocab: int, n_edges: int,
                   max_label: int, n_accept: int = 1, allow_parallel: bool = True) -> Automaton:
    """Small random DFA/NFA for brute-force checks (parallel edges allowed when asked)."""
    edges = []
    seen = set()
    while len(edges) < n_edges:
        s = int(rng.integers(0, n_states))
        d = int(rng.integers(0, n_states))
        if not allow_parallel and (s, d) in seen:
            continue
        seen.add((s, d))
        k = int(rng.integers(1, max_label + 1))
        edges.append((s, d, np.sort(rng.choice(vocab, size=min(k, vocab), replace=False))))
    accept = rng.choice(n_states, size=n_accept, replace=False).tolist()
    return _from_edge_lists(n_states, 0, accept, edges, vocab)


# --------------------------------------------------------------------------- probabilities

def gaussian_probs(rng: np.random.Generator, B: int, L: int, V: int, sigma: float) -> np.ndarray:
    """probs[b, t, :] = softmax(sigma * N(0, 1) logits), float32, one row per position."""
    out = np.empty((B, L, V), dtype=np.float32)
    for b in range(B):
        x = rng.standard_normal((L, V), dtype=np.float32)
        x *= np.float32(sigma)
        x -= x.max(axis=1, keepdims=True)
        np.exp(x, out=x)
        x /= x.sum(axis=1, keepdims=True, dtype=np.float32)
        out[b] = x
    return out


def uniform_probs(B: int, L: int, V: int) -> np.ndarray:
    return np.full((B, L, V), np.float32(1.0 / V), dtype=np.float32)


def gaussian_probs_torch(seed: int, B: int, L: int, V: int, sigma: float, device="cuda"):
    """Device-side draw of the same recipe (softmax of sigma * N(0,1) logits) for large
    workloads whose per-step redraw would be slow on the host."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((B, L, V), generator=g, device=device, dtype=torch.float32)
    x.mul_(sigma)
    return torch.softmax(x, dim=-1)


# --------------------------------------------------------------------------- committed tokens

def _reach_table(fa: Automaton, L: int) -> np.ndarray:
    """reach[t, s]: state s can still end in an accepting state after L - t more tokens."""
    reach = np.zeros((L + 1, fa.n_states), dtype=bool)
    reach[L, fa.accept] = True
    nonempty = np.diff(fa.label_offsets) > 0
    src, dst = fa.edge_src[nonempty], fa.edge_dst[nonempty]
    for t in range(L, 0, -1):
        ok = reach[t, dst]
        reach[t - 1, src[ok]] = True
    return reach


def random_accepted_string(fa: Automaton, L: int, rng: np.random.Generator) -> np.ndarray:
    """A random accepted string of length L (not uniform over the language): walk from the
    start state, picking uniformly among out-edges whose destination can still reach an
    accepting state in time, then a uniform token of that edge."""
    reach = _reach_table(fa, L)
    if not reach[0, fa.start]:
        raise ValueError("automaton accepts no string of this length")
    order = np.argsort(fa.edge_src, kind="stable")
    bounds = np.searchsorted(fa.edge_src[order], np.arange(fa.n_states + 1))
    s = fa.start
    out = np.empty(L, dtype=np.int32)
    for t in range(1, L + 1):
        cand = order[bounds[s]:bounds[s + 1]]
        cand = cand[reach[t, fa.edge_dst[cand]] & (np.diff(fa.label_offsets)[cand] > 0)]
        e = int(cand[rng.integers(0, cand.shape[0])])
        lab = fa.labels(e)
        out[t - 1] = lab[rng.integers(0, lab.shape[0])]
        s = int(fa.edge_dst[e])
    return out


def committed_from_string(rng: np.random.Generator, string: np.ndarray, n_commit: int) -> np.ndarray:
    """Copy n_commit randomly chosen positions of an accepted string; -1 marks masked."""
    L = string.shape[0]
    out = np.full(L, -1, dtype=np.int32)
    pos = rng.choice(L, size=n_commit, replace=False)
    out[pos] = string[pos]
    return out


# --------------------------------------------------------------------------- named workloads

@dataclasses.dataclass
class Workload:
    name: str
    fa: Automaton
    B: int
    L: int
    sigma: float
    seed: int
    committed: np.ndarray            # int32 [B, L], -1 = masked
    k: int
    window: int                      # commit window length (L = whole sequence)
    steps: int = 1                   # remasking steps in the schedule

    @property
    def V(self) -> int:
        return self.fa.vocab

    @property
    def S(self) -> int:
        return self.fa.n_states

    def probs(self, step: int = 0, n_rows: Optional[int] = None) -> np.ndarray:
        """The workload's probabilities at one remasking step; n_rows keeps only the first
        sequences (the same values as the first rows of the whole batch)."""
        rng = np.random.default_rng([self.seed, 1000 + step])
        nb = self.B if n_rows is None else min(self.B, n_rows)
        return gaussian_probs(rng, nb, self.L, self.V, self.sigma)


WORKLOADS = ("real_number_L6", "random_dfa_S64_L128", "layered_chain_S256_L256",
             "random_nfa_S2048_L256", "blockwise_dfa_S512_L512")


def workload(name: str, B: Optional[int] = None) -> Workload:
    """Build one of the five named workloads (seed = its index).  B overrides the batch
    for sampled parity checks at full L, S and V."""
    if name == "real_number_L6":
        fa = real_number_dfa()
        bb = 1 if B is None else B
        return Workload(name, fa, bb, 6, 2.0, 0, np.full((bb, 6), -1, np.int32), k=2, window=6)
    if name == "random_dfa_S64_L128":
        fa = random_dfa(64, 32000, 0.7, 8, seed=1)
        bb = 1 if B is None else B
        rng = np.random.default_rng([1, 7])
        com = np.stack([committed_from_string(rng, random_accepted_string(fa, 128, rng), 64)
                        for _ in range(bb)])
        return Workload(name, fa, bb, 128, 3.0, 1, com, k=8, window=128)
    if name == "layered_chain_S256_L256":
        fa = layered_chain(256, 151936, seed=2)
        bb = 4 if B is None else B
        rng = np.random.default_rng([2, 7])
        com = np.stack([committed_from_string(rng, random_accepted_string(fa, 256, rng), 64)
                        for _ in range(bb)])
        return Workload(name, fa, bb, 256, 4.0, 2, com, k=16, window=256)
    if name == "random_nfa_S2048_L256":
        fa = random_nfa(2048, 151936, 16, 488, 64, seed=3)
        bb = 1 if B is None else B
        return Workload(name, fa, bb, 256, 3.0, 3, np.full((bb, 256), -1, np.int32), k=16, window=256)
    if name == "blockwise_dfa_S512_L512":
        fa = random_dfa(512, 151936, 0.9, 8, seed=4)
        bb = 16 if B is None else B
        return Workload(name, fa, bb, 512, 3.0, 4, np.full((bb, 512), -1, np.int32), k=8, window=64,
                        steps=64)
    raise KeyError(name)
