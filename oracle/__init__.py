"""Float64 CPU oracle for the finite-automaton constrained denoising step.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the CPU-baseline
leg of the benchmark use it; the product path never imports it.  It shares no
code with the CUDA path.

`oracle.c` holds the chain forward-backward, forward-filter/backward-sample
sampler, acceptor, commit rule and Philox4x32-10; `brute.py` enumerates every
string for tiny cases.  Citations are in the C file's header.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

OR_OK, OR_INVALID, OR_NOMEM, OR_EMPTY = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, no target-specific flags)."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_SO)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.or_fa_new.argtypes = [ctypes.c_int, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, P, P, P, P,
                              ctypes.c_int, ctypes.POINTER(P)]
    lib.or_fa_new.restype = ctypes.c_int
    lib.or_fa_free.argtypes = [P]
    lib.or_fa_sizes.argtypes = [P, P, P, P, P]
    lib.or_fa_export.argtypes = [P] * 10
    lib.or_transition_matrix.argtypes = [P, P, i32, P]
    lib.or_transition_matrix.restype = ctypes.c_int
    lib.or_posterior.argtypes = [P, ctypes.c_int, P, P, P, P, P, P, P, P, P]
    lib.or_posterior.restype = ctypes.c_int
    lib.or_sample.argtypes = [P, ctypes.c_int, P, P, ctypes.c_uint64, ctypes.c_int, P]
    lib.or_sample.restype = ctypes.c_int
    lib.or_path_count.argtypes = [P, ctypes.c_int, P]
    lib.or_path_count.restype = ctypes.c_double
    lib.or_topk.argtypes = [ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    lib.or_philox4x32_10.argtypes = [P, P, P]
    _lib = lib
    return lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleFA:
    """The oracle's own compiled view of an automaton (see synth.Automaton for the fields)."""

    def __init__(self, fa):
        lib = _load()
        self._keep = [np.ascontiguousarray(fa.accept, np.int32), np.ascontiguousarray(fa.edge_src, np.int32),
                      np.ascontiguousarray(fa.edge_dst, np.int32), np.ascontiguousarray(fa.label_offsets, np.int64),
                      np.ascontiguousarray(fa.label_tokens, np.int32)]
        acc, src, dst, off, tok = self._keep
        h = ctypes.c_void_p()
        rc = lib.or_fa_new(fa.n_states, fa.start, _p(acc), acc.shape[0], src.shape[0], _p(src), _p(dst),
                           _p(off), _p(tok), fa.vocab, ctypes.byref(h))
        if rc != OR_OK:
            raise ValueError("oracle rejected the automaton (code %d)" % rc)
        self.h = h
        self.S, self.V = fa.n_states, fa.vocab
        e, i, d, na = np.zeros(1, np.int64), np.zeros(1, np.int64), np.zeros(1, np.int32), np.zeros(1, np.int32)
        lib.or_fa_sizes(h, _p(e), _p(i), _p(d), _p(na))
        self.E, self.I, self.is_dfa, self.n_accept = int(e[0]), int(i[0]), bool(d[0]), int(na[0])

    def __del__(self):
        if getattr(self, "h", None) and _lib is not None:
            _lib.or_fa_free(self.h)
            self.h = None

    def canonical(self) -> dict:
        """The canonical compiled arrays (label CSR, by-src, by-dst, token->edge)."""
        E, I, S, V = self.E, self.I, self.S, self.V
        out = dict(lab_off=np.zeros(E + 1, np.int64), lab_tok=np.zeros(max(I, 1), np.int32),
                   src_off=np.zeros(S + 1, np.int32), src_edges=np.zeros(max(E, 1), np.int32),
                   dst_off=np.zeros(S + 1, np.int32), dst_edges=np.zeros(max(E, 1), np.int32),
                   tok_off=np.zeros(V + 1, np.int64), tok_edges=np.zeros(max(I, 1), np.int32),
                   accept=np.zeros(max(self.n_accept, 1), np.int32))
        _lib.or_fa_export(self.h, *[_p(out[k]) for k in ("lab_off", "lab_tok", "src_off", "src_edges", "dst_off",
                                                          "dst_edges", "tok_off", "tok_edges", "accept")])
        out["lab_tok"] = out["lab_tok"][:I]
        out["tok_edges"] = out["tok_edges"][:I]
        out["src_edges"] = out["src_edges"][:E]
        out["dst_edges"] = out["dst_edges"][:E]
        out["accept"] = out["accept"][:self.n_accept]
        return out

    def transition_matrix(self, probs_row: np.ndarray, committed_token: int = -1) -> np.ndarray:
        row = np.ascontiguousarray(probs_row, np.float32)
        M = np.zeros((self.S, self.S), np.float64)
        rc = _lib.or_transition_matrix(self.h, _p(row), int(committed_token), _p(M))
        assert rc == OR_OK
        return M

    def posterior(self, probs: np.ndarray, committed: Optional[np.ndarray] = None,
                  tokens: Optional[np.ndarray] = None, want_all: bool = False,
                  want_states: bool = False, want_messages: bool = False) -> dict:
        """One sequence (probs [L, V]): logZ and the requested marginals / messages."""
        probs = np.ascontiguousarray(probs, np.float32)
        L = probs.shape[0]
        com = None if committed is None else np.ascontiguousarray(committed, np.int32)
        tok = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
        lz = np.zeros(1, np.float64)
        mt = np.zeros(L, np.float64) if tok is not None else None
        ma = np.zeros((L, self.V), np.float64) if want_all else None
        sp = np.zeros((L + 1, self.S), np.float64) if want_states else None
        la = np.zeros((L + 1, self.S), np.float64) if want_messages else None
        lb = np.zeros((L + 1, self.S), np.float64) if want_messages else None
        rc = _lib.or_posterior(self.h, L, _p(probs), _p(com), _p(tok), _p(lz), _p(mt), _p(ma), _p(sp),
                               _p(la), _p(lb))
        if rc not in (OR_OK, OR_EMPTY):
            raise MemoryError("oracle out of memory")
        return dict(logZ=float(lz[0]), empty=(rc == OR_EMPTY), marg_tokens=mt, marg_all=ma,
                    state_post=sp, log_alpha=la, log_beta=lb)

    def sample(self, probs: np.ndarray, committed: Optional[np.ndarray], n: int, seed: int) -> np.ndarray:
        probs = np.ascontiguousarray(probs, np.float32)
        L = probs.shape[0]
        com = None if committed is None else np.ascontiguousarray(committed, np.int32)
        out = np.zeros((n, L), np.int32)
        rc = _lib.or_sample(self.h, L, _p(probs), _p(com), ctypes.c_uint64(seed), n, _p(out))
        if rc == OR_EMPTY:
            raise ValueError("empty constrained distribution")
        assert rc == OR_OK
        return out

    def path_count(self, tokens: np.ndarray) -> float:
        tok = np.ascontiguousarray(tokens, np.int32)
        return float(_lib.or_path_count(self.h, tok.shape[0], _p(tok)))

    def accepts(self, tokens: np.ndarray) -> bool:
        return self.path_count(tokens) > 0.0


def entropy(marg_all: np.ndarray) -> np.ndarray:
    """Entropy in nats of each position's token distribution, H_t = -sum_v p_t(v) ln p_t(v)
    with 0 ln 0 = 0.  Applied to the exact constrained marginals (posterior(want_all=True))
    it is the Dream-style confidence (lowest entropy first) computed from the constrained
    distribution instead of the mean-field one (paperfeed.app summary, "Constrained remasking
    confidence"; papernotes.org notes, key design 3)."""
    p = np.asarray(marg_all, np.float64)
    out = np.zeros(p.shape[:-1], np.float64)
    pos = p > 0.0
    terms = np.zeros_like(p)
    terms[pos] = p[pos] * np.log(p[pos])
    out[...] = -terms.sum(axis=-1)
    return out


def confidence(mode: str, probs: np.ndarray, tokens: np.ndarray, marg_tokens: np.ndarray,
               marg_all: Optional[np.ndarray] = None) -> np.ndarray:
    """Remasking confidence per position of one sequence, larger = commit first:
    "marginal": the constrained marginal of the sampled token (the "Mar" rule);
    "neg_entropy": minus the entropy of the full constrained marginal (Dream's lowest
    entropy, on the constrained distribution);
    "unconstrained": the mean-field probability p_t(x_t) of the sampled token (the "Mf"
    ablation: constrained samples, unconstrained confidence).
    (paperfeed.app summary, "Constrained remasking confidence" and the ablation of Table 2.)"""
    if mode == "marginal":
        return np.asarray(marg_tokens, np.float64)
    if mode == "neg_entropy":
        return -entropy(marg_all)
    if mode == "unconstrained":
        t = np.arange(probs.shape[0])
        tok = np.where(np.asarray(tokens) >= 0, tokens, 0)
        return np.asarray(probs, np.float64)[t, tok]
    raise ValueError(mode)


def viterbi(fa, probs: np.ndarray, committed: Optional[np.ndarray] = None):
    """Greedy (T = 0) constrained decoding of one sequence: the accepted string with the
    largest mean-field product, argmax over x in C of prod_t w_t(x_t), by max-product over
    (state path, string) along the chain (paperfeed.app summary: greedy decoding with the
    constraint; the "greedy / MAP" variant of the same HMM).  Because the product depends
    only on the string, the best (path, string) pair carries the best accepted string; NFA
    path counts weight sampling and play no part here.  w_t is probs[t] at masked positions
    and one-hot at committed ones.

    Returns (score, tokens): score = ln of the maximum in float64 (-inf and tokens None when
    no accepted string has positive weight)."""
    probs = np.asarray(probs, np.float64)
    L, V = probs.shape
    S = fa.n_states
    src = np.asarray(fa.edge_src, np.int64)
    dst = np.asarray(fa.edge_dst, np.int64)
    off = np.asarray(fa.label_offsets, np.int64)
    lab = np.asarray(fa.label_tokens, np.int64)
    E = src.shape[0]
    with np.errstate(divide="ignore"):
        logw = np.log(probs)
    if committed is not None:
        for t in range(L):
            if committed[t] >= 0:
                logw[t] = -np.inf
                if committed[t] < V:
                    logw[t, committed[t]] = 0.0
    delta = np.full(S, -np.inf)
    delta[fa.start] = 0.0
    back_edge = np.zeros((L, S), np.int64)
    back_tok = np.zeros((L, E), np.int64)
    for t in range(L):
        # the best token of every edge at position t
        best = np.full(E, -np.inf)
        for e in range(E):
            toks = lab[off[e]:off[e + 1]]
            if toks.shape[0]:
                j = int(np.argmax(logw[t, toks]))
                best[e] = logw[t, toks[j]]
                back_tok[t, e] = toks[j]
        cand = delta[src] + best
        new = np.full(S, -np.inf)
        for e in range(E):
            if cand[e] > new[dst[e]]:
                new[dst[e]] = cand[e]
                back_edge[t, dst[e]] = e
        delta = new
    acc = np.asarray(fa.accept, np.int64)
    f = int(acc[np.argmax(delta[acc])])
    score = float(delta[f])
    if score == -np.inf:
        return score, None
    out = np.zeros(L, np.int32)
    s = f
    for t in range(L - 1, -1, -1):
        e = int(back_edge[t, s])
        out[t] = back_tok[t, e]
        s = int(src[e])
    return score, out


def string_log_weight(probs: np.ndarray, tokens: np.ndarray, committed: Optional[np.ndarray] = None) -> float:
    """ln prod_t w_t(x_t) of a given string (w_t one-hot at committed positions)."""
    probs = np.asarray(probs, np.float64)
    tot = 0.0
    for t, v in enumerate(tokens):
        if committed is not None and committed[t] >= 0:
            if v != committed[t]:
                return -np.inf
            continue
        tot += math.log(probs[t, v]) if probs[t, v] > 0 else -np.inf
    return tot


def topk(marg: np.ndarray, committed: np.ndarray, k: int, lo: int, hi: int) -> np.ndarray:
    lib = _load()
    m = np.ascontiguousarray(marg, np.float64)
    c = np.ascontiguousarray(committed, np.int32)
    out = np.zeros(max(k, 1), np.int32)
    lib.or_topk(m.shape[0], _p(m), _p(c), k, lo, hi, _p(out))
    return out[:k]


def philox4x32_10(ctr, key) -> np.ndarray:
    lib = _load()
    c = np.asarray(ctr, np.uint32)
    k = np.asarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib.or_philox4x32_10(_p(c), _p(k), _p(out))
    return out
