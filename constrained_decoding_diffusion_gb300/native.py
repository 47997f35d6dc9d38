"""Thin ctypes binding of libfa.so with the C ABI's names (include/fa.h).

Argument marshalling only: torch tensors are checked for device, dtype and
contiguity and passed as raw pointers on torch's current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; if the library is
missing this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_CUDA = 2
FA_ERR_OOM = 3
FA_ERR_WORKSPACE_TOO_SMALL = 4
FA_ERR_UNSUPPORTED = 5
FA_ROW_OK, FA_ROW_EMPTY, FA_ROW_UNDERFLOW, FA_ROW_TIMEOUT = 0, 1, 2, 3
FA_CONF_MARGINAL, FA_CONF_NEG_ENTROPY, FA_CONF_UNCONSTRAINED = 0, 1, 2
CONFIDENCE = {"marginal": FA_CONF_MARGINAL, "neg_entropy": FA_CONF_NEG_ENTROPY,
              "unconstrained": FA_CONF_UNCONSTRAINED}

# every entry point include/fa.h declares
EXPORTS = ("fa_compile", "fa_destroy", "fa_query", "fa_export_csr", "fa_step_workspace_bytes",
           "fa_transition_matrices", "fa_constrained_step", "fa_constrained_step_ex", "fa_constrained_step_chain",
           "fa_token_marginals", "fa_map_step", "fa_constrained_step_host",
           "fa_apply_commits", "fa_constrained_step_noalloc", "fa_debug_inject_wait_timeouts",
           "fa_profile_enable", "fa_profile_read",
           "fa_launch_count", "fa_last_error")
N_STAGES = 4
STAGES = ("reweight", "upsweep", "topdown", "leaf_commit")

_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("fa error %d: %s" % (code, msg))
        self.code = code


def load(path: str = LIB_PATH):
    """Load libfa.so and declare the C signatures (no CUDA call is made)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libfa.so not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                          "(expected at %s)" % path)
    lib = ctypes.CDLL(path)
    P, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    st = ctypes.c_int
    lib.fa_compile.argtypes = [i32, i32, P, i32, i32, P, P, P, P, i32, P, ctypes.POINTER(P)]
    lib.fa_compile.restype = st
    lib.fa_destroy.argtypes = [P]
    lib.fa_destroy.restype = st
    lib.fa_query.argtypes = [P, P, P, P, P, P, P]
    lib.fa_query.restype = st
    lib.fa_export_csr.argtypes = [P] * 10
    lib.fa_export_csr.restype = st
    lib.fa_step_workspace_bytes.argtypes = [P, i32, i32, ctypes.POINTER(sz)]
    lib.fa_step_workspace_bytes.restype = st
    lib.fa_transition_matrices.argtypes = [P, i32, i32, P, P, P, P, P]
    lib.fa_transition_matrices.restype = st
    lib.fa_constrained_step.argtypes = [P, i32, i32, P, P, u64, u64, i32, i32, i32, P, sz, P, P, P, P, P, P]
    lib.fa_constrained_step.restype = st
    lib.fa_constrained_step_ex.argtypes = [P, i32, i32, P, P, u64, u64, i32, i32, i32, i32, P, sz, P, P, P, P, P, P, P]
    lib.fa_constrained_step_ex.restype = st
    lib.fa_constrained_step_chain.argtypes = lib.fa_constrained_step_ex.argtypes
    lib.fa_constrained_step_chain.restype = st
    lib.fa_map_step.argtypes = [P, i32, i32, P, P, P, sz, P, P, P, P]
    lib.fa_map_step.restype = st
    lib.fa_token_marginals.argtypes = [P, i32, i32, P, P, P, sz, P, P, P, P]
    lib.fa_token_marginals.restype = st
    lib.fa_apply_commits.argtypes = [i32, i32, i32, P, P, P, P]
    lib.fa_apply_commits.restype = st
    lib.fa_constrained_step_host.argtypes = [P, i32, i32, P, P, P, P, u64, u64, i32, i32, i32, P, sz, P, P, P, P, P, P]
    lib.fa_constrained_step_host.restype = st
    lib.fa_constrained_step_noalloc.argtypes = [P, i32, i32, P, P, u64, u64, i32, i32, i32, P, P, P, P, P, P]
    lib.fa_constrained_step_noalloc.restype = st
    lib.fa_debug_inject_wait_timeouts.argtypes = [i32]
    lib.fa_debug_inject_wait_timeouts.restype = st
    lib.fa_profile_enable.argtypes = [i32]
    lib.fa_profile_enable.restype = st
    lib.fa_profile_read.argtypes = [P]
    lib.fa_profile_read.restype = st
    lib.fa_launch_count.argtypes = [P]
    lib.fa_launch_count.restype = st
    lib.fa_last_error.argtypes = []
    lib.fa_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(rc: int):
    if rc != FA_OK:
        raise FaError(rc, _lib.fa_last_error().decode(errors="replace"))


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, dtype, name, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return ctypes.c_void_p(t.data_ptr())


class CompiledAutomaton:
    """An automaton compiled and resident on the current device (fa_compile / fa_destroy)."""

    def __init__(self, handle, n_states: int, vocab: int):
        self.handle = handle
        self.n_states = n_states
        self.vocab = vocab
        n_e, n_i, dfa, n_acc = (np.zeros(1, np.int64), np.zeros(1, np.int64), np.zeros(1, np.int32),
                                np.zeros(1, np.int32))
        _check(_lib.fa_query(handle, _np_ptr(n_e), _np_ptr(n_i), _np_ptr(dfa), _np_ptr(n_acc), None, None))
        self.n_edges, self.n_incidences = int(n_e[0]), int(n_i[0])
        self.is_dfa, self.n_accept = bool(dfa[0]), int(n_acc[0])

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.fa_destroy(self.handle)
            self.handle = None


def fa_compile(fa, stream=None) -> CompiledAutomaton:
    """Compile a synth.Automaton-like object (n_states, start, accept, edge_src, edge_dst,
    label_offsets, label_tokens, vocab) onto the current CUDA device."""
    load()
    acc = np.ascontiguousarray(fa.accept, np.int32)
    src = np.ascontiguousarray(fa.edge_src, np.int32)
    dst = np.ascontiguousarray(fa.edge_dst, np.int32)
    off = np.ascontiguousarray(fa.label_offsets, np.int64)
    tok = np.ascontiguousarray(fa.label_tokens, np.int32)
    h = ctypes.c_void_p()
    _check(_lib.fa_compile(int(fa.n_states), int(fa.start), _np_ptr(acc), acc.shape[0], src.shape[0], _np_ptr(src),
                           _np_ptr(dst), _np_ptr(off), _np_ptr(tok), int(fa.vocab), _stream_ptr(stream),
                           ctypes.byref(h)))
    return CompiledAutomaton(h, int(fa.n_states), int(fa.vocab))


def fa_export_csr(aut: CompiledAutomaton) -> dict:
    S, V, E, I = aut.n_states, aut.vocab, aut.n_edges, aut.n_incidences
    out = dict(lab_off=np.zeros(E + 1, np.int64), lab_tok=np.zeros(max(I, 1), np.int32),
               src_off=np.zeros(S + 1, np.int32), src_edges=np.zeros(max(E, 1), np.int32),
               dst_off=np.zeros(S + 1, np.int32), dst_edges=np.zeros(max(E, 1), np.int32),
               tok_off=np.zeros(V + 1, np.int64), tok_edges=np.zeros(max(I, 1), np.int32),
               accept=np.zeros(max(aut.n_accept, 1), np.int32))
    _check(_lib.fa_export_csr(aut.handle, *[_np_ptr(out[k]) for k in (
        "lab_off", "lab_tok", "src_off", "src_edges", "dst_off", "dst_edges", "tok_off", "tok_edges", "accept")]))
    out["lab_tok"], out["tok_edges"] = out["lab_tok"][:I], out["tok_edges"][:I]
    out["src_edges"], out["dst_edges"] = out["src_edges"][:E], out["dst_edges"][:E]
    out["accept"] = out["accept"][:aut.n_accept]
    return out


def fa_step_workspace_bytes(aut: CompiledAutomaton, B: int, L: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fa_step_workspace_bytes(aut.handle, int(B), int(L), ctypes.byref(n)))
    return int(n.value)


def fa_transition_matrices(aut: CompiledAutomaton, probs, committed, mant, row_exp, stream=None):
    """M_t = mant * 2^row_exp for every (b, t): probs [B,L,V] f32, committed [B,L] i32,
    mant [B,L,S,S] f32 out, row_exp [B,L,S] i32 out."""
    import torch
    B, L, V = probs.shape
    S = aut.n_states
    _check(_lib.fa_transition_matrices(aut.handle, B, L, _dev(probs, torch.float32, "probs", (B, L, aut.vocab)),
                                       _dev(committed, torch.int32, "committed", (B, L)),
                                       _dev(mant, torch.float32, "mant", (B, L, S, S)),
                                       _dev(row_exp, torch.int32, "row_exp", (B, L, S)), _stream_ptr(stream)))


def fa_constrained_step(aut: CompiledAutomaton, probs, committed, philox_seed: int, philox_offset: int, k: int,
                        commit_lo: int, commit_hi: int, workspace, tokens, logZ, marg, commit_idx, row_status,
                        stream=None):
    """One constrained denoising step (include/fa.h); all tensors on the current device."""
    import torch
    B, L, V = probs.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.fa_constrained_step(
        aut.handle, B, L, _dev(probs, torch.float32, "probs", (B, L, aut.vocab)),
        _dev(committed, torch.int32, "committed", (B, L)), ctypes.c_uint64(philox_seed & (2 ** 64 - 1)),
        ctypes.c_uint64(philox_offset & (2 ** 64 - 1)), int(k), int(commit_lo), int(commit_hi),
        _dev(workspace, workspace.dtype, "workspace"), ws_bytes, _dev(tokens, torch.int32, "tokens", (B, L)),
        _dev(logZ, torch.float64, "logZ", (B,)), _dev(marg, torch.float32, "marg", (B, L)),
        _dev(commit_idx, torch.int32, "commit_idx", (B, k)) if k > 0 else None,
        _dev(row_status, torch.int32, "row_status", (B,)), _stream_ptr(stream)))


def _host(t, dtype, name, shape):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("%s must be a host tensor" % name)
    if t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError("%s must be a contiguous %s tensor of shape %s" % (name, dtype, tuple(shape)))
    return ctypes.c_void_p(t.data_ptr())


def fa_constrained_step_host(aut: CompiledAutomaton, h_probs, h_committed, d_probs, d_committed, philox_seed: int,
                             philox_offset: int, k: int, commit_lo: int, commit_hi: int, workspace, tokens, logZ,
                             marg, commit_idx, row_status, stream=None):
    """fa_constrained_step with the inputs in (page-locked) host tensors: copied into d_probs
    and d_committed in pieces of positions, overlapped with the emission reweighting."""
    import torch
    B, L, V = h_probs.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.fa_constrained_step_host(
        aut.handle, B, L, _host(h_probs, torch.float32, "h_probs", (B, L, aut.vocab)),
        _host(h_committed, torch.int32, "h_committed", (B, L)), _dev(d_probs, torch.float32, "d_probs", (B, L, aut.vocab)),
        _dev(d_committed, torch.int32, "d_committed", (B, L)), ctypes.c_uint64(philox_seed & (2 ** 64 - 1)),
        ctypes.c_uint64(philox_offset & (2 ** 64 - 1)), int(k), int(commit_lo), int(commit_hi),
        _dev(workspace, workspace.dtype, "workspace"), ws_bytes, _dev(tokens, torch.int32, "tokens", (B, L)),
        _dev(logZ, torch.float64, "logZ", (B,)), _dev(marg, torch.float32, "marg", (B, L)),
        _dev(commit_idx, torch.int32, "commit_idx", (B, k)) if k > 0 else None,
        _dev(row_status, torch.int32, "row_status", (B,)), _stream_ptr(stream)))


def fa_constrained_step_ex(aut: CompiledAutomaton, probs, committed, philox_seed: int, philox_offset: int, k: int,
                           commit_lo: int, commit_hi: int, confidence: str, workspace, tokens, logZ, marg, entropy,
                           commit_idx, row_status, stream=None, method: str = "tree"):
    """fa_constrained_step with a remasking confidence ("marginal", "neg_entropy" or
    "unconstrained"), an optional entropy output [B, L] (None to skip), and the tree
    (fa_constrained_step_ex) or chain (fa_constrained_step_chain) form of the step."""
    import torch
    B, L, V = probs.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    fn = {"tree": _lib.fa_constrained_step_ex, "chain": _lib.fa_constrained_step_chain}[method]
    _check(fn(
        aut.handle, B, L, _dev(probs, torch.float32, "probs", (B, L, aut.vocab)),
        _dev(committed, torch.int32, "committed", (B, L)), ctypes.c_uint64(philox_seed & (2 ** 64 - 1)),
        ctypes.c_uint64(philox_offset & (2 ** 64 - 1)), int(k), int(commit_lo), int(commit_hi),
        CONFIDENCE[confidence], _dev(workspace, workspace.dtype, "workspace"), ws_bytes,
        _dev(tokens, torch.int32, "tokens", (B, L)), _dev(logZ, torch.float64, "logZ", (B,)),
        _dev(marg, torch.float32, "marg", (B, L)),
        _dev(entropy, torch.float32, "entropy", (B, L)) if entropy is not None else None,
        _dev(commit_idx, torch.int32, "commit_idx", (B, k)) if k > 0 else None,
        _dev(row_status, torch.int32, "row_status", (B,)), _stream_ptr(stream)))


def fa_token_marginals(aut: CompiledAutomaton, probs, committed, workspace, row_status, marg_all=None, entropy=None,
                       stream=None):
    """Full constrained marginals [B, L, V] and/or entropies [B, L] from the messages of the
    step that last used `workspace` (same inputs)."""
    import torch
    B, L, V = probs.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.fa_token_marginals(
        aut.handle, B, L, _dev(probs, torch.float32, "probs", (B, L, aut.vocab)),
        _dev(committed, torch.int32, "committed", (B, L)), _dev(workspace, workspace.dtype, "workspace"), ws_bytes,
        _dev(row_status, torch.int32, "row_status", (B,)),
        _dev(marg_all, torch.float32, "marg_all", (B, L, aut.vocab)) if marg_all is not None else None,
        _dev(entropy, torch.float32, "entropy", (B, L)) if entropy is not None else None, _stream_ptr(stream)))


def fa_map_step(aut: CompiledAutomaton, probs, committed, workspace, tokens, score, row_status, stream=None):
    """Greedy (T = 0) constrained decoding: the accepted string with the largest mean-field
    product (include/fa.h); all tensors on the current device."""
    import torch
    B, L, V = probs.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.fa_map_step(
        aut.handle, B, L, _dev(probs, torch.float32, "probs", (B, L, aut.vocab)),
        _dev(committed, torch.int32, "committed", (B, L)), _dev(workspace, workspace.dtype, "workspace"), ws_bytes,
        _dev(tokens, torch.int32, "tokens", (B, L)), _dev(score, torch.float64, "score", (B,)),
        _dev(row_status, torch.int32, "row_status", (B,)), _stream_ptr(stream)))


class GreedyStep:
    """Owner of the workspace and outputs of fa_map_step for a fixed (B, L)."""

    def __init__(self, aut: CompiledAutomaton, B: int, L: int, device="cuda"):
        import torch
        self.aut, self.B, self.L = aut, B, L
        nbytes = fa_step_workspace_bytes(aut, B, L)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        self.tokens = torch.empty((B, L), dtype=torch.int32, device=device)
        self.score = torch.empty((B,), dtype=torch.float64, device=device)
        self.row_status = torch.empty((B,), dtype=torch.int32, device=device)

    def __call__(self, probs, committed, stream=None):
        fa_map_step(self.aut, probs, committed, self.workspace, self.tokens, self.score, self.row_status, stream)
        return self.tokens, self.score, self.row_status


def fa_apply_commits(commit_idx, tokens, committed, stream=None):
    """committed[b, t] = tokens[b, t] for every t in commit_idx[b] (t >= 0), on the device."""
    import torch
    B, L = committed.shape
    k = commit_idx.shape[1]
    _check(_lib.fa_apply_commits(B, L, k, _dev(commit_idx, torch.int32, "commit_idx", (B, k)),
                                 _dev(tokens, torch.int32, "tokens", (B, L)),
                                 _dev(committed, torch.int32, "committed", (B, L)), _stream_ptr(stream)))


class ConstrainedStep:
    """Convenience owner of the workspace and output tensors for a fixed (B, L, k)."""

    def __init__(self, aut: CompiledAutomaton, B: int, L: int, k: int, device="cuda", confidence: str = "marginal",
                 want_entropy: bool = False, method: str = "tree"):
        import torch
        if confidence not in CONFIDENCE:
            raise ValueError("confidence must be one of %s" % sorted(CONFIDENCE))
        if method not in ("tree", "chain"):
            raise ValueError("method must be 'tree' or 'chain'")
        self.method = method
        self.aut, self.B, self.L, self.k = aut, B, L, k
        self.confidence = confidence
        self.entropy = torch.empty((B, L), dtype=torch.float32, device=device) if want_entropy else None
        nbytes = fa_step_workspace_bytes(aut, B, L)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        self.tokens = torch.empty((B, L), dtype=torch.int32, device=device)
        self.logZ = torch.empty((B,), dtype=torch.float64, device=device)
        self.marg = torch.empty((B, L), dtype=torch.float32, device=device)
        self.commit_idx = torch.empty((B, k), dtype=torch.int32, device=device)
        self.row_status = torch.empty((B,), dtype=torch.int32, device=device)

    def __call__(self, probs, committed, seed: int, offset: int = 0, lo: int = 0, hi: Optional[int] = None,
                 stream=None):
        hi = self.L if hi is None else hi
        if self.method == "tree" and self.confidence == "marginal" and self.entropy is None:
            fa_constrained_step(self.aut, probs, committed, seed, offset, self.k, lo, hi, self.workspace, self.tokens,
                                self.logZ, self.marg, self.commit_idx, self.row_status, stream)
        else:
            fa_constrained_step_ex(self.aut, probs, committed, seed, offset, self.k, lo, hi, self.confidence,
                                   self.workspace, self.tokens, self.logZ, self.marg, self.entropy, self.commit_idx,
                                   self.row_status, stream, method=self.method)
        return self.tokens, self.logZ, self.marg, self.commit_idx, self.row_status

    def token_marginals(self, probs, committed, stream=None):
        """Full constrained marginals [B, L, V] and entropies [B, L] of the last call's inputs."""
        import torch
        marg_all = torch.empty((self.B, self.L, self.aut.vocab), dtype=torch.float32, device=self.tokens.device)
        ent = torch.empty((self.B, self.L), dtype=torch.float32, device=self.tokens.device)
        fa_token_marginals(self.aut, probs, committed, self.workspace, self.row_status, marg_all, ent, stream)
        return marg_all, ent


def fa_profile_enable(enable: bool):
    load()
    _check(_lib.fa_profile_enable(1 if enable else 0))


def fa_profile_read() -> dict:
    """Stage durations (ms) of the most recent step recorded with profiling enabled."""
    ms = np.zeros(N_STAGES, np.float32)
    _check(_lib.fa_profile_read(_np_ptr(ms)))
    return dict(zip(STAGES, (float(x) for x in ms)))


def fa_debug_inject_wait_timeouts(n_launches: int):
    """Failure tests: the next n_launches tensor-core span launches let a bounded wait run
    out (the step reports FA_ROW_TIMEOUT); 0 disarms."""
    load()
    _check(_lib.fa_debug_inject_wait_timeouts(int(n_launches)))


def fa_launch_count() -> int:
    load()
    n = np.zeros(1, np.uint64)
    _check(_lib.fa_launch_count(_np_ptr(n)))
    return int(n[0])


NOALLOC_SCRATCH_BYTES = 16 << 20


def fa_constrained_step_noalloc(aut: CompiledAutomaton, probs, committed, philox_seed: int, philox_offset: int,
                                k: int, commit_lo: int, commit_hi: int, tokens, logZ, marg, commit_idx, row_status,
                                stream=None):
    """fa_constrained_step without a workspace argument: for callers that cannot allocate
    device memory.  The library's built-in scratch array (NOALLOC_SCRATCH_BYTES per device)
    is used instead; calls that overlap on the GPU must be serialised by the caller."""
    import torch
    B, L, V = probs.shape
    _check(_lib.fa_constrained_step_noalloc(
        aut.handle, B, L, _dev(probs, torch.float32, "probs", (B, L, aut.vocab)),
        _dev(committed, torch.int32, "committed", (B, L)), ctypes.c_uint64(philox_seed & (2 ** 64 - 1)),
        ctypes.c_uint64(philox_offset & (2 ** 64 - 1)), int(k), int(commit_lo), int(commit_hi),
        _dev(tokens, torch.int32, "tokens", (B, L)), _dev(logZ, torch.float64, "logZ", (B,)),
        _dev(marg, torch.float32, "marg", (B, L)),
        _dev(commit_idx, torch.int32, "commit_idx", (B, k)) if k > 0 else None,
        _dev(row_status, torch.int32, "row_status", (B,)), _stream_ptr(stream)))
