/*
 * fa.h -- C ABI of the GB300 finite-automaton constrained denoising step.
 *
 * The method: "Constrained Decoding for Diffusion Language Models via
 * Efficient Inference over Finite Automata" (arXiv 2607.07026), as summarised
 * by the paperfeed.app page (sections "The insight: the constraint is a hidden
 * Markov model" and "The scan trick: log-depth exact sampling") and the
 * papernotes.org NeurIPS 2026 notes (method section, key designs 1-3).
 *
 * At one denoising step a diffusion LM gives a fully factorised distribution
 * p(x | x^t) = prod_t p_t(x_t).  The constraint is an automaton
 * M = (S, V, delta, s0, F) whose edges carry token label sets.  Viewing M as
 * a hidden Markov model whose latent is the edge taken, the step samples
 *     x ~ q(x) / Z,   q(x) = prod_t w_t(x_t) * N(x),
 * where w_t = p_t for a masked position and the indicator of the committed
 * token otherwise, and N(x) is the number of accepting paths labelled x (0/1
 * for a DFA).  It returns logZ, the constrained marginal p(x_t = x^_t | x^t, C)
 * of each sampled token, and the k masked positions with the highest such
 * marginal (the "Mar" remasking rule of the notes' key design 3).
 *
 * Conventions
 *  - Every pointer argument of fa_compile is HOST memory; every array argument
 *    of the step calls is DEVICE memory owned by the caller.
 *  - Calls that take a stream are asynchronous on it.  Their return value
 *    reports only argument, launch and workspace errors; data-dependent
 *    outcomes go to row_status on the device, with no host synchronisation.
 *  - A compiled automaton is immutable and may be used by concurrent steps on
 *    different streams, each with its own workspace.
 *  - Results are a pure function of (inputs, philox_seed, philox_offset).
 *  - On any error the call returns a non-zero fa_status and fa_last_error()
 *    gives a message (thread-local).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fa_automaton fa_automaton; /* opaque, library-owned */
typedef void *fa_stream;                  /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,
    FA_ERR_CUDA = 2,
    FA_ERR_OOM = 3,
    FA_ERR_WORKSPACE_TOO_SMALL = 4,
    FA_ERR_UNSUPPORTED = 5
} fa_status;

/* Per-sequence outcome written by the step into row_status[b]. */
enum {
    FA_ROW_OK = 0,
    FA_ROW_EMPTY = 1,     /* Z == 0: no accepted string has positive weight */
    FA_ROW_UNDERFLOW = 2, /* range loss: a span product pushed nonzero mass below the fp32
                             range, or a categorical the sampler needed summed to 0 */
    FA_ROW_TIMEOUT = 3    /* a bounded wait inside a kernel ran out (work abandoned) */
};

/* Library limits. */
#define FA_MAX_STATES 4096
#define FA_MAX_LENGTH 65536

/*
 * fa_compile -- validate an automaton and upload it to the current device.
 *
 * The automaton as a hidden Markov model (paperfeed.app, "The insight": latent
 * z_i = edge taken at step i, transition = the indicator that consecutive
 * edges chain, emission = the indicator that x_i is in z_i's label set, start
 * pinned to s0, final state accepting).
 *
 *   n_states            |S| in [1, FA_MAX_STATES]
 *   start               s0 in [0, n_states)
 *   accept[n_accept]    accepting states (repeats allowed; n_accept may be 0)
 *   n_edges             E >= 0
 *   edge_src/edge_dst   [E] state ids
 *   label_offsets[E+1]  int64, label_offsets[0] = 0, non-decreasing; edge e reads
 *                       label_tokens[label_offsets[e] .. label_offsets[e+1])
 *   label_tokens        token ids in [0, vocab); a token repeated inside one set
 *                       counts once; an empty set is rejected
 *   vocab               |V| >= 1
 *   stream              stream for the uploads
 *   out                 receives the handle; release with fa_destroy
 *
 * Parallel edges s -> s' are kept: each is its own path (NFA path counting,
 * paperfeed.app "Arbitrary schedules and NFAs").  Every edge consumes one
 * token, so there are no epsilon edges.  The call synchronises the stream
 * before returning (host staging buffers are freed).
 * Errors: FA_ERR_INVALID_ARG (ids out of range, empty label set, bad offsets),
 * FA_ERR_OOM, FA_ERR_CUDA.
 */
fa_status fa_compile(int32_t n_states, int32_t start, const int32_t *accept, int32_t n_accept,
                     int32_t n_edges, const int32_t *edge_src, const int32_t *edge_dst,
                     const int64_t *label_offsets, const int32_t *label_tokens, int32_t vocab,
                     fa_stream stream, fa_automaton **out);

/* Free the device copy and the handle (NULL is accepted). */
fa_status fa_destroy(fa_automaton *aut);

/* Sizes of the compiled automaton: edges, token-edge incidences after
 * de-duplication, whether no (state, token) pair has two edges, the number of
 * distinct accepting states, |S| and |V|.  Any output pointer may be NULL. */
fa_status fa_query(const fa_automaton *aut, int64_t *n_edges, int64_t *n_incidences, int32_t *is_dfa,
                   int32_t *n_accept, int32_t *n_states, int32_t *vocab);

/*
 * fa_export_csr -- copy the canonical compiled arrays back to HOST buffers.
 *
 *   lab_off[E+1], lab_tok[I]     label sets, each sorted ascending, repeats removed
 *   src_off[S+1], src_edges[E]   edge ids sorted by (src, dst, id)
 *   dst_off[S+1], dst_edges[E]   edge ids sorted by (dst, src, id)
 *   tok_off[V+1], tok_edges[I]   token -> edge incidence sorted by (token, src, dst, id)
 *   accept[n_accept]             distinct accepting states, ascending
 * Synchronous.  Errors: FA_ERR_INVALID_ARG (NULL buffer), FA_ERR_CUDA.
 */
fa_status fa_export_csr(const fa_automaton *aut, int64_t *lab_off, int32_t *lab_tok, int32_t *src_off,
                        int32_t *src_edges, int32_t *dst_off, int32_t *dst_edges, int64_t *tok_off,
                        int32_t *tok_edges, int32_t *accept);

/* Bytes of device workspace fa_constrained_step needs for batch B and length L.
 * Errors: FA_ERR_INVALID_ARG (B < 0, L < 0 or L > FA_MAX_LENGTH). */
fa_status fa_step_workspace_bytes(const fa_automaton *aut, int32_t B, int32_t L, size_t *bytes);

/*
 * fa_transition_matrices -- the emission-reweighting stage alone.
 *
 * Key design 1 of the papernotes.org notes: the automaton's transitions stay
 * fixed and every edge's emission is reweighted by the model's per-position
 * probability, g(x_i = v | z_i = e) = 1[v in label(e)] * p_i(v), which folds
 * into per-position state matrices
 *     M_t(s, s') = sum_{e: s -> s'} sum_{v in label(e)} w_t(v).
 * A committed position (committed[b,t] >= 0) has w_t = one-hot, so M_t counts
 * the edges s -> s' that carry the committed token.
 *
 *   probs      [B, L, V] fp32, row-major, V contiguous; non-negative, finite
 *   committed  [B, L] int32: a token id, or -1 = masked
 *   mant       [B, L, S, S] fp32 out and row_exp [B, L, S] int32 out, with
 *              M_t(s, s') = mant[b,t,s,s'] * 2^row_exp[b,t,s]
 * A committed id outside [0, V) is treated as a token no edge carries.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_CUDA (launch).
 */
fa_status fa_transition_matrices(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                 const int32_t *committed, float *mant, int32_t *row_exp,
                                 fa_stream stream);

/*
 * fa_constrained_step -- one constrained denoising step.
 *
 * Exact sampling from the constrained mean-field posterior by the log-depth
 * tree of the paperfeed.app page ("The scan trick") and key design 2 of the
 * notes: span matrices A[l, r) = M_{l+1} ... M_r are built bottom-up over
 * 2^k steps by batched products, the end state is drawn from the root
 * (z_0 = s0, z_L ~ A_root[s0, .] restricted to F), every midpoint
 * z_m ~ A[l, m)[z_l, .] * A[m, r)[., z_r] top-down level by level, and finally
 * every token is drawn from the label sets of the edges z_{t-1} -> z_t in
 * proportion to w_t.  The constrained marginals of the sampled tokens come from
 * prefix/suffix messages over the same tree (key design 3), and the commit set
 * is the top k of those marginals among masked positions of [commit_lo,
 * commit_hi), descending, ties to the lower position, padded with -1.
 *
 *   B, L            batch and length (B >= 0, 0 <= L <= FA_MAX_LENGTH)
 *   probs           [B, L, V] fp32 device, read only
 *   committed       [B, L] int32 device: token id, or -1 = masked
 *   philox_seed,
 *   philox_offset   Philox4x32-10 key and counter offset (Salmon et al., SC'11);
 *                   advance the offset between steps
 *   k               commit count >= 0
 *   commit_lo/hi    commit window, 0 <= lo <= hi <= L
 *   workspace       device scratch of at least fa_step_workspace_bytes(B, L)
 *                   bytes, 256-byte aligned, caller-owned; contents are
 *                   overwritten; concurrent steps need separate workspaces
 *   tokens          [B, L] int32 out: sampled x^ (committed positions echoed)
 *   logZ            [B] double out: ln Z (-inf when FA_ROW_EMPTY or FA_ROW_TIMEOUT,
 *                   NaN when the up-sweep lost range: FA_ROW_UNDERFLOW)
 *   marg            [B, L] fp32 out: constrained marginal of x^_t (1 for committed)
 *   commit_idx      [B, k] int32 out
 *   row_status      [B] int32 out: FA_ROW_*
 * When row_status[b] != FA_ROW_OK, tokens[b] echo committed (-1 where masked),
 * marg[b] is 0 where masked and commit_idx[b] is all -1.
 *
 * Range.  Span matrices keep an fp32 mantissa and a power-of-two exponent per row, so an
 * entry more than about 2^126 below the largest entry of its row cannot be represented.
 * Every span product checks its prescaled left operand: when a nonzero entry would leave
 * the fp32 normal range, the sequence is reported as FA_ROW_UNDERFLOW (logZ NaN, no
 * tokens, no commits) instead of being sampled from spans that lost mass.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_WORKSPACE_TOO_SMALL, FA_ERR_CUDA (launch).
 */
fa_status fa_constrained_step(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                              const int32_t *committed, uint64_t philox_seed, uint64_t philox_offset,
                              int32_t k, int32_t commit_lo, int32_t commit_hi, void *workspace,
                              size_t ws_bytes, int32_t *tokens, double *logZ, float *marg,
                              int32_t *commit_idx, int32_t *row_status, fa_stream stream);

/*
 * Remasking confidence: what the commit ranks masked positions by, larger first.  The
 * paperfeed.app summary ("Constrained remasking confidence" and the ablation of its
 * Table 2) and key design 3 of the papernotes.org notes: a dLLM commits the positions with
 * the best confidence (LLaDA: highest probability, Dream: lowest entropy), and the method
 * computes it from the constrained distribution ("Mar") instead of the mean-field one ("Mf").
 */
enum {
    FA_CONF_MARGINAL = 0,      /* constrained marginal of the sampled token ("Mar"; the default) */
    FA_CONF_NEG_ENTROPY = 1,   /* minus the entropy of the position's full constrained token distribution */
    FA_CONF_UNCONSTRAINED = 2  /* the mean-field probability p_t(x^_t) of the sampled token ("Mf") */
};

/*
 * fa_constrained_step_ex -- fa_constrained_step with a choice of remasking confidence.
 *
 *   confidence  FA_CONF_*: the commit takes the k masked positions of [commit_lo, commit_hi)
 *               with the largest confidence, descending, ties to the lower position
 *   entropy     [B, L] fp32 device out, or NULL: entropy in nats of every position's full
 *               constrained token distribution (see fa_token_marginals); 0 for committed
 *               positions and for sequences whose status is not FA_ROW_OK
 * FA_CONF_NEG_ENTROPY or a non-NULL entropy costs one more pass over the token-edge
 * incidences of every masked position (about the work of the reweight).  Every other
 * argument is as for fa_constrained_step, which is this call with FA_CONF_MARGINAL and
 * entropy = NULL.
 * Errors: as fa_constrained_step; FA_ERR_INVALID_ARG for an unknown confidence.
 */
fa_status fa_constrained_step_ex(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                 const int32_t *committed, uint64_t philox_seed, uint64_t philox_offset,
                                 int32_t k, int32_t commit_lo, int32_t commit_hi, int32_t confidence,
                                 void *workspace, size_t ws_bytes, int32_t *tokens, double *logZ, float *marg,
                                 float *entropy, int32_t *commit_idx, int32_t *row_status, fa_stream stream);

/*
 * fa_constrained_step_host -- fa_constrained_step with the per-position inputs in host
 * memory (the step a caller runs when the model's probabilities are still on the host).
 * The method is the one of fa_constrained_step (paperfeed.app summary, "The scan trick";
 * papernotes.org notes, key designs 1-3); this call only moves the inputs.
 *
 *   h_probs      [B, L, V] fp32 host, page-locked (cudaHostAlloc or cudaHostRegister) for
 *                the copies to run asynchronously; read-only
 *   h_committed  [B, L] int32 host, page-locked; read-only
 *   d_probs      [B, L, V] fp32 device, caller-owned: receives the copy of h_probs
 *   d_committed  [B, L] int32 device, caller-owned: receives the copy of h_committed
 *   every other argument and output as for fa_constrained_step (outputs in device memory)
 *
 * The committed tokens and then the probabilities, in up to eight pieces of consecutive
 * positions (the first a thirty-second of the batch, each next one 1.4 times larger), are
 * copied on a copy stream the library keeps per host thread and device, after the work
 * already queued on `stream`; the emission reweighting of each piece starts on `stream` as
 * soon as its rows have landed, so the copy of later pieces overlaps the reweighting of
 * earlier ones.  The results are those of fa_constrained_step on the copied inputs, bit for
 * bit.  The host buffers must stay unchanged until `stream` has passed the call.
 * Errors: as fa_constrained_step; FA_ERR_INVALID_ARG for a NULL input buffer; FA_ERR_CUDA
 * when the copy stream or its events cannot be created.
 */
fa_status fa_constrained_step_host(const fa_automaton *aut, int32_t B, int32_t L, const float *h_probs,
                                   const int32_t *h_committed, float *d_probs, int32_t *d_committed,
                                   uint64_t philox_seed, uint64_t philox_offset, int32_t k, int32_t commit_lo,
                                   int32_t commit_hi, void *workspace, size_t ws_bytes, int32_t *tokens,
                                   double *logZ, float *marg, int32_t *commit_idx, int32_t *row_status,
                                   fa_stream stream);

/*
 * fa_constrained_step_chain -- the same step computed in chain form: forward messages
 * alpha_t = alpha_{t-1} M_t for t = 1..L, then backward messages beta_{t-1} = M_t beta_t with
 * forward-filtering backward-sampling of the states (z_L ~ alpha_L restricted to F,
 * z_{t-1} ~ alpha_{t-1}(s) M_t(s, z_t)).  This is the O(L)-depth chain that the paperfeed.app
 * summary ("The scan trick") and key design 2 of the papernotes.org notes replace by the
 * log-depth tree; it samples the same distribution with O(L S^2) instead of O(L S^3) work,
 * one sequence per thread block.  Arguments, workspace size and outputs are those of
 * fa_constrained_step_ex; the draws differ from the tree's for the same seed (another
 * sequence of Philox counters), the distribution does not.
 */
fa_status fa_constrained_step_chain(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                    const int32_t *committed, uint64_t philox_seed, uint64_t philox_offset,
                                    int32_t k, int32_t commit_lo, int32_t commit_hi, int32_t confidence,
                                    void *workspace, size_t ws_bytes, int32_t *tokens, double *logZ, float *marg,
                                    float *entropy, int32_t *commit_idx, int32_t *row_status, fa_stream stream);

/*
 * fa_map_step -- greedy (T = 0) constrained decoding: the accepted string with the largest
 * mean-field product, argmax over x in the language of prod_t w_t(x_t) (w_t one-hot at
 * committed positions), by max-product over the same log-depth tree (paperfeed.app summary,
 * greedy decoding with the constraint; key design 2 of the papernotes.org notes with max in
 * place of sum).  The product of a string does not depend on its accepting path, so the
 * best (path, string) pair carries the best accepted string; NFA path counts play no part.
 * Ties go to the lowest state and token index.  Span products run on the CUDA cores (the
 * tensor cores have no max).
 *
 *   workspace   as for fa_constrained_step (fa_step_workspace_bytes(B, L))
 *   tokens      [B, L] int32 out (committed positions echoed; -1 where masked when
 *               row_status[b] != FA_ROW_OK)
 *   score       [B] double out: ln of the best product (-inf when no accepted string has a
 *               positive product)
 *   row_status  [B] int32 out: FA_ROW_*
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_WORKSPACE_TOO_SMALL, FA_ERR_CUDA (launch).
 */
fa_status fa_map_step(const fa_automaton *aut, int32_t B, int32_t L, const float *probs, const int32_t *committed,
                      void *workspace, size_t ws_bytes, int32_t *tokens, double *score, int32_t *row_status,
                      fa_stream stream);

/*
 * fa_token_marginals -- the full constrained marginal of every token at every position,
 *     p(x_t = v) = w_t(v) * sum_{e carries v} alpha_{t-1}(src e) beta_t(dst e) / (same summed over v)
 * (key design 3 of the papernotes.org notes), from the prefix/suffix messages that the
 * preceding fa_constrained_step or fa_constrained_step_ex left in its workspace.  Call it on
 * the same stream after that step, with the same automaton, B, L, probs, committed and
 * workspace, before the workspace is used again.
 *
 *   row_status  [B] int32 device: that step's status
 *   marg_all    [B, L, V] fp32 device out, or NULL; one-hot at committed positions, zero
 *               at the masked positions of sequences whose status is not FA_ROW_OK
 *   entropy     [B, L] fp32 device out, or NULL: -sum_v p ln p (nats), 0 where marg_all is
 *               one-hot or zero
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_WORKSPACE_TOO_SMALL, FA_ERR_CUDA (launch).
 */
fa_status fa_token_marginals(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                             const int32_t *committed, const void *workspace, size_t ws_bytes,
                             const int32_t *row_status, float *marg_all, float *entropy, fa_stream stream);

/*
 * fa_apply_commits -- the commit of a remasking schedule: committed[b, t] = tokens[b, t] for
 * every t = commit_idx[b, i] >= 0 (i < k).  With fa_constrained_step this gives any
 * schedule of the papernotes.org notes (key design 3) or the paperfeed.app summary
 * ("Arbitrary schedules and NFAs"): parallel, block-wise (through the commit window) or
 * fewer steps with larger k.  All arrays are device memory: commit_idx [B, k], tokens and
 * committed [B, L].  Asynchronous on stream.  Errors: FA_ERR_INVALID_ARG, FA_ERR_CUDA.
 */
fa_status fa_apply_commits(int32_t B, int32_t L, int32_t k, const int32_t *commit_idx, const int32_t *tokens,
                           int32_t *committed, fa_stream stream);

/*
 * fa_constrained_step_noalloc -- fa_constrained_step for callers that cannot allocate.
 *
 * No counterpart in the paper: this is a deployment convenience.  Some callers may not
 * allocate device memory where they decode (an engine whose pool owns all device memory,
 * a plugin or real-time loop where cudaMalloc would synchronise the device, code that only
 * receives pointers).  They pass inputs and outputs exactly as for fa_constrained_step,
 * but no workspace: the scratch is a fixed FA_NOALLOC_SCRATCH_BYTES array built into the
 * library, which every GPU that loads the library holds until the process exits.  The call
 * itself allocates nothing.
 *
 * Every call looks up the array's device address on the current device (so the address
 * stays right after a device reset); the first call on a device also loads the library's
 * device code there, so make it before any stream capture.  All calls on a device share
 * the array and it keeps the last call's contents (the step initialises what it reads, so
 * no clearing is needed); calls whose GPU work overlaps race on it and must be serialised
 * by the caller.
 * Errors: as fa_constrained_step (B, L and k are range-checked first), plus
 * FA_ERR_WORKSPACE_TOO_SMALL when fa_step_workspace_bytes(B, L) exceeds
 * FA_NOALLOC_SCRATCH_BYTES, FA_ERR_CUDA if the array's address cannot be obtained.
 */
#define FA_NOALLOC_SCRATCH_BYTES (16u << 20)
fa_status fa_constrained_step_noalloc(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                      const int32_t *committed, uint64_t philox_seed, uint64_t philox_offset,
                                      int32_t k, int32_t commit_lo, int32_t commit_hi, int32_t *tokens,
                                      double *logZ, float *marg, int32_t *commit_idx, int32_t *row_status,
                                      fa_stream stream);

/*
 * fa_debug_inject_wait_timeouts -- failure-injection hook for tests (no counterpart on the
 * pages).  The next n_launches launches of the tensor-core span product (|S| >= 128) make
 * their MMA-issuing thread wait, with a short limit (about half a millisecond), on a
 * barrier that nothing completes.  The wait runs out, every CTA of the launch abandons its
 * tile after the copies and products it already issued have completed, and the step reports
 * FA_ROW_TIMEOUT for every sequence; the next step is unaffected.  n_launches = 0 disarms.
 * Process-wide.  Errors: FA_ERR_INVALID_ARG (n_launches < 0).
 */
fa_status fa_debug_inject_wait_timeouts(int32_t n_launches);

/*
 * Stage timing and launch accounting (measurement support; no counterpart on the pages).
 *
 * fa_profile_enable(1) makes later fa_constrained_step calls on this host thread record
 * FA_N_STAGES + 1 CUDA events on their stream at the stage boundaries: 0 reweight,
 * 1 span up-sweep, 2 root + top-down sampling and messages, 3 leaf tokens, marginals and
 * the commit.  Inside a stream capture they become event-record graph nodes.
 * fa_profile_read waits for the last boundary event and writes the FA_N_STAGES elapsed
 * times (ms) of the most recent recorded step into ms[FA_N_STAGES].
 * fa_launch_count gives the number of kernel launches this library has issued in the
 * process (one per kernel node when a step is captured into a graph).
 * Errors: FA_ERR_INVALID_ARG (NULL pointer, profiling never enabled), FA_ERR_CUDA.
 */
#define FA_N_STAGES 4
fa_status fa_profile_enable(int32_t enable);
fa_status fa_profile_read(float *ms);
fa_status fa_launch_count(uint64_t *n);

/* Message for the last failing call on this thread ("" if none). */
const char *fa_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_H_ */
