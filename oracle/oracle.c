/*
 * Float64 CPU oracle for the finite-automaton constrained denoising step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke entry and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA path; the two meet only through the seeded
 * input generators.
 *
 * What it computes (all citations are to "Constrained Decoding for Diffusion
 * Language Models via Efficient Inference over Finite Automata"):
 *
 *  - The target (paperfeed.app summary, section "The insight: the constraint is
 *    a hidden Markov model"; papernotes.org notes, key design 1):
 *        q(x) = prod_t w_t(x_t) * N(x),  Z = sum_x q(x),  p = q / Z,
 *    where w_t(v) is the model's probability of token v at position t (a
 *    one-hot weight for a committed position) and N(x) is the number of
 *    accepting paths from s0 labelled x (1 or 0 for a DFA, the path count for
 *    an NFA, page 1 "Arbitrary schedules and NFAs").
 *  - The latent at step t is the edge taken; transition and emission factors
 *    are indicators (page 1, same section), so the per-step transition weight
 *    of edge e is W_t(e) = sum_{v in label(e)} w_t(v) and the state-level
 *    matrix is M_t(s, s') = sum_{e: s->s'} W_t(e) (page 2, key design 1).
 *  - Z, the state posteriors and the per-token constrained marginals
 *    p(x_t = v | x^t, C) come from plain chain forward-backward (page 1: exact
 *    sampling, marginals and normalisation "fall out of forward-backward
 *    message passing"; page 2, key design 3 for the marginals), done here in
 *    log space so no range is lost.  The oracle never uses the log-depth tree.
 *  - Exact samples come from forward filtering / backward sampling along the
 *    chain: the final state from the forward message restricted to F, then each
 *    earlier edge given the later state, then a token of that edge in
 *    proportion to w_t (page 1: sampling is exact, every token emitted from its
 *    edge's label set).  Its random numbers come from its own splitmix64
 *    stream, so draws are compared with the GPU only in distribution.
 *  - The remasking commit: the k positions with the highest constrained
 *    marginal of their sampled token among the masked ones (page 2, key design
 *    3, "Mar"; page 1, "Constrained remasking confidence", LLaDA's highest
 *    probability rule), ties to the lower position.
 *  - Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *    Easy as 1, 2, 3", SC'11), as published, for cross-checking a device
 *    generator.
 *
 * Canonical compiled form (shared definition, independent implementation):
 *  label sets sorted ascending with duplicates removed; edges by source sorted
 *  by (src, dst, id); edges by destination sorted by (dst, src, id); the
 *  token->edge incidence sorted by (token, src, dst, id).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_INVALID 1
#define OR_NOMEM 2
#define OR_EMPTY 3

typedef struct or_fa {
    int S, start, E, V, n_accept;
    int32_t *accept;          /* sorted unique */
    unsigned char *is_accept; /* [S] */
    int32_t *src, *dst;       /* [E] */
    int64_t *lab_off;         /* [E+1] */
    int32_t *lab_tok;         /* [I] */
    int64_t I;
    int32_t *src_off, *src_edges; /* [S+1], [E] */
    int32_t *dst_off, *dst_edges; /* [S+1], [E] */
    int64_t *tok_off;             /* [V+1] */
    int32_t *tok_edges;           /* [I] */
    int is_dfa;
} or_fa;

/* ------------------------------------------------------------------ sorting helpers */

typedef struct { int32_t a, b, c, id; } key4;

static int cmp_key4(const void *x, const void *y) {
    const key4 *p = (const key4 *)x, *q = (const key4 *)y;
    if (p->a != q->a) return p->a < q->a ? -1 : 1;
    if (p->b != q->b) return p->b < q->b ? -1 : 1;
    if (p->c != q->c) return p->c < q->c ? -1 : 1;
    if (p->id != q->id) return p->id < q->id ? -1 : 1;
    return 0;
}

static int cmp_i32(const void *x, const void *y) {
    int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;
    return a < b ? -1 : (a > b);
}

void or_fa_free(or_fa *fa) {
    if (!fa) return;
    free(fa->accept); free(fa->is_accept); free(fa->src); free(fa->dst);
    free(fa->lab_off); free(fa->lab_tok); free(fa->src_off); free(fa->src_edges);
    free(fa->dst_off); free(fa->dst_edges); free(fa->tok_off); free(fa->tok_edges);
    free(fa);
}

/* Validate and build the canonical arrays.  Returns OR_OK or OR_INVALID/OR_NOMEM. */
int or_fa_new(int S, int start, const int32_t *accept, int n_accept, int E,
              const int32_t *src, const int32_t *dst, const int64_t *loff,
              const int32_t *ltok, int V, or_fa **out) {
    *out = NULL;
    if (S < 1 || V < 1 || E < 0 || n_accept < 0 || start < 0 || start >= S) return OR_INVALID;
    if (loff[0] != 0) return OR_INVALID;
    for (int i = 0; i < n_accept; i++)
        if (accept[i] < 0 || accept[i] >= S) return OR_INVALID;
    for (int e = 0; e < E; e++) {
        if (src[e] < 0 || src[e] >= S || dst[e] < 0 || dst[e] >= S) return OR_INVALID;
        if (loff[e + 1] <= loff[e]) return OR_INVALID; /* empty label set */
        for (int64_t j = loff[e]; j < loff[e + 1]; j++)
            if (ltok[j] < 0 || ltok[j] >= V) return OR_INVALID;
    }
    or_fa *fa = (or_fa *)calloc(1, sizeof(or_fa));
    if (!fa) return OR_NOMEM;
    fa->S = S; fa->start = start; fa->E = E; fa->V = V;

    /* accepting set, deduplicated */
    fa->is_accept = (unsigned char *)calloc((size_t)S, 1);
    fa->accept = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_accept > 0 ? n_accept : 1));
    for (int i = 0; i < n_accept; i++) fa->is_accept[accept[i]] = 1;
    for (int s = 0; s < S; s++) if (fa->is_accept[s]) fa->accept[fa->n_accept++] = s;

    fa->src = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    fa->dst = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    memcpy(fa->src, src, sizeof(int32_t) * (size_t)E);
    memcpy(fa->dst, dst, sizeof(int32_t) * (size_t)E);

    /* label sets: sort each, drop repeats */
    int64_t total = loff[E];
    fa->lab_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
    fa->lab_tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total > 0 ? total : 1));
    int64_t w = 0;
    fa->lab_off[0] = 0;
    for (int e = 0; e < E; e++) {
        int64_t n = loff[e + 1] - loff[e];
        int32_t *tmp = fa->lab_tok + w;
        memcpy(tmp, ltok + loff[e], sizeof(int32_t) * (size_t)n);
        qsort(tmp, (size_t)n, sizeof(int32_t), cmp_i32);
        int64_t k = 0;
        for (int64_t j = 0; j < n; j++)
            if (k == 0 || tmp[j] != tmp[k - 1]) tmp[k++] = tmp[j];
        w += k;
        fa->lab_off[e + 1] = w;
    }
    fa->I = w;

    /* edges by source and by destination */
    key4 *ks = (key4 *)malloc(sizeof(key4) * (size_t)(E > 0 ? E : 1));
    fa->src_off = (int32_t *)calloc((size_t)S + 1, sizeof(int32_t));
    fa->dst_off = (int32_t *)calloc((size_t)S + 1, sizeof(int32_t));
    fa->src_edges = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    fa->dst_edges = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; e++) { ks[e].a = src[e]; ks[e].b = dst[e]; ks[e].c = 0; ks[e].id = e; }
    qsort(ks, (size_t)E, sizeof(key4), cmp_key4);
    for (int e = 0; e < E; e++) { fa->src_edges[e] = ks[e].id; fa->src_off[ks[e].a + 1]++; }
    for (int e = 0; e < E; e++) { ks[e].a = dst[e]; ks[e].b = src[e]; ks[e].c = 0; ks[e].id = e; }
    qsort(ks, (size_t)E, sizeof(key4), cmp_key4);
    for (int e = 0; e < E; e++) { fa->dst_edges[e] = ks[e].id; fa->dst_off[ks[e].a + 1]++; }
    for (int s = 0; s < S; s++) { fa->src_off[s + 1] += fa->src_off[s]; fa->dst_off[s + 1] += fa->dst_off[s]; }
    free(ks);

    /* token -> edge incidence */
    key4 *ki = (key4 *)malloc(sizeof(key4) * (size_t)(fa->I > 0 ? fa->I : 1));
    int64_t p = 0;
    for (int e = 0; e < E; e++)
        for (int64_t j = fa->lab_off[e]; j < fa->lab_off[e + 1]; j++) {
            ki[p].a = fa->lab_tok[j]; ki[p].b = src[e]; ki[p].c = dst[e]; ki[p].id = e; p++;
        }
    qsort(ki, (size_t)fa->I, sizeof(key4), cmp_key4);
    fa->tok_off = (int64_t *)calloc((size_t)V + 1, sizeof(int64_t));
    fa->tok_edges = (int32_t *)malloc(sizeof(int32_t) * (size_t)(fa->I > 0 ? fa->I : 1));
    fa->is_dfa = 1;
    for (int64_t j = 0; j < fa->I; j++) {
        fa->tok_edges[j] = ki[j].id;
        fa->tok_off[ki[j].a + 1]++;
        if (j > 0 && ki[j].a == ki[j - 1].a && ki[j].b == ki[j - 1].b) fa->is_dfa = 0;
    }
    for (int v = 0; v < V; v++) fa->tok_off[v + 1] += fa->tok_off[v];
    free(ki);
    *out = fa;
    return OR_OK;
}

void or_fa_sizes(const or_fa *fa, int64_t *n_edges, int64_t *n_incidences, int32_t *is_dfa,
                 int32_t *n_accept) {
    *n_edges = fa->E; *n_incidences = fa->I; *is_dfa = fa->is_dfa; *n_accept = fa->n_accept;
}

void or_fa_export(const or_fa *fa, int64_t *lab_off, int32_t *lab_tok, int32_t *src_off,
                  int32_t *src_edges, int32_t *dst_off, int32_t *dst_edges, int64_t *tok_off,
                  int32_t *tok_edges, int32_t *accept) {
    memcpy(lab_off, fa->lab_off, sizeof(int64_t) * (size_t)(fa->E + 1));
    memcpy(lab_tok, fa->lab_tok, sizeof(int32_t) * (size_t)fa->I);
    memcpy(src_off, fa->src_off, sizeof(int32_t) * (size_t)(fa->S + 1));
    memcpy(src_edges, fa->src_edges, sizeof(int32_t) * (size_t)fa->E);
    memcpy(dst_off, fa->dst_off, sizeof(int32_t) * (size_t)(fa->S + 1));
    memcpy(dst_edges, fa->dst_edges, sizeof(int32_t) * (size_t)fa->E);
    memcpy(tok_off, fa->tok_off, sizeof(int64_t) * (size_t)(fa->V + 1));
    memcpy(tok_edges, fa->tok_edges, sizeof(int32_t) * (size_t)fa->I);
    memcpy(accept, fa->accept, sizeof(int32_t) * (size_t)fa->n_accept);
}

/* ------------------------------------------------------------------ emission weights */

/* W[t*E + e] = sum_{v in label(e)} w_t(v), with w_t = probs row t, or the indicator of
 * the committed token. */
static void edge_weights(const or_fa *fa, int L, const float *probs, const int32_t *committed,
                         double *W) {
    const int E = fa->E, V = fa->V;
    for (int t = 0; t < L; t++) {
        double *Wt = W + (size_t)t * (size_t)E;
        int c = committed ? committed[t] : -1;
        if (c >= 0) {
            for (int e = 0; e < E; e++) Wt[e] = 0.0;
            for (int64_t j = fa->tok_off[c]; j < fa->tok_off[c + 1]; j++) Wt[fa->tok_edges[j]] += 1.0;
        } else {
            const float *row = probs + (size_t)t * (size_t)V;
            for (int e = 0; e < E; e++) {
                double acc = 0.0;
                for (int64_t j = fa->lab_off[e]; j < fa->lab_off[e + 1]; j++) acc += (double)row[fa->lab_tok[j]];
                Wt[e] = acc;
            }
        }
    }
}

/* The state-level transition matrix of one position, M(s, s') = sum_{e: s->s'} W(e). */
int or_transition_matrix(const or_fa *fa, const float *probs_row, int32_t committed_token,
                         double *M) {
    double *W = (double *)malloc(sizeof(double) * (size_t)(fa->E > 0 ? fa->E : 1));
    if (!W) return OR_NOMEM;
    edge_weights(fa, 1, probs_row, &committed_token, W);
    memset(M, 0, sizeof(double) * (size_t)fa->S * (size_t)fa->S);
    for (int e = 0; e < fa->E; e++) M[(size_t)fa->src[e] * fa->S + fa->dst[e]] += W[e];
    free(W);
    return OR_OK;
}

/* ------------------------------------------------------------------ forward-backward */

static double lse_pair(double m, double acc) { return m + log(acc); }

/* log_alpha[t][s]: log total weight of paths from s0 that read positions 1..t and sit in s.
 * log_beta[t][s]: log total weight of paths from s that read positions t+1..L and end in F. */
static void forward_backward(const or_fa *fa, int L, const double *W, double *la, double *lb) {
    const int S = fa->S, E = fa->E;
    for (int s = 0; s < S; s++) la[s] = (s == fa->start) ? 0.0 : -INFINITY;
    for (int t = 1; t <= L; t++) {
        const double *Wt = W + (size_t)(t - 1) * (size_t)E;
        const double *prev = la + (size_t)(t - 1) * S;
        double *cur = la + (size_t)t * S;
        for (int s = 0; s < S; s++) {
            double m = -INFINITY;
            for (int j = fa->dst_off[s]; j < fa->dst_off[s + 1]; j++) {
                int e = fa->dst_edges[j];
                if (Wt[e] <= 0.0 || prev[fa->src[e]] == -INFINITY) continue;
                double x = prev[fa->src[e]] + log(Wt[e]);
                if (x > m) m = x;
            }
            if (m == -INFINITY) { cur[s] = -INFINITY; continue; }
            double acc = 0.0;
            for (int j = fa->dst_off[s]; j < fa->dst_off[s + 1]; j++) {
                int e = fa->dst_edges[j];
                if (Wt[e] <= 0.0 || prev[fa->src[e]] == -INFINITY) continue;
                acc += exp(prev[fa->src[e]] + log(Wt[e]) - m);
            }
            cur[s] = lse_pair(m, acc);
        }
    }
    double *last = lb + (size_t)L * S;
    for (int s = 0; s < S; s++) last[s] = fa->is_accept[s] ? 0.0 : -INFINITY;
    for (int t = L; t >= 1; t--) {
        const double *Wt = W + (size_t)(t - 1) * (size_t)E;
        const double *next = lb + (size_t)t * S;
        double *cur = lb + (size_t)(t - 1) * S;
        for (int s = 0; s < S; s++) {
            double m = -INFINITY;
            for (int j = fa->src_off[s]; j < fa->src_off[s + 1]; j++) {
                int e = fa->src_edges[j];
                if (Wt[e] <= 0.0 || next[fa->dst[e]] == -INFINITY) continue;
                double x = log(Wt[e]) + next[fa->dst[e]];
                if (x > m) m = x;
            }
            if (m == -INFINITY) { cur[s] = -INFINITY; continue; }
            double acc = 0.0;
            for (int j = fa->src_off[s]; j < fa->src_off[s + 1]; j++) {
                int e = fa->src_edges[j];
                if (Wt[e] <= 0.0 || next[fa->dst[e]] == -INFINITY) continue;
                acc += exp(log(Wt[e]) + next[fa->dst[e]] - m);
            }
            cur[s] = lse_pair(m, acc);
        }
    }
}

/* log of the constrained marginal p(x_t = v | x^t, C) for 1 <= t <= L. */
static double log_token_marginal(const or_fa *fa, int t, int v, const float *probs,
                                 const int32_t *committed, const double *la, const double *lb,
                                 double logZ) {
    const int S = fa->S;
    double lw;
    int c = committed ? committed[t - 1] : -1;
    if (c >= 0) {
        if (v != c) return -INFINITY;
        lw = 0.0;
    } else {
        double pv = (double)probs[(size_t)(t - 1) * fa->V + v];
        if (pv <= 0.0) return -INFINITY;
        lw = log(pv);
    }
    const double *a = la + (size_t)(t - 1) * S, *b = lb + (size_t)t * S;
    double m = -INFINITY;
    for (int64_t j = fa->tok_off[v]; j < fa->tok_off[v + 1]; j++) {
        int e = fa->tok_edges[j];
        double x = a[fa->src[e]] + b[fa->dst[e]];
        if (x > m) m = x;
    }
    if (m == -INFINITY) return -INFINITY;
    double acc = 0.0;
    for (int64_t j = fa->tok_off[v]; j < fa->tok_off[v + 1]; j++) {
        int e = fa->tok_edges[j];
        double x = a[fa->src[e]] + b[fa->dst[e]];
        if (x != -INFINITY) acc += exp(x - m);
    }
    return lw + m + log(acc) - logZ;
}

/*
 * One sequence: logZ, and optionally the marginals of given tokens [L], every
 * token's marginal [L*V], the state posteriors [(L+1)*S] and the log messages.
 * Returns OR_OK, or OR_EMPTY when no accepted string has positive weight (logZ=-inf).
 */
int or_posterior(const or_fa *fa, int L, const float *probs, const int32_t *committed,
                 const int32_t *tokens, double *logZ, double *marg_tokens, double *marg_all,
                 double *state_post, double *log_alpha, double *log_beta) {
    const int S = fa->S;
    double *W = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)(fa->E > 0 ? fa->E : 1));
    double *la = (double *)malloc(sizeof(double) * (size_t)(L + 1) * S);
    double *lb = (double *)malloc(sizeof(double) * (size_t)(L + 1) * S);
    if (!W || !la || !lb) { free(W); free(la); free(lb); return OR_NOMEM; }
    edge_weights(fa, L, probs, committed, W);
    forward_backward(fa, L, W, la, lb);
    const double *fin = la + (size_t)L * S;
    double m = -INFINITY;
    for (int i = 0; i < fa->n_accept; i++) if (fin[fa->accept[i]] > m) m = fin[fa->accept[i]];
    double lz = -INFINITY;
    if (m != -INFINITY) {
        double acc = 0.0;
        for (int i = 0; i < fa->n_accept; i++)
            if (fin[fa->accept[i]] != -INFINITY) acc += exp(fin[fa->accept[i]] - m);
        lz = m + log(acc);
    }
    *logZ = lz;
    int status = (lz == -INFINITY) ? OR_EMPTY : OR_OK;
    if (status == OR_OK) {
        if (marg_tokens)
            for (int t = 1; t <= L; t++)
                marg_tokens[t - 1] = exp(log_token_marginal(fa, t, tokens[t - 1], probs, committed, la, lb, lz));
        if (marg_all)
            for (int t = 1; t <= L; t++)
                for (int v = 0; v < fa->V; v++)
                    marg_all[(size_t)(t - 1) * fa->V + v] =
                        exp(log_token_marginal(fa, t, v, probs, committed, la, lb, lz));
        if (state_post)
            for (size_t i = 0; i < (size_t)(L + 1) * S; i++) {
                double x = la[i] + lb[i];
                state_post[i] = (x == -INFINITY) ? 0.0 : exp(x - lz);
            }
    }
    if (log_alpha) memcpy(log_alpha, la, sizeof(double) * (size_t)(L + 1) * S);
    if (log_beta) memcpy(log_beta, lb, sizeof(double) * (size_t)(L + 1) * S);
    free(W); free(la); free(lb);
    return status;
}

/* ------------------------------------------------------------------ sampling */

static uint64_t splitmix64(uint64_t *s) {
    uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static double uniform01(uint64_t *s) { return (double)(splitmix64(s) >> 11) * (1.0 / 9007199254740992.0); }

/* Pick index i with probability w[i] / sum(w); weights are non-negative. */
static int categorical(const double *w, int n, uint64_t *rng) {
    double tot = 0.0;
    for (int i = 0; i < n; i++) tot += w[i];
    double u = uniform01(rng) * tot, c = 0.0;
    int last = -1;
    for (int i = 0; i < n; i++) {
        if (w[i] <= 0.0) continue;
        last = i;
        c += w[i];
        if (u < c) return i;
    }
    return last;
}

/* n_samples exact draws from p (forward filtering, backward sampling); out is [n_samples, L]. */
int or_sample(const or_fa *fa, int L, const float *probs, const int32_t *committed,
              uint64_t seed, int n_samples, int32_t *out) {
    const int S = fa->S, E = fa->E;
    double *W = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)(E > 0 ? E : 1));
    double *la = (double *)malloc(sizeof(double) * (size_t)(L + 1) * S);
    double *lb = (double *)malloc(sizeof(double) * (size_t)(L + 1) * S);
    int maxdeg = 1;
    for (int s = 0; s < S; s++) if (fa->dst_off[s + 1] - fa->dst_off[s] > maxdeg) maxdeg = fa->dst_off[s + 1] - fa->dst_off[s];
    int64_t maxlab = 1;
    for (int e = 0; e < E; e++) if (fa->lab_off[e + 1] - fa->lab_off[e] > maxlab) maxlab = fa->lab_off[e + 1] - fa->lab_off[e];
    double *buf = (double *)malloc(sizeof(double) * (size_t)(maxdeg > maxlab ? maxdeg : maxlab) + sizeof(double) * (size_t)(S + 1));
    if (!W || !la || !lb || !buf) { free(W); free(la); free(lb); free(buf); return OR_NOMEM; }
    edge_weights(fa, L, probs, committed, W);
    forward_backward(fa, L, W, la, lb);
    const double *fin = la + (size_t)L * S;
    double m = -INFINITY;
    for (int i = 0; i < fa->n_accept; i++) if (fin[fa->accept[i]] > m) m = fin[fa->accept[i]];
    if (m == -INFINITY) { free(W); free(la); free(lb); free(buf); return OR_EMPTY; }
    uint64_t rng = seed;
    for (int n = 0; n < n_samples; n++) {
        int32_t *x = out + (size_t)n * L;
        for (int i = 0; i < fa->n_accept; i++) {
            double a = fin[fa->accept[i]];
            buf[i] = (a == -INFINITY) ? 0.0 : exp(a - m);
        }
        int z = fa->accept[categorical(buf, fa->n_accept, &rng)];
        for (int t = L; t >= 1; t--) {
            const double *Wt = W + (size_t)(t - 1) * E;
            const double *prev = la + (size_t)(t - 1) * S;
            int lo = fa->dst_off[z], hi = fa->dst_off[z + 1];
            double mm = -INFINITY;
            for (int j = lo; j < hi; j++) {
                int e = fa->dst_edges[j];
                if (Wt[e] > 0.0 && prev[fa->src[e]] != -INFINITY) {
                    double xx = prev[fa->src[e]] + log(Wt[e]);
                    if (xx > mm) mm = xx;
                }
            }
            for (int j = lo; j < hi; j++) {
                int e = fa->dst_edges[j];
                buf[j - lo] = (Wt[e] > 0.0 && prev[fa->src[e]] != -INFINITY)
                                  ? exp(prev[fa->src[e]] + log(Wt[e]) - mm) : 0.0;
            }
            int e = fa->dst_edges[lo + categorical(buf, hi - lo, &rng)];
            int c = committed ? committed[t - 1] : -1;
            if (c >= 0) {
                x[t - 1] = c;
            } else {
                const float *row = probs + (size_t)(t - 1) * fa->V;
                int64_t a = fa->lab_off[e], b = fa->lab_off[e + 1];
                for (int64_t j = a; j < b; j++) buf[j - a] = (double)row[fa->lab_tok[j]];
                x[t - 1] = fa->lab_tok[a + categorical(buf, (int)(b - a), &rng)];
            }
            z = fa->src[e];
        }
    }
    free(W); free(la); free(lb); free(buf);
    return OR_OK;
}

/* ------------------------------------------------------------------ acceptor, commit */

/* Number of accepting paths from s0 labelled with tokens[0..L) (0 = rejected). */
double or_path_count(const or_fa *fa, int L, const int32_t *tokens) {
    const int S = fa->S;
    double *cur = (double *)calloc((size_t)S, sizeof(double));
    double *nxt = (double *)calloc((size_t)S, sizeof(double));
    cur[fa->start] = 1.0;
    for (int t = 0; t < L; t++) {
        memset(nxt, 0, sizeof(double) * (size_t)S);
        int v = tokens[t];
        if (v >= 0 && v < fa->V)
            for (int64_t j = fa->tok_off[v]; j < fa->tok_off[v + 1]; j++) {
                int e = fa->tok_edges[j];
                nxt[fa->dst[e]] += cur[fa->src[e]];
            }
        double *tmp = cur; cur = nxt; nxt = tmp;
    }
    double n = 0.0;
    for (int i = 0; i < fa->n_accept; i++) n += cur[fa->accept[i]];
    free(cur); free(nxt);
    return n;
}

/* The k masked positions of [lo, hi) with the largest marginal, in descending order, ties
 * to the lower position; -1 pads when fewer are eligible. */
void or_topk(int L, const double *marg, const int32_t *committed, int k, int lo, int hi,
             int32_t *out) {
    int n = 0;
    for (int i = 0; i < k; i++) out[i] = -1;
    unsigned char *used = (unsigned char *)calloc((size_t)(L > 0 ? L : 1), 1);
    for (int r = 0; r < k; r++) {
        int best = -1;
        for (int t = (lo > 0 ? lo : 0); t < (hi < L ? hi : L); t++) {
            if (committed[t] >= 0 || used[t]) continue;
            if (best < 0 || marg[t] > marg[best]) best = t;
        }
        if (best < 0) break;
        used[best] = 1;
        out[n++] = best;
    }
    free(used);
}

/* ------------------------------------------------------------------ Philox4x32-10 */

void or_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; r++) {
        if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}
