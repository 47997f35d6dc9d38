// Host side of the C ABI: automaton compilation (validation, canonical CSR, cell layout,
// row blocks), upload, query, export and the thread-local error string.
//
// The automaton is the hidden Markov model of the paperfeed.app summary of "Constrained
// Decoding for Diffusion Language Models via Efficient Inference over Finite Automata"
// (section "The insight: the constraint is a hidden Markov model"): latent = the edge taken,
// transition = the edges chain, emission = the token lies in the edge's label set.
#include <algorithm>
#include <climits>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

#include "fa_internal.cuh"

static thread_local std::string g_last_error;

void fa_set_error(const std::string &msg) { g_last_error = msg; }

extern "C" const char *fa_last_error(void) { return g_last_error.c_str(); }

namespace {

struct BlobBuilder {
    struct Item { void **dst; const void *src; size_t bytes; size_t off; };
    std::vector<Item> items;
    size_t total = 0;
    template <class T>
    void add(T **dst, const std::vector<T> &v) {
        size_t bytes = v.size() * sizeof(T);
        total = (total + 255) & ~size_t(255);
        items.push_back({(void **)dst, v.data(), bytes, total});
        total += bytes > 0 ? bytes : sizeof(T);
    }
};

fa_status cuda_fail(const char *what, cudaError_t e) {
    fa_set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return e == cudaErrorMemoryAllocation ? FA_ERR_OOM : FA_ERR_CUDA;
}

}  // namespace

extern "C" fa_status fa_compile(int32_t n_states, int32_t start, const int32_t *accept, int32_t n_accept,
                                int32_t n_edges, const int32_t *edge_src, const int32_t *edge_dst,
                                const int64_t *label_offsets, const int32_t *label_tokens, int32_t vocab,
                                fa_stream stream, fa_automaton **out) {
    if (!out) { fa_set_error("fa_compile: out is NULL"); return FA_ERR_INVALID_ARG; }
    *out = nullptr;
    const int S = n_states, V = vocab, E = n_edges;
    if (S < 1 || S > FA_MAX_STATES) { fa_set_error("fa_compile: n_states out of [1, FA_MAX_STATES]"); return FA_ERR_INVALID_ARG; }
    if (V < 1) { fa_set_error("fa_compile: vocab < 1"); return FA_ERR_INVALID_ARG; }
    if (E < 0 || n_accept < 0) { fa_set_error("fa_compile: negative count"); return FA_ERR_INVALID_ARG; }
    if (start < 0 || start >= S) { fa_set_error("fa_compile: start state out of range"); return FA_ERR_INVALID_ARG; }
    if ((n_accept > 0 && !accept) || (E > 0 && (!edge_src || !edge_dst || !label_tokens)) || !label_offsets) {
        fa_set_error("fa_compile: NULL array"); return FA_ERR_INVALID_ARG;
    }
    if (label_offsets[0] != 0) { fa_set_error("fa_compile: label_offsets[0] != 0"); return FA_ERR_INVALID_ARG; }
    for (int i = 0; i < n_accept; ++i)
        if (accept[i] < 0 || accept[i] >= S) { fa_set_error("fa_compile: accepting state out of range"); return FA_ERR_INVALID_ARG; }
    for (int e = 0; e < E; ++e) {
        if (edge_src[e] < 0 || edge_src[e] >= S || edge_dst[e] < 0 || edge_dst[e] >= S) {
            fa_set_error("fa_compile: edge endpoint out of range"); return FA_ERR_INVALID_ARG;
        }
        if (label_offsets[e + 1] <= label_offsets[e]) {
            fa_set_error("fa_compile: empty label set (edge " + std::to_string(e) + ")"); return FA_ERR_INVALID_ARG;
        }
    }
    const int64_t raw_total = label_offsets[E];
    for (int64_t j = 0; j < raw_total; ++j)
        if (label_tokens[j] < 0 || label_tokens[j] >= V) { fa_set_error("fa_compile: token id out of range"); return FA_ERR_INVALID_ARG; }

    fa_automaton *a = new fa_automaton();
    a->S = S; a->V = V; a->E = E; a->start = start;
    cudaGetDevice(&a->device);

    // accepting set
    std::vector<int32_t> acc_mask(S, 0), acc;
    for (int i = 0; i < n_accept; ++i) acc_mask[accept[i]] = 1;
    for (int s = 0; s < S; ++s) if (acc_mask[s]) acc.push_back(s);
    a->n_accept = (int)acc.size();

    // canonical label sets
    std::vector<int64_t> lab_off(E + 1, 0);
    std::vector<int32_t> lab_tok;
    lab_tok.reserve((size_t)raw_total);
    for (int e = 0; e < E; ++e) {
        std::vector<int32_t> tmp(label_tokens + label_offsets[e], label_tokens + label_offsets[e + 1]);
        std::sort(tmp.begin(), tmp.end());
        tmp.erase(std::unique(tmp.begin(), tmp.end()), tmp.end());
        lab_tok.insert(lab_tok.end(), tmp.begin(), tmp.end());
        lab_off[e + 1] = (int64_t)lab_tok.size();
    }
    const int64_t I = (int64_t)lab_tok.size();
    a->I = I;

    // edges by (src, dst, id) and by (dst, src, id)
    std::vector<int32_t> src_edges(E), dst_edges(E), src_off(S + 1, 0), dst_off(S + 1, 0);
    std::iota(src_edges.begin(), src_edges.end(), 0);
    std::iota(dst_edges.begin(), dst_edges.end(), 0);
    std::stable_sort(src_edges.begin(), src_edges.end(), [&](int x, int y) {
        return edge_src[x] != edge_src[y] ? edge_src[x] < edge_src[y] : edge_dst[x] < edge_dst[y];
    });
    std::stable_sort(dst_edges.begin(), dst_edges.end(), [&](int x, int y) {
        return edge_dst[x] != edge_dst[y] ? edge_dst[x] < edge_dst[y] : edge_src[x] < edge_src[y];
    });
    for (int e = 0; e < E; ++e) { src_off[edge_src[e] + 1]++; dst_off[edge_dst[e] + 1]++; }
    for (int s = 0; s < S; ++s) { src_off[s + 1] += src_off[s]; dst_off[s + 1] += dst_off[s]; }

    // token -> edge incidence: a counting sort by token over edges visited in (src, dst, id)
    // order leaves every token's bucket sorted by (src, dst, id)
    std::vector<int64_t> tok_off(V + 1, 0);
    for (int64_t j = 0; j < I; ++j) tok_off[lab_tok[j] + 1]++;
    for (int v = 0; v < V; ++v) tok_off[v + 1] += tok_off[v];
    std::vector<int32_t> tok_edges(I);
    {
        std::vector<int64_t> fill(tok_off.begin(), tok_off.end() - 1);
        for (int q = 0; q < E; ++q) {
            int e = src_edges[q];
            for (int64_t j = lab_off[e]; j < lab_off[e + 1]; ++j) tok_edges[fill[lab_tok[j]]++] = e;
        }
    }
    int is_dfa = 1;
    for (int v = 0; v < V && is_dfa; ++v)
        for (int64_t j = tok_off[v] + 1; j < tok_off[v + 1]; ++j)
            if (edge_src[tok_edges[j]] == edge_src[tok_edges[j - 1]]) { is_dfa = 0; break; }
    a->is_dfa = is_dfa;

    // cells: distinct (src, dst) pairs in (src, dst) order, tokens = sorted multiset union
    std::vector<int32_t> row_cell_off(S + 1, 0), cell_dst, cell_src;
    std::vector<int64_t> cell_off(1, 0);
    std::vector<int32_t> cell_tok;
    cell_tok.reserve((size_t)I);
    std::vector<int64_t> row_cost(S, 0);
    int32_t max_cell_len = 0;
    for (int q = 0; q < E;) {
        int e0 = src_edges[q];
        int s = edge_src[e0], d = edge_dst[e0];
        size_t begin = cell_tok.size();
        while (q < E && edge_src[src_edges[q]] == s && edge_dst[src_edges[q]] == d) {
            int e = src_edges[q];
            cell_tok.insert(cell_tok.end(), lab_tok.begin() + lab_off[e], lab_tok.begin() + lab_off[e + 1]);
            ++q;
        }
        std::sort(cell_tok.begin() + begin, cell_tok.end());
        int32_t len = (int32_t)(cell_tok.size() - begin);
        max_cell_len = std::max(max_cell_len, len);
        cell_dst.push_back(d);
        cell_src.push_back(s);
        cell_off.push_back((int64_t)cell_tok.size());
        row_cell_off[s + 1]++;
        row_cost[s] += len + 16;  // a cell's gather length plus a fixed per-cell cost
    }
    for (int s = 0; s < S; ++s) row_cell_off[s + 1] += row_cell_off[s];
    a->n_cells = (int32_t)cell_dst.size();
    a->max_cell_len = max_cell_len;

    // Reweight layout (sliced, ELL-like).  The vocabulary is read in chunks of CH tokens
    // staged in shared memory.  Every cell's tokens in a chunk are cut into pieces of at most
    // FA_PIECE_TOKENS; piece ids are cell-major (cell c owns pieces [pc[c], pc[c+1])).  For
    // each (chunk, row) the row's pieces, longest first, form slices of 32: lane l of a slice
    // sums piece l, reading 16-byte groups of 8 in-chunk token indices stored interleaved
    // (group k of lane l at slice_start + 32 k + l, padded with the index CH, a zero slot).
    const int CH = (V <= FA_REWEIGHT_MAX_CHUNK) ? V : FA_REWEIGHT_MAX_CHUNK;
    const int nch = (V + CH - 1) / CH;
    a->chunk_tokens = CH;
    a->n_chunks = nch;
    struct Piece { int32_t cell, chunk; int64_t first; int32_t len; };
    std::vector<Piece> pieces;
    std::vector<int32_t> pc(a->n_cells + 1, 0);
    for (int c = 0; c < a->n_cells; ++c) {
        pc[c] = (int32_t)pieces.size();
        const int32_t *b0 = cell_tok.data() + cell_off[c], *b1 = cell_tok.data() + cell_off[c + 1];
        for (int ch = 0; ch < nch; ++ch) {
            const int32_t lo = ch * CH, hi = (int32_t)std::min<int64_t>((int64_t)(ch + 1) * CH, V);
            const int32_t *q0 = std::lower_bound(b0, b1, lo), *q1 = std::lower_bound(b0, b1, hi);
            for (const int32_t *q = q0; q < q1; q += FA_PIECE_TOKENS)
                pieces.push_back({c, ch, (int64_t)(q - cell_tok.data()), (int32_t)std::min<int64_t>(FA_PIECE_TOKENS, q1 - q)});
        }
    }
    pc[a->n_cells] = (int32_t)pieces.size();
    std::vector<int32_t> row_pieces(S, 0);
    for (auto &pz : pieces) row_pieces[cell_src[pz.cell]]++;
    {
        // dynamic shared memory of the reweight: staged chunk, per-piece sums, per-row maxima
        const long budget = 232448L - 256 - 4L * (CH + 4) - 4L * S;
        a->max_unit_pieces = (int32_t)std::min<long>(1 << 20, budget / 4);
        int32_t mx = 0;
        for (int r = 0; r < S; ++r) mx = std::max(mx, row_pieces[r]);
        if (mx > a->max_unit_pieces) { delete a; fa_set_error("fa_compile: a state has too many token pieces for one block"); return FA_ERR_UNSUPPORTED; }
    }
    std::vector<int32_t> sl_row_off((size_t)nch * (S + 1)), sl_goff(1, 0), sl_piece;
    std::vector<uint16_t> tok8;
    {
        std::vector<std::vector<int32_t>> by_row(S);
        for (int ch = 0; ch < nch; ++ch) {
            for (auto &v : by_row) v.clear();
            for (int32_t pid = 0; pid < (int32_t)pieces.size(); ++pid)
                if (pieces[pid].chunk == ch) by_row[cell_src[pieces[pid].cell]].push_back(pid);
            for (int r = 0; r < S; ++r) {
                sl_row_off[(size_t)ch * (S + 1) + r] = (int32_t)(sl_goff.size() - 1);
                auto &v = by_row[r];
                std::stable_sort(v.begin(), v.end(), [&](int32_t x, int32_t y) { return pieces[x].len > pieces[y].len; });
                for (size_t s0 = 0; s0 < v.size(); s0 += 32) {
                    const size_t n = std::min<size_t>(32, v.size() - s0);
                    int32_t len = 0;
                    for (size_t l = 0; l < n; ++l) len = std::max(len, (pieces[v[s0 + l]].len + 7) / 8);
                    const size_t g0 = tok8.size() / 8;
                    tok8.resize(tok8.size() + (size_t)len * 32 * 8, (uint16_t)CH);
                    for (size_t l = 0; l < 32; ++l) {
                        sl_piece.push_back(l < n ? v[s0 + l] : -1);
                        if (l >= n) continue;
                        const Piece &pz = pieces[v[s0 + l]];
                        for (int32_t j = 0; j < pz.len; ++j)
                            tok8[(g0 + (size_t)(j / 8) * 32 + l) * 8 + (j % 8)] =
                                (uint16_t)(cell_tok[pz.first + j] - (int32_t)ch * CH);
                    }
                    // spread the 32 lanes' gathers of each group position over distinct banks:
                    // permute the 8 entries of every group (their sum is order-free)
                    for (int32_t k = 0; k < len; ++k) {
                        uint16_t rem[32][8];
                        int nrem[32];
                        for (int l = 0; l < 32; ++l) {
                            nrem[l] = 8;
                            for (int h = 0; h < 8; ++h) rem[l][h] = tok8[(g0 + (size_t)k * 32 + l) * 8 + h];
                        }
                        for (int h = 0; h < 8; ++h) {
                            int used[33] = {0};
                            for (int l = 0; l < 32; ++l) {
                                int best = 0, bc = 1 << 30;
                                for (int x = 0; x < nrem[l]; ++x) {
                                    const int cost = (rem[l][x] == (uint16_t)CH) ? used[32] : used[rem[l][x] & 31];
                                    if (cost < bc) { bc = cost; best = x; }
                                }
                                const uint16_t tk = rem[l][best];
                                rem[l][best] = rem[l][--nrem[l]];
                                used[tk == (uint16_t)CH ? 32 : (tk & 31)]++;
                                tok8[(g0 + (size_t)k * 32 + l) * 8 + h] = tk;
                            }
                        }
                    }
                    sl_goff.push_back((int32_t)(tok8.size() / 8));
                }
            }
            sl_row_off[(size_t)ch * (S + 1) + S] = (int32_t)(sl_goff.size() - 1);
        }
        if (tok8.size() / 8 > (size_t)INT32_MAX) { delete a; fa_set_error("fa_compile: automaton too large"); return FA_ERR_INVALID_ARG; }
        tok8.resize(tok8.size() + 64, (uint16_t)CH);
    }
    a->n_slices = (int32_t)(sl_goff.size() - 1);

    // row blocks of balanced gather cost with at most max_unit_pieces pieces each, for target
    // block counts 1, 2, 4, ...
    int64_t total_cost = 0;
    for (int r = 0; r < S; ++r) total_cost += row_cost[r] + 1;
    std::vector<int32_t> rb, rbm;  // rbm: per block {r0, r1, first cell, end cell, first piece, pad}
    for (int target = 1; ; target *= 2) {
        const int64_t cap = std::max<int64_t>(1, (total_cost + target - 1) / target);
        a->part_first.push_back((int32_t)rb.size());
        rb.push_back(0);
        int64_t cost = 0;
        int32_t np = 0;
        for (int r = 0; r < S; ++r) {
            const int64_t rc = row_cost[r] + 1;
            if (r > rb.back() && (cost + rc > cap || np + row_pieces[r] > a->max_unit_pieces)) {
                rb.push_back(r);
                cost = 0;
                np = 0;
            }
            cost += rc;
            np += row_pieces[r];
        }
        rb.push_back(S);
        a->part_count.push_back((int32_t)(rb.size() - a->part_first.back() - 1));
        int32_t mp = 0, mr = 0;
        for (size_t q = a->part_first.back(); q + 1 < rb.size(); ++q) {
            mp = std::max(mp, pc[row_cell_off[rb[q + 1]]] - pc[row_cell_off[rb[q]]]);
            mr = std::max(mr, rb[q + 1] - rb[q]);
        }
        a->part_max_pieces.push_back(mp);
        a->part_max_rows.push_back(mr);
        for (size_t q = a->part_first.back(); q + 1 < rb.size(); ++q) {
            const int32_t c0 = row_cell_off[rb[q]], c1 = row_cell_off[rb[q + 1]];
            rbm.insert(rbm.end(), {rb[q], rb[q + 1], c0, c1, pc[c0], 0, 0, 0});
        }
        if (a->part_count.back() >= S || target >= 4096) break;
    }

    std::vector<int32_t> esrc(edge_src, edge_src + E), edst(edge_dst, edge_dst + E);

    BlobBuilder bb;
    bb.add(&a->lab_off, lab_off);
    bb.add(&a->lab_tok, lab_tok);
    bb.add(&a->src_off, src_off);
    bb.add(&a->src_edges, src_edges);
    bb.add(&a->dst_off, dst_off);
    bb.add(&a->dst_edges, dst_edges);
    bb.add(&a->tok_off, tok_off);
    bb.add(&a->tok_edges, tok_edges);
    bb.add(&a->accept, acc);
    bb.add(&a->accept_mask, acc_mask);
    bb.add(&a->edge_src, esrc);
    bb.add(&a->edge_dst, edst);
    bb.add(&a->row_cell_off, row_cell_off);
    bb.add(&a->cell_dst, cell_dst);
    bb.add(&a->cell_src, cell_src);
    bb.add(&a->cell_off, cell_off);
    bb.add(&a->cell_tok, cell_tok);
    bb.add(&a->rb_bounds, rb);
    bb.add(&a->rb_meta, rbm);
    bb.add(&a->tok8, tok8);
    bb.add(&a->piece_cell_off, pc);
    bb.add(&a->sl_row_off, sl_row_off);
    bb.add(&a->sl_goff, sl_goff);
    bb.add(&a->sl_piece, sl_piece);

    cudaError_t err = cudaMalloc(&a->blob, bb.total);
    if (err != cudaSuccess) { delete a; return cuda_fail("fa_compile: cudaMalloc", err); }
    a->blob_bytes = bb.total;
    cudaStream_t st = (cudaStream_t)stream;
    for (auto &it : bb.items) {
        *it.dst = (char *)a->blob + it.off;
        if (it.bytes) {
            err = cudaMemcpyAsync(*it.dst, it.src, it.bytes, cudaMemcpyHostToDevice, st);
            if (err != cudaSuccess) { cudaFree(a->blob); delete a; return cuda_fail("fa_compile: upload", err); }
        }
    }
    err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) { cudaFree(a->blob); delete a; return cuda_fail("fa_compile: synchronize", err); }
    *out = a;
    return FA_OK;
}

extern "C" fa_status fa_destroy(fa_automaton *aut) {
    if (!aut) return FA_OK;
    if (aut->blob) cudaFree(aut->blob);
    delete aut;
    return FA_OK;
}

extern "C" fa_status fa_query(const fa_automaton *aut, int64_t *n_edges, int64_t *n_incidences, int32_t *is_dfa,
                              int32_t *n_accept, int32_t *n_states, int32_t *vocab) {
    if (!aut) { fa_set_error("fa_query: NULL automaton"); return FA_ERR_INVALID_ARG; }
    if (n_edges) *n_edges = aut->E;
    if (n_incidences) *n_incidences = aut->I;
    if (is_dfa) *is_dfa = aut->is_dfa;
    if (n_accept) *n_accept = aut->n_accept;
    if (n_states) *n_states = aut->S;
    if (vocab) *vocab = aut->V;
    return FA_OK;
}

extern "C" fa_status fa_export_csr(const fa_automaton *aut, int64_t *lab_off, int32_t *lab_tok, int32_t *src_off,
                                   int32_t *src_edges, int32_t *dst_off, int32_t *dst_edges, int64_t *tok_off,
                                   int32_t *tok_edges, int32_t *accept) {
    if (!aut || !lab_off || !lab_tok || !src_off || !src_edges || !dst_off || !dst_edges || !tok_off || !tok_edges ||
        !accept) {
        fa_set_error("fa_export_csr: NULL argument");
        return FA_ERR_INVALID_ARG;
    }
    struct C { void *h; const void *d; size_t n; } cps[] = {
        {lab_off, aut->lab_off, sizeof(int64_t) * (size_t)(aut->E + 1)},
        {lab_tok, aut->lab_tok, sizeof(int32_t) * (size_t)aut->I},
        {src_off, aut->src_off, sizeof(int32_t) * (size_t)(aut->S + 1)},
        {src_edges, aut->src_edges, sizeof(int32_t) * (size_t)aut->E},
        {dst_off, aut->dst_off, sizeof(int32_t) * (size_t)(aut->S + 1)},
        {dst_edges, aut->dst_edges, sizeof(int32_t) * (size_t)aut->E},
        {tok_off, aut->tok_off, sizeof(int64_t) * (size_t)(aut->V + 1)},
        {tok_edges, aut->tok_edges, sizeof(int32_t) * (size_t)aut->I},
        {accept, aut->accept, sizeof(int32_t) * (size_t)aut->n_accept},
    };
    for (auto &c : cps) {
        if (!c.n) continue;
        cudaError_t err = cudaMemcpy(c.h, c.d, c.n, cudaMemcpyDeviceToHost);
        if (err != cudaSuccess) return cuda_fail("fa_export_csr", err);
    }
    return FA_OK;
}
