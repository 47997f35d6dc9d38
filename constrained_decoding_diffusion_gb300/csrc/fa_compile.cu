// Host side of the C ABI: automaton compilation (validation, canonical CSR, cell layout,
// row blocks), upload, query, export and the thread-local error string.
//
// The automaton is the hidden Markov model of the paperfeed.app summary of "Constrained
// Decoding for Diffusion Language Models via Efficient Inference over Finite Automata"
// (section "The insight: the constraint is a hidden Markov model"): latent = the edge taken,
// transition = the edges chain, emission = the token lies in the edge's label set.
#include <algorithm>
#include <climits>
#include <functional>
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

// Reweight layout (runs) over the cells of an automaton: see fa_automaton for the format.
// Returns an empty string, or what went wrong.
struct RunLayout {
    int32_t chunk_tokens = 0, n_chunks = 1, n_units = 0;
    std::vector<int32_t> row_unit0, crun_off, ru_goff, rbm, part_first, part_count, part_max_units, part_max_rows;
    std::vector<int64_t> part_tile_floats;
    std::vector<uint16_t> crun_slot, ru_tok;
};

// Entry order of one warp unit for one vocabulary chunk.  lr[l] holds lane l's runs (in slot
// order), each as its in-chunk token indices.  A run takes whole groups of FA_GROUP_ENTRIES
// entries (at least one), the first entry of its last group flagged with FA_RUN_END (the
// reweight reads a group's flag before summing it); every lane's stream is as
// long as the longest one.  A pad reads one of the FA_PAD_SLOTS zero slots that follow the
// chunk (index chunk + j, one per shared-memory bank), and the entries of one step (lane l's
// k-th entry for l = 0..31) are chosen so that the lanes' real entries fall into distinct
// banks: a run's sum is order-free, so at each step every lane picks any remaining token of
// its current run, by a maximum bipartite matching of lanes to banks; a lane left without a
// bank takes a pad if it has room (the rounding of its run to whole groups, or a spare group
// of the lanes shorter than the longest), and only a lane with no room reads a conflicting
// bank.  All the step's pads share one zero slot in a bank no real entry uses.  The result
// is one shared-memory wavefront per warp gather in almost every step.
// out[l] receives lane l's entries; returns the number of groups per lane.
size_t schedule_unit_chunk(int CH, const std::vector<std::vector<std::vector<uint16_t>>> &lr,
                           std::vector<std::vector<uint16_t>> &out) {
    const int G = FA_GROUP_ENTRIES;
    int64_t gmax = 0;
    int64_t glane[32];
    for (int l = 0; l < 32; ++l) {
        glane[l] = 0;
        for (const auto &r : lr[l]) glane[l] += std::max<int64_t>(1, ((int64_t)r.size() + G - 1) / G);
        gmax = std::max(gmax, glane[l]);
    }
    struct Lane {
        size_t q = 0;          // current run
        int64_t u = 0, cap = 0, spare = 0;  // entries placed in the run, its room, spare entries
        std::vector<uint16_t> bank[32];
        int cnt[32] = {0}, left = 0;
        uint32_t mask = 0;
    };
    std::vector<Lane> st(32);
    auto open_run = [&](int l) {
        Lane &s = st[l];
        s.u = 0;
        for (int b = 0; b < 32; ++b) { s.bank[b].clear(); s.cnt[b] = 0; }
        s.mask = 0;
        s.left = 0;
        if (s.q >= lr[l].size()) { s.cap = 0; return; }
        const auto &r = lr[l][s.q];
        s.cap = G * std::max<int64_t>(1, ((int64_t)r.size() + G - 1) / G);
        for (uint16_t t : r) { s.bank[t & 31].push_back(t); s.cnt[t & 31]++; s.mask |= 1u << (t & 31); }
        s.left = (int)r.size();
    };
    for (int l = 0; l < 32; ++l) {
        out[l].clear();
        out[l].reserve((size_t)(gmax * G));
        st[l].spare = G * (gmax - glane[l]);
        open_run(l);
    }
    const int64_t steps = gmax * G;
    int match[32];                 // bank -> lane
    int order[32];
    for (int64_t step = 0; step < steps; ++step) {
        for (int b = 0; b < 32; ++b) match[b] = -1;
        // lanes with real entries left, those without room for a pad first, then by room
        int n = 0;
        for (int l = 0; l < 32; ++l)
            if (st[l].q < lr[l].size() && st[l].left > 0) order[n++] = l;
        auto room = [&](int l) { return (st[l].cap - st[l].u - st[l].left) + st[l].spare; };
        std::sort(order, order + n, [&](int x, int y) {
            const int64_t rx = room(x), ry = room(y);
            return rx != ry ? rx < ry : st[x].left > st[y].left;
        });
        uint32_t seen = 0;
        // a lane tries its banks with the most tokens first (fewer forced choices later)
        int bank_order[32][32], n_banks[32];
        for (int i = 0; i < n; ++i) {
            const int l = order[i];
            int c = 0;
            for (uint32_t m = st[l].mask; m; m &= m - 1) bank_order[l][c++] = __builtin_ctz(m);
            std::sort(bank_order[l], bank_order[l] + c, [&](int x, int y) { return st[l].cnt[x] > st[l].cnt[y]; });
            n_banks[l] = c;
        }
        std::function<bool(int)> augment = [&](int l) -> bool {
            for (int j = 0; j < n_banks[l]; ++j) {
                const int b = bank_order[l][j];
                if (seen & (1u << b)) continue;
                seen |= 1u << b;
                if (match[b] < 0 || augment(match[b])) { match[b] = l; return true; }
            }
            return false;
        };
        int lane_bank[32];
        for (int l = 0; l < 32; ++l) lane_bank[l] = -1;
        for (int i = 0; i < n; ++i) { seen = 0; augment(order[i]); }
        for (int b = 0; b < 32; ++b)
            if (match[b] >= 0) lane_bank[match[b]] = b;
        // banks used by real entries this step (addresses per bank for the forced conflicts)
        int used[32] = {0};
        for (int b = 0; b < 32; ++b) used[b] = match[b] >= 0;
        uint16_t pick[32];
        bool is_pad[32];
        for (int l = 0; l < 32; ++l) {
            Lane &s = st[l];
            is_pad[l] = false;
            if (s.q >= lr[l].size() || s.left == 0) { is_pad[l] = true; continue; }
            int b = lane_bank[l];
            if (b < 0) {
                if (s.cap - s.u > s.left) { is_pad[l] = true; continue; }          // rounding room
                if (s.spare >= G) { s.cap += G; s.spare -= G; is_pad[l] = true; continue; }  // a spare group
                // no room: the least used of its banks (a conflict)
                int best = -1;
                for (uint32_t m = s.mask; m; m &= m - 1) {
                    const int c = __builtin_ctz(m);
                    if (best < 0 || used[c] < used[best]) best = c;
                }
                b = best;
                used[b]++;
            }
            pick[l] = s.bank[b].back();
            s.bank[b].pop_back();
            if (--s.cnt[b] == 0) s.mask &= ~(1u << b);
            s.left--;
        }
        int pad_bank = 0;
        for (int b = 1; b < 32; ++b)
            if (used[(CH + b) & 31] < used[(CH + pad_bank) & 31]) pad_bank = b;
        for (int l = 0; l < 32; ++l) {
            Lane &s = st[l];
            uint16_t e = is_pad[l] ? (uint16_t)(CH + pad_bank) : pick[l];
            if (s.q < lr[l].size()) {
                s.u++;
                if (s.u == s.cap) {          // the run's last entry
                    e = (uint16_t)(e | FA_RUN_END);
                    s.q++;
                    open_run(l);
                }
            }
            out[l].push_back(e);
        }
    }
    return (size_t)gmax;
}

// Token-major incidence streams of the all-token marginals: the (src, dst) pair of every
// token-edge incidence (|S| <= 4096 fits 16 bits), the tokens ordered by incidence count
// (ties by id) and interleaved by groups of 32, each group as many rows as its longest
// token (tokens of nearly equal counts share a group, so the padding stays near one row per
// incidence however skewed the counts are), padding (S, S).  A token's incidences may come
// in any order, so each row is filled greedily to keep the 32 lanes' gathers of alpha(src)
// (shared-memory word src) and of beta(dst) (word S + 1 + dst) in distinct banks, or on a
// shared address: a lane takes the first of its next incidences (a window of 48) that adds
// no conflict, else the one adding fewest.
void build_token_streams(int S, int V, const std::vector<int64_t> &tok_off, const std::vector<int32_t> &tok_edges,
                         const int32_t *edge_src, const int32_t *edge_dst, std::vector<int32_t> &tok_perm,
                         std::vector<int64_t> &tok_goff, std::vector<uint32_t> &tok_sd) {
    const int64_t n_tg = ((int64_t)V + 31) / 32;
    tok_perm.resize(V);
    std::iota(tok_perm.begin(), tok_perm.end(), 0);
    std::stable_sort(tok_perm.begin(), tok_perm.end(), [&](int32_t x, int32_t y) {
        return tok_off[x + 1] - tok_off[x] < tok_off[y + 1] - tok_off[y];
    });
    tok_goff.assign(n_tg + 1, 0);
    for (int64_t g = 0; g < n_tg; ++g) {
        int64_t cnt = 0;
        for (int64_t i = 32 * g; i < std::min<int64_t>(32 * g + 32, V); ++i)
            cnt = std::max(cnt, tok_off[tok_perm[i] + 1] - tok_off[tok_perm[i]]);
        tok_goff[g + 1] = tok_goff[g] + cnt;
    }
    const uint32_t pad = ((uint32_t)S << 16) | (uint32_t)S;
    tok_sd.assign((size_t)tok_goff[n_tg] * 32, pad);
    const int kWin = 48;
    std::vector<uint32_t> rem[32];
    for (int64_t g = 0; g < n_tg; ++g) {
        for (int l = 0; l < 32; ++l) {
            rem[l].clear();
            const int64_t i = 32 * g + l;
            if (i >= V) continue;
            const int v = tok_perm[i];
            for (int64_t k = tok_off[v]; k < tok_off[v + 1]; ++k) {
                const int e = tok_edges[k];
                rem[l].push_back(((uint32_t)edge_src[e] << 16) | (uint32_t)edge_dst[e]);
            }
        }
        for (int64_t row = tok_goff[g]; row < tok_goff[g + 1]; ++row) {
            int a_addr[32], b_addr[32];   // the address a bank holds (-1: free, -2: several)
            for (int q = 0; q < 32; ++q) a_addr[q] = b_addr[q] = -1;
            auto cost = [&](uint32_t sd) {
                const int a = (int)(sd >> 16), bw = S + 1 + (int)(sd & 0xffffu);
                const int qa = a & 31, qb = bw & 31;
                return (int)(a_addr[qa] != -1 && a_addr[qa] != a) + (int)(b_addr[qb] != -1 && b_addr[qb] != bw);
            };
            bool padded = false;   // the lanes past their token's count read the padding
            for (int l = 0; l < 32; ++l) padded |= rem[l].empty();
            if (padded) { a_addr[S & 31] = S; b_addr[(2 * S + 1) & 31] = 2 * S + 1; }
            for (int l = 0; l < 32; ++l) {
                if (rem[l].empty()) continue;
                const int n = (int)std::min<size_t>(rem[l].size(), kWin);
                int best = 0, bc = 3;
                for (int x = 0; x < n && bc > 0; ++x) {
                    const int c = cost(rem[l][rem[l].size() - 1 - x]);
                    if (c < bc) { bc = c; best = x; }
                }
                const size_t at = rem[l].size() - 1 - best;
                const uint32_t sd = rem[l][at];
                rem[l][at] = rem[l].back();
                rem[l].pop_back();
                const int a = (int)(sd >> 16), bw = S + 1 + (int)(sd & 0xffffu);
                a_addr[a & 31] = a_addr[a & 31] == -1 || a_addr[a & 31] == a ? a : -2;
                b_addr[bw & 31] = b_addr[bw & 31] == -1 || b_addr[bw & 31] == bw ? bw : -2;
                tok_sd[(size_t)row * 32 + l] = sd;
            }
        }
    }
}

std::string build_run_layout(int S, int V, int n_cells, const std::vector<int32_t> &row_cell_off,
                             const std::vector<int64_t> &cell_off, const std::vector<int32_t> &cell_tok,
                             RunLayout &out) {
    // Reweight layout (runs).  The vocabulary is read in chunks of CH tokens staged in shared
    // memory.  Rows are taken in groups: a row with many tokens or cells gets one or more
    // warp units of its own, consecutive small rows share one unit.  Within a group every
    // cell's sorted tokens are cut into runs of about the group's tokens / (2 x its lanes),
    // and the runs are dealt longest first, each to the least-loaded lane that still has a
    // free slot.  A lane's stream for one chunk is its runs' in-chunk tokens, run after run,
    // each run padded to whole groups of FA_GROUP_ENTRIES (a run with no token in the chunk
    // is one group of pads), the last entry of each run flagged, the 32 lanes padded to a
    // common number of groups.
    const int CH = (V <= FA_REWEIGHT_MAX_CHUNK) ? V : FA_REWEIGHT_MAX_CHUNK;
    const int nch = (V + CH - 1) / CH;
    out.chunk_tokens = CH;
    out.n_chunks = nch;
    const int64_t kUnitTokens = 8192;        // tokens per warp unit (over all chunks)
    const int kSmallCells = 128, kUnitCells = 256;  // at most 8 runs per lane on average
    struct Group { int32_t r0, r1, u0, nu, c0, c1; };
    std::vector<Group> groups;
    std::vector<int32_t> &row_unit0 = out.row_unit0;
    row_unit0.assign(S, 0);
    auto row_tokens = [&](int r) { return cell_off[row_cell_off[r + 1]] - cell_off[row_cell_off[r]]; };
    auto row_is_big = [&](int r) {
        return row_tokens(r) * 2 >= kUnitTokens || row_cell_off[r + 1] - row_cell_off[r] > kSmallCells;
    };
    int32_t n_units = 0;
    for (int r = 0; r < S;) {
        Group g{};
        g.r0 = r;
        g.u0 = n_units;
        if (row_is_big(r)) {
            const int64_t rt = row_tokens(r), rc = row_cell_off[r + 1] - row_cell_off[r];
            int64_t nu = std::max<int64_t>((rt + kUnitTokens - 1) / kUnitTokens, (rc + kUnitCells - 1) / kUnitCells);
            g.nu = (int32_t)std::min<int64_t>(std::max<int64_t>(nu, 1), FA_RW_MAX_UNITS);
            g.r1 = r + 1;
        } else {
            int64_t tok = 0;
            int cells = 0, r1 = r;
            while (r1 < S && !row_is_big(r1)) {
                const int64_t t2 = row_tokens(r1);
                const int c2 = row_cell_off[r1 + 1] - row_cell_off[r1];
                if (r1 > r && (tok + t2 > kUnitTokens || cells + c2 > kUnitCells)) break;
                tok += t2;
                cells += c2;
                ++r1;
            }
            g.nu = 1;
            g.r1 = r1;
        }
        r = g.r1;
        g.c0 = row_cell_off[g.r0];
        g.c1 = row_cell_off[g.r1];
        for (int q = g.r0; q < g.r1; ++q) row_unit0[q] = g.u0;
        n_units += g.nu;
        groups.push_back(g);
    }
    out.n_units = n_units;

    std::vector<int32_t> &crun_off = out.crun_off, &ru_goff = out.ru_goff;
    std::vector<uint16_t> &crun_slot = out.crun_slot, &ru_tok = out.ru_tok;
    crun_off.assign(n_cells + 1, 0);
    std::vector<std::vector<uint16_t>> cell_slots(n_cells);
    struct Run { int32_t cell; int64_t q, nr; };  // tokens cell_tok[cell_off[cell] + q + nr i]
    for (const Group &g : groups) {
        const int lanes = 32 * g.nu;
        const int64_t gt = cell_off[g.c1] - cell_off[g.c0];
        const int64_t T = std::max<int64_t>(8, (gt + 2 * lanes - 1) / (2 * lanes));
        // run q of a cell of nr runs takes the cell's tokens q, q + nr, q + 2 nr, ... (so every
        // run follows the cell's spread over the chunks); per-chunk token counts of each run
        std::vector<Run> runs;
        std::vector<int32_t> rch;  // [run][chunk]
        for (int c = g.c0; c < g.c1; ++c) {
            const int64_t len = cell_off[c + 1] - cell_off[c];
            const int64_t nr = std::max<int64_t>(1, (len + T - 1) / T);
            for (int64_t q = 0; q < nr; ++q) {
                runs.push_back({c, q, nr});
                for (int ch = 0; ch < nch; ++ch) rch.push_back(0);
                int32_t *rc = rch.data() + (runs.size() - 1) * nch;
                for (int64_t x = cell_off[c] + q; x < cell_off[c + 1]; x += nr) rc[cell_tok[x] / CH]++;
                // a run's entries in a chunk are padded to whole groups; an empty run still
                // ends once, with a group of pads
                for (int ch = 0; ch < nch; ++ch)
                    rc[ch] = std::max(FA_GROUP_ENTRIES, (rc[ch] + FA_GROUP_ENTRIES - 1) / FA_GROUP_ENTRIES * FA_GROUP_ENTRIES);
            }
        }
        std::vector<int64_t> rsize(runs.size(), 0);
        for (size_t ri = 0; ri < runs.size(); ++ri)
            for (int ch = 0; ch < nch; ++ch) rsize[ri] += rch[ri * nch + ch];
        std::vector<int32_t> order(runs.size());
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return rsize[x] > rsize[y]; });
        // deal longest first to the lane where the run raises its unit's per-chunk maxima (the
        // padded stream lengths) least, then to the least-loaded such lane
        std::vector<int64_t> load(lanes, 0), lch((size_t)lanes * nch, 0), umax((size_t)g.nu * nch, 0);
        std::vector<std::vector<int32_t>> lane_runs(lanes);
        std::vector<int32_t> slot_of(runs.size(), 0);
        for (int32_t ri : order) {
            const int32_t *rc = rch.data() + (size_t)ri * nch;
            int best = -1;
            int64_t best_inc = 0;
            for (int l = 0; l < lanes; ++l) {
                if ((int)lane_runs[l].size() >= FA_RUN_SLOTS) continue;
                int64_t inc = 0;
                const int64_t *ll = lch.data() + (size_t)l * nch, *um = umax.data() + (size_t)(l >> 5) * nch;
                for (int ch = 0; ch < nch; ++ch) inc += std::max<int64_t>(0, ll[ch] + rc[ch] - um[ch]);
                if (best < 0 || inc < best_inc || (inc == best_inc && load[l] < load[best])) { best = l; best_inc = inc; }
            }
            if (best < 0) return "reweight layout overflow";
            slot_of[ri] = (best >> 5) * FA_UNIT_SLOTS + (int32_t)lane_runs[best].size() * 32 + (best & 31);
            lane_runs[best].push_back(ri);
            load[best] += rsize[ri];
            int64_t *ll = lch.data() + (size_t)best * nch, *um = umax.data() + (size_t)(best >> 5) * nch;
            for (int ch = 0; ch < nch; ++ch) { ll[ch] += rc[ch]; um[ch] = std::max(um[ch], ll[ch]); }
        }
        for (size_t ri = 0; ri < runs.size(); ++ri) cell_slots[runs[ri].cell].push_back((uint16_t)slot_of[ri]);
        for (int w = 0; w < g.nu; ++w) {
            for (int ch = 0; ch < nch; ++ch) {
                const int32_t lo = ch * CH, hi = (int32_t)std::min<int64_t>((int64_t)(ch + 1) * CH, V);
                // every lane's runs as lists of in-chunk indices
                std::vector<std::vector<std::vector<uint16_t>>> lr(32);
                for (int l = 0; l < 32; ++l) {
                    for (int32_t ri : lane_runs[w * 32 + l]) {
                        const Run &rn = runs[ri];
                        std::vector<uint16_t> e;
                        for (int64_t x = cell_off[rn.cell] + rn.q; x < cell_off[rn.cell + 1]; x += rn.nr)
                            if (cell_tok[x] >= lo && cell_tok[x] < hi) e.push_back((uint16_t)(cell_tok[x] - lo));
                        lr[l].push_back(std::move(e));
                    }
                }
                std::vector<std::vector<uint16_t>> out(32);
                const int G = FA_GROUP_ENTRIES;
                const size_t len = schedule_unit_chunk(CH, lr, out);
                const size_t g0 = ru_tok.size() / G;
                ru_goff.push_back((int32_t)g0);
                ru_tok.resize(ru_tok.size() + len * 32 * G, (uint16_t)CH);
                // the scheduler flags a run's last entry; the stored group carries the flag on
                // its first entry instead (no other entry has bit 15 set)
                for (int l = 0; l < 32; ++l)
                    for (size_t k = 0; k < out[l].size(); k += G) {
                        const uint16_t end = out[l][k + G - 1] & FA_RUN_END;
                        for (int h = 0; h < G; ++h) {
                            uint16_t e = (uint16_t)(out[l][k + h] & ~FA_RUN_END);
                            if (e >= CH + FA_PAD_SLOTS) return "reweight layout: entry out of range";
                            if (h == 0) e = (uint16_t)(e | end);
                            ru_tok[(g0 + (k / G) * 32 + l) * G + h] = e;
                        }
                    }
                if (ru_tok.size() / G > (size_t)INT32_MAX / 2) return "automaton too large";
            }
        }
    }
    ru_goff.push_back((int32_t)(ru_tok.size() / FA_GROUP_ENTRIES));
    // the reweight reads up to eight groups per lane past a stream's end
    ru_tok.resize(ru_tok.size() + 8 * 32 * FA_GROUP_ENTRIES, (uint16_t)CH);
    for (int c = 0; c < n_cells; ++c) {
        crun_off[c] = (int32_t)crun_slot.size();
        crun_slot.insert(crun_slot.end(), cell_slots[c].begin(), cell_slots[c].end());
    }
    crun_off[n_cells] = (int32_t)crun_slot.size();

    // reweight blocks: whole row groups, at most caps[p] units per block in partition p
    std::vector<int32_t> &rbm = out.rbm;
    std::vector<int> caps{FA_RW_MAX_UNITS};
    for (int c = 32; c >= 1; c >>= 1)
        if (c < caps.back()) caps.push_back(c);
    for (int p = 0;; ++p) {
        const int cap = caps[p];
        out.part_first.push_back((int32_t)(rbm.size() / 8));
        int count = 0, maxu = 1, maxr = 1;
        int64_t maxt = 0;
        for (size_t gi = 0; gi < groups.size();) {
            size_t gj = gi;
            int nu = 0;
            while (gj < groups.size() && (gj == gi || nu + groups[gj].nu <= cap)) nu += groups[gj++].nu;
            const Group &A = groups[gi], &Z = groups[gj - 1];
            rbm.insert(rbm.end(), {A.r0, Z.r1, A.u0, Z.u0 + Z.nu, A.c0, Z.c1, 0, 0});
            maxu = std::max(maxu, nu);
            maxr = std::max(maxr, Z.r1 - A.r0);
            maxt = std::max<int64_t>(maxt, (int64_t)nu * FA_UNIT_SLOTS + (int64_t)(Z.r1 - A.r0) * S);
            ++count;
            gi = gj;
        }
        out.part_count.push_back(count);
        out.part_max_units.push_back(maxu);
        out.part_max_rows.push_back(maxr);
        out.part_tile_floats.push_back(maxt);
        if (p + 1 == (int)caps.size() || count == (int)groups.size()) break;
    }
    return std::string();
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
    }
    for (int s = 0; s < S; ++s) row_cell_off[s + 1] += row_cell_off[s];
    a->n_cells = (int32_t)cell_dst.size();
    a->max_cell_len = max_cell_len;

    RunLayout rl;
    {
        const std::string why = build_run_layout(S, V, a->n_cells, row_cell_off, cell_off, cell_tok, rl);
        if (!why.empty()) {
            delete a;
            fa_set_error("fa_compile: " + why);
            return why == "automaton too large" ? FA_ERR_INVALID_ARG : FA_ERR_UNSUPPORTED;
        }
    }
    a->chunk_tokens = rl.chunk_tokens;
    a->n_chunks = rl.n_chunks;
    a->n_units = rl.n_units;
    a->part_first = rl.part_first;
    a->part_count = rl.part_count;
    a->part_max_units = rl.part_max_units;
    a->part_max_rows = rl.part_max_rows;
    a->part_tile_floats = rl.part_tile_floats;

    std::vector<int2> cell_rec(a->n_cells);
    for (int c = 0; c < a->n_cells; ++c) {
        const int s = cell_src[c];
        cell_rec[c].x = s * S + cell_dst[c];
        cell_rec[c].y = rl.crun_off[c + 1] - rl.crun_off[c] == 1
                            ? rl.row_unit0[s] * FA_UNIT_SLOTS + (int32_t)rl.crun_slot[rl.crun_off[c]]
                            : -1;
    }

    std::vector<int32_t> esrc(edge_src, edge_src + E), edst(edge_dst, edge_dst + E);
    std::vector<int32_t> tok_perm;
    std::vector<int64_t> tok_goff;
    std::vector<uint32_t> tok_sd;
    build_token_streams(S, V, tok_off, tok_edges, edge_src, edge_dst, tok_perm, tok_goff, tok_sd);

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
    bb.add(&a->tok_sd, tok_sd);
    bb.add(&a->tok_goff, tok_goff);
    bb.add(&a->tok_perm, tok_perm);
    bb.add(&a->row_cell_off, row_cell_off);
    bb.add(&a->cell_dst, cell_dst);
    bb.add(&a->cell_src, cell_src);
    bb.add(&a->cell_off, cell_off);
    bb.add(&a->cell_tok, cell_tok);
    bb.add(&a->rb_meta, rl.rbm);
    bb.add(&a->ru_tok, rl.ru_tok);
    bb.add(&a->ru_goff, rl.ru_goff);
    bb.add(&a->row_unit0, rl.row_unit0);
    bb.add(&a->crun_off, rl.crun_off);
    bb.add(&a->crun_slot, rl.crun_slot);
    bb.add(&a->cell_rec, cell_rec);

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
