// Host-only check of the reweight's run layout (build_run_layout in csrc/fa_compile.cu):
// builds the layout of an automaton read from a file, replays the reweight kernel's walk
// over the entry streams on the CPU (run sums per chunk, run ends, slot folding, per-cell
// combination) for random probabilities, and compares every cell with a float64 sum of
// its tokens.  It also checks the layout's invariants: every row and cell covered once per
// partition, run-end flags only on a group's first entry, no lane above FA_RUN_SLOTS runs,
// indices inside their chunk or its zero pad slots.  Prints one line "bad=N ..." and exits non-zero when N > 0.
#include "../constrained_decoding_diffusion_gb300/csrc/fa_compile.cu"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <map>
#include <random>

int main(int argc, char **argv) {
    if (argc < 2) return 2;
    FILE *f = fopen(argv[1], "rb");
    if (!f) return 2;
    int64_t hdr[3];
    if (fread(hdr, 8, 3, f) != 3) return 2;
    const int S = (int)hdr[0], V = (int)hdr[1], E = (int)hdr[2];
    std::vector<int32_t> es(E), ed(E);
    std::vector<int64_t> lo(E + 1);
    if (fread(es.data(), 4, E, f) != (size_t)E || fread(ed.data(), 4, E, f) != (size_t)E ||
        fread(lo.data(), 8, E + 1, f) != (size_t)E + 1)
        return 2;
    std::vector<int32_t> lt(lo[E]);
    if (fread(lt.data(), 4, lo[E], f) != (size_t)lo[E]) return 2;
    fclose(f);
    // cells as fa_compile forms them: distinct (src, dst), sorted multiset of tokens
    std::map<std::pair<int, int>, std::vector<int32_t>> cm;
    for (int e = 0; e < E; ++e) {
        auto &v = cm[{es[e], ed[e]}];
        v.insert(v.end(), lt.begin() + lo[e], lt.begin() + lo[e + 1]);
    }
    std::vector<int32_t> row_cell_off(S + 1, 0), cell_src, cell_tok;
    std::vector<int64_t> cell_off(1, 0);
    for (auto &kv : cm) {
        auto v = kv.second;
        std::sort(v.begin(), v.end());
        cell_src.push_back(kv.first.first);
        cell_tok.insert(cell_tok.end(), v.begin(), v.end());
        cell_off.push_back((int64_t)cell_tok.size());
        row_cell_off[kv.first.first + 1]++;
    }
    for (int s = 0; s < S; ++s) row_cell_off[s + 1] += row_cell_off[s];
    const int nc = (int)cell_src.size();
    RunLayout rl;
    const std::string why = build_run_layout(S, V, nc, row_cell_off, cell_off, cell_tok, rl);
    if (!why.empty()) { printf("bad=1 layout error: %s\n", why.c_str()); return 1; }
    const int CH = rl.chunk_tokens, nch = rl.n_chunks, G = FA_GROUP_ENTRIES;
    std::mt19937 rng(1);
    std::uniform_real_distribution<float> U(0.0f, 1.0f);
    std::vector<float> probs(V);
    for (auto &x : probs) x = U(rng);
    std::vector<double> exact(nc);
    for (int c = 0; c < nc; ++c) {
        double t = 0;
        for (int64_t q = cell_off[c]; q < cell_off[c + 1]; ++q) t += probs[cell_tok[q]];
        exact[c] = t;
    }
    long bad = 0, entries = 0;
    double worst = 0;
    for (size_t p = 0; p < rl.part_count.size(); ++p) {
        std::vector<int> seen(nc, 0);
        int prev_r1 = 0;
        for (int i = 0; i < rl.part_count[p]; ++i) {
            const int32_t *m = rl.rbm.data() + 8 * (rl.part_first[p] + i);
            const int r0 = m[0], r1 = m[1], u0 = m[2], u1 = m[3], c0 = m[4], c1 = m[5], nu = u1 - u0;
            bad += r0 != prev_r1;
            prev_r1 = r1;
            bad += nu > rl.part_max_units[p] || r1 - r0 > rl.part_max_rows[p];
            bad += c0 != row_cell_off[r0] || c1 != row_cell_off[r1];
            std::vector<float> tot((size_t)nu * FA_UNIT_SLOTS, 0.0f);
            for (int ch = 0; ch < nch; ++ch) {
                const int base = ch * CH, n = std::min(CH, V - base);
                std::vector<float> sp(CH + FA_PAD_SLOTS, 0.0f);
                for (int q = 0; q < n; ++q) sp[q] = probs[base + q];
                for (int w = 0; w < nu; ++w) {
                    const size_t ui = (size_t)(u0 + w) * nch + ch;
                    const int gb = rl.ru_goff[ui], ge = rl.ru_goff[ui + 1];
                    bad += (ge - gb) % 32 != 0;
                    const int ng = (ge - gb) / 32;
                    std::vector<float> slot((size_t)FA_UNIT_SLOTS, 0.0f);
                    for (int l = 0; l < 32; ++l) {
                        float acc = 0.0f;
                        int j = 0;
                        for (int k = 0; k < ng; ++k) {
                            bool end = false;
                            for (int h = 0; h < G; ++h) {
                                const uint32_t e = rl.ru_tok[((size_t)gb + (size_t)k * 32 + l) * G + h];
                                if (e & FA_RUN_END) {
                                    if (h != 0) ++bad;                // the flag sits on a group's first entry
                                    end = true;
                                }
                                const int idx = e & 0x7fff;
                                if (idx >= CH + FA_PAD_SLOTS || (idx < CH && idx >= n)) { ++bad; continue; }
                                acc += sp[idx];
                                ++entries;
                            }
                            if (end) {                                // the group ends the lane's run
                                if (j >= FA_RUN_SLOTS) { ++bad; continue; }
                                slot[(size_t)j * 32 + l] = acc;       // the chunk's run sum
                                acc = 0.0f;
                                ++j;
                            }
                        }
                    }
                    for (size_t q = 0; q < slot.size(); ++q) tot[(size_t)w * FA_UNIT_SLOTS + q] += slot[q];
                }
            }
            for (int c = c0; c < c1; ++c) {
                const int s = cell_src[c];
                const long sb = (long)(rl.row_unit0[s] - u0) * FA_UNIT_SLOTS;
                if (sb < 0) { ++bad; continue; }
                double v = 0;
                for (int q = rl.crun_off[c]; q < rl.crun_off[c + 1]; ++q) {
                    const long si = sb + rl.crun_slot[q];
                    if (si >= (long)tot.size()) { ++bad; continue; }
                    v += tot[si];
                }
                const double err = std::fabs(v - exact[c]) / std::max(1e-30, exact[c]);
                worst = std::max(worst, err);
                if (err > 1e-5) ++bad;
                seen[c]++;
            }
        }
        bad += prev_r1 != S;
        for (int c = 0; c < nc; ++c) bad += seen[c] != 1;
    }
    // shared-memory wavefronts per warp gather: distinct addresses in the busiest bank, over
    // every step of every unit's stream (the zero pad slots count as addresses too)
    long steps = 0, waves = 0;
    for (int u = 0; u < rl.n_units; ++u)
        for (int ch = 0; ch < nch; ++ch) {
            const size_t ui = (size_t)u * nch + ch;
            const int gb = rl.ru_goff[ui], ng = (rl.ru_goff[ui + 1] - gb) / 32;
            for (int k = 0; k < ng; ++k)
                for (int h = 0; h < G; ++h) {
                    std::map<int, std::vector<int>> bank;
                    int w = 1;
                    for (int l = 0; l < 32; ++l) {
                        const int idx = rl.ru_tok[((size_t)gb + (size_t)k * 32 + l) * G + h] & 0x7fff;
                        auto &v = bank[idx & 31];
                        if (std::find(v.begin(), v.end(), idx) == v.end()) v.push_back(idx);
                        w = std::max(w, (int)v.size());
                    }
                    ++steps;
                    waves += w;
                }
        }
    printf("wavefronts_per_gather=%.3f ", steps ? (double)waves / steps : 1.0);
    // token-major streams of the all-token marginals (build_token_streams): every token's
    // incidences exactly once, padding (S, S) past its count, and the alpha / beta gathers'
    // wavefronts after the bank ordering
    {
        std::vector<int64_t> tok_off(V + 1, 0);
        for (int e = 0; e < E; ++e) for (int64_t q = lo[e]; q < lo[e + 1]; ++q) tok_off[lt[q] + 1]++;
        for (int v = 0; v < V; ++v) tok_off[v + 1] += tok_off[v];
        std::vector<int32_t> tok_edges(tok_off[V]);
        std::vector<int64_t> fill(tok_off.begin(), tok_off.end() - 1);
        for (int e = 0; e < E; ++e) for (int64_t q = lo[e]; q < lo[e + 1]; ++q) tok_edges[fill[lt[q]]++] = e;
        std::vector<int32_t> perm;
        std::vector<int64_t> goff;
        std::vector<uint32_t> sd;
        build_token_streams(S, V, tok_off, tok_edges, es.data(), ed.data(), perm, goff, sd);
        const uint32_t pad = ((uint32_t)S << 16) | (uint32_t)S;
        long wa = 0, wb = 0, rows = 0;
        for (int64_t g = 0; g * 32 < V; ++g) {
            for (int l = 0; l < 32 && g * 32 + l < V; ++l) {
                const int v = perm[g * 32 + l];
                std::vector<uint32_t> want, got;
                for (int64_t q = tok_off[v]; q < tok_off[v + 1]; ++q)
                    want.push_back(((uint32_t)es[tok_edges[q]] << 16) | (uint32_t)ed[tok_edges[q]]);
                for (int64_t r = goff[g]; r < goff[g + 1]; ++r) {
                    const uint32_t x = sd[(size_t)r * 32 + l];
                    if (r - goff[g] < (int64_t)want.size()) got.push_back(x);
                    else bad += x != pad;
                }
                std::sort(want.begin(), want.end());
                std::sort(got.begin(), got.end());
                bad += want != got;
            }
            for (int64_t r = goff[g]; r < goff[g + 1]; ++r) {
                for (int which = 0; which < 2; ++which) {
                    std::map<int, std::vector<int>> bank;
                    int w = 1;
                    for (int l = 0; l < 32; ++l) {
                        const uint32_t x = sd[(size_t)r * 32 + l];
                        const int a = which == 0 ? (int)(x >> 16) : S + 1 + (int)(x & 0xffffu);
                        auto &vv = bank[a & 31];
                        if (std::find(vv.begin(), vv.end(), a) == vv.end()) vv.push_back(a);
                        w = std::max(w, (int)vv.size());
                    }
                    (which == 0 ? wa : wb) += w;
                }
                ++rows;
            }
        }
        printf("token_rows_wavefronts=%.3f/%.3f ", rows ? (double)wa / rows : 1.0, rows ? (double)wb / rows : 1.0);
    }
    printf("bad=%ld S=%d V=%d cells=%d incidences=%zu units=%d chunks=%d partitions=%zu entries_per_incidence=%.3f "
           "worst_rel=%.2e\n",
           bad, S, V, nc, cell_tok.size(), rl.n_units, nch, rl.part_count.size(),
           (double)entries / (double)rl.part_count.size() / std::max<size_t>(1, cell_tok.size()), worst);
    return bad ? 1 : 0;
}
