// The constrained denoising step on one GPU: emission reweighting, the span-matrix up-sweep,
// top-down midpoint sampling, prefix/suffix messages, leaf tokens and marginals, and the
// top-k commit.  Method: "Constrained Decoding for Diffusion Language Models via Efficient
// Inference over Finite Automata" (paperfeed.app summary, sections "The insight" and "The
// scan trick"; papernotes.org notes, key designs 1-3).
//
// Span number format.  A span matrix A[l, r) = M_{l+1} ... M_r is stored as an fp32
// mantissa matrix Ã and one power-of-two exponent per row: A[i, j] = Ã[i, j] * 2^rho[i].
// rmax[i] holds the bit pattern of max_j Ã[i, j] (0 for an all-zero row) and rminc[i] the
// complement 0x7fffffff - bits of the smallest nonzero Ã[i, j] (0 for an all-zero row), so
// both accumulate with atomicMax from zero.  Products of
// hundreds of probabilities leave the fp32 range long before a sequence ends, and rows of one
// span differ by far more than 2^254 once committed tokens pin the path, so a single
// exponent per matrix would flush whole rows; per-row exponents keep every row at full
// relative precision.  Only entries more than ~2^-126 below their own row's maximum are lost.
#include <atomic>
#include <cfloat>
#include <cmath>
#include <string>
#include <vector>

#include "fa_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kHostChunks = FA_HOST_PIECES;  // pieces of fa_constrained_step_host's input copies
constexpr int kTmChunkMax = 4096, kTmChunkMin = 1024;  // tokens per block of the all-token marginals
constexpr int kWarps = kThreads / 32;

// ----------------------------------------------------------------------------- workspace plan

struct Plan {
    int B = 0, L = 0, S = 0, V = 0, K = 0, Lp = 1;
    int nk[18] = {0};
    size_t mant[18] = {0}, rho[18] = {0}, rmax[18] = {0}, rminc[18] = {0}, mu[18] = {0};
    size_t z = 0, am = 0, ae = 0, bm = 0, be = 0, keys = 0, conf = 0, den_m = 0, den_e = 0, tm_part = 0, zsum = 0, zexp = 0;
    int tm_chunks = 1, tm_chunk = kTmChunkMax;
    size_t rmax_hi = 0, rmax_hi_bytes = 0, leaf_done = 0, tc_err = 0, range_lost = 0, img = 0;
    // functional spans (a DFA on the tensor-core path): per tree level, one flag per node and,
    // for flagged nodes, the partial function s -> the one state its row reaches (-1: none)
    bool functional = false;
    size_t fflag[18] = {0}, fmap[18] = {0};
    size_t total = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Plan make_plan(const fa_automaton *a, int B, int L) {
    Plan p;
    p.B = B; p.L = L; p.S = a->S; p.V = a->V;
    p.Lp = 1; p.K = 0;
    while (p.Lp < L) { p.Lp <<= 1; p.K++; }
    size_t off = 0;
    const size_t S = (size_t)a->S;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + (bytes ? bytes : 1)); return o; };
    for (int k = 0; k <= p.K; ++k) {
        p.nk[k] = (L + (1 << k) - 1) >> k;
        size_t nodes = (size_t)B * (size_t)p.nk[k];
        p.mant[k] = take(nodes * S * S * sizeof(float));
        p.rho[k] = take(nodes * S * sizeof(int32_t));
        p.mu[k] = take(k ? nodes * S * sizeof(int32_t) : 0);
    }
    // row maxima and complemented row minima: level 0 (written whole by the reweight), then
    // levels 1..K back to back with the step's counters and flags (cleared together by the
    // reweight; the products accumulate into them with atomicMax)
    p.rmax[0] = take((size_t)B * p.nk[0] * S * sizeof(int32_t));
    p.rminc[0] = take((size_t)B * p.nk[0] * S * sizeof(int32_t));
    p.rmax_hi = off;
    {
        size_t o = p.rmax_hi;
        for (int k = 1; k <= p.K; ++k) { p.rmax[k] = o; o += (size_t)B * p.nk[k] * S * sizeof(int32_t); }
        for (int k = 1; k <= p.K; ++k) { p.rminc[k] = o; o += (size_t)B * p.nk[k] * S * sizeof(int32_t); }
        p.tc_err = o;                          // timeout word of the tensor-core span products
        p.leaf_done = p.tc_err + sizeof(int32_t);  // per-sequence ticket counters of the leaf blocks
        // per-sequence range-loss flags: set when a span product may push nonzero mass below
        // the fp32 normal range
        p.range_lost = p.leaf_done + (size_t)B * sizeof(int32_t);
        p.rmax_hi_bytes = (p.range_lost - p.rmax_hi) + (size_t)B * sizeof(int32_t);
        off = align256(p.rmax_hi + p.rmax_hi_bytes);
    }
    size_t bnd = (size_t)B * (size_t)(L + 1);
    p.z = take(bnd * sizeof(int32_t));
    p.am = take(bnd * S * sizeof(float));
    p.ae = take(bnd * S * sizeof(int32_t));
    p.bm = take(bnd * S * sizeof(float));
    p.be = take(bnd * S * sizeof(int32_t));
    p.keys = take((size_t)B * (size_t)L * sizeof(unsigned long long));
    p.conf = take((size_t)B * (size_t)L * sizeof(float));   // remasking confidence the commit ranks by
    // the local normaliser D_t of every position (mantissa, exponent), from the leaves
    p.den_m = take((size_t)B * (size_t)L * sizeof(float));
    p.den_e = take((size_t)B * (size_t)L * sizeof(int32_t));
    // per (position, vocabulary chunk) partial sums of p ln p for the entropies
    // (4096 tokens per block, halved down to 1024 while that gives under 4096 blocks in all:
    //  few positions need the narrower blocks to fill the GPU)
    p.tm_chunk = kTmChunkMax;
    while (p.tm_chunk > kTmChunkMin && (long)B * L * ((a->V + p.tm_chunk - 1) / p.tm_chunk) < 4096) p.tm_chunk >>= 1;
    p.tm_chunks = (a->V + p.tm_chunk - 1) / p.tm_chunk;
    p.tm_part = take((size_t)B * (size_t)L * (size_t)p.tm_chunks * sizeof(double));
    // tensor-core operand images, sized for the level with the most node slots (level 1)
    if (fa_span_tc_supported(a->S) && p.K >= 1) p.img = take(fa_span_tc_image_bytes(a->S, (long)B * p.nk[1]));
    p.zsum = take((size_t)B * sizeof(float));
    p.zexp = take((size_t)B * sizeof(int32_t));
    p.functional = a->is_dfa && fa_span_tc_supported(a->S) && p.K >= 1;
    if (p.functional)
        for (int k = 0; k <= p.K; ++k) {
            const size_t nodes = (size_t)B * (size_t)p.nk[k];
            p.fflag[k] = take(nodes * sizeof(int32_t));
            p.fmap[k] = take(nodes * S * sizeof(int32_t));
        }
    p.total = off;
    return p;
}

// Device view of the compiled automaton.
struct DevFA {
    int S, V, start, n_accept;
    const int32_t *accept, *accept_mask, *edge_src, *edge_dst;
    const uint32_t *tok_sd;
    const int64_t *tok_goff;
    const int32_t *tok_perm;
    const int64_t *tok_off;
    const int32_t *tok_edges;
    const int32_t *row_cell_off, *cell_dst, *cell_src;
    const int64_t *cell_off;
    const int32_t *cell_tok;
    const uint16_t *ru_tok, *crun_slot;
    const int2 *cell_rec;
    const int32_t *ru_goff, *row_unit0, *crun_off;
    int chunk_tokens, n_chunks, n_cells;
};

DevFA dev_view(const fa_automaton *a) {
    DevFA d;
    d.S = a->S; d.V = a->V; d.start = a->start; d.n_accept = a->n_accept;
    d.accept = a->accept; d.accept_mask = a->accept_mask; d.edge_src = a->edge_src; d.edge_dst = a->edge_dst;
    d.tok_sd = a->tok_sd;
    d.tok_goff = a->tok_goff;
    d.tok_perm = a->tok_perm;
    d.tok_off = a->tok_off; d.tok_edges = a->tok_edges;
    d.row_cell_off = a->row_cell_off; d.cell_dst = a->cell_dst; d.cell_src = a->cell_src;
    d.cell_off = a->cell_off; d.cell_tok = a->cell_tok;
    d.ru_tok = a->ru_tok; d.crun_slot = a->crun_slot; d.ru_goff = a->ru_goff;
    d.row_unit0 = a->row_unit0; d.crun_off = a->crun_off;
    d.cell_rec = a->cell_rec;
    d.chunk_tokens = a->chunk_tokens; d.n_chunks = a->n_chunks; d.n_cells = a->n_cells;
    return d;
}

// ----------------------------------------------------------------------------- block helpers

// Inverse-CDF draw over n weights given by w(i) >= 0: the first i whose running sum exceeds
// u * total (total from the same loop order), clamped to the last positive weight.  Returns
// -1 when every weight is zero.  Executed by one full warp; all lanes get the result.
template <class WF>
__device__ int warp_categorical(int n, float u, WF w) {
    const int lane = threadIdx.x & 31;
    float total = 0.0f;
    for (int base = 0; base < n; base += 32) {
        int i = base + lane;
        float x = (i < n) ? w(i) : 0.0f;
        total += fa_warp_sum(x);
    }
    if (!(total > 0.0f)) return -1;
    const float target = u * total;
    float run = 0.0f;
    int last_pos = -1;
    for (int base = 0; base < n; base += 32) {
        int i = base + lane;
        float x = (i < n) ? w(i) : 0.0f;
        float incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        unsigned hit = __ballot_sync(0xffffffffu, x > 0.0f && run + incl > target);
        if (hit) return base + __ffs(hit) - 1;
        unsigned pos = __ballot_sync(0xffffffffu, x > 0.0f);
        if (pos) last_pos = base + 31 - __clz(pos);
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    return last_pos;
}

// ----------------------------------------------------------------------------- 1. reweight

// The reweight's entry groups.  A group is four 16-bit entries (x: entries 0 and 1, y: 2 and
// 3); bits 0-14 of each index the staged chunk, whose shared address is base, and bit 15 of
// entry 0 says that the group ends the lane's current run (no other entry has bit 15 set).
// Written as PTX so that a group costs four shared loads and a handful of integer and float
// instructions, with no branch.
#define FA_RW_GATHER_PTX(OP)                                                                  \
    "{\n\t.reg .u32 a0, a1, a2, a3;\n\t.reg .f32 f0, f1, f2, f3;\n\t"                         \
    "and.b32 a0, %1, 32767;\n\tshr.u32 a1, %1, 16;\n\tand.b32 a2, %2, 65535;\n\tshr.u32 a3, %2, 16;\n\t" \
    "mad.lo.u32 a0, a0, 4, %3;\n\tmad.lo.u32 a1, a1, 4, %3;\n\t"                               \
    "mad.lo.u32 a2, a2, 4, %3;\n\tmad.lo.u32 a3, a3, 4, %3;\n\t"                               \
    "ld.shared.f32 f0, [a0];\n\tld.shared.f32 f1, [a1];\n\t"                                   \
    "ld.shared.f32 f2, [a2];\n\tld.shared.f32 f3, [a3];\n\t"                                   \
    OP ".f32 f0, f0, f1;\n\t" OP ".f32 f2, f2, f3;\n\t" OP ".f32 %0, f0, f2;\n\t}"

// Sum (MAX: maximum) of the four staged probabilities a group names.
template <bool MAX>
__device__ __forceinline__ float rw_gather(const uint2 v, uint32_t base) {
    float s;
    if constexpr (MAX) asm volatile(FA_RW_GATHER_PTX("max") : "=f"(s) : "r"(v.x), "r"(v.y), "r"(base));
    else asm volatile(FA_RW_GATHER_PTX("add") : "=f"(s) : "r"(v.x), "r"(v.y), "r"(base));
    return s;
}

#define FA_RW_END_PTX(OP)                                                                     \
    "{\n\t.reg .u32 t, ad;\n\t.reg .pred p;\n\t" OP ".f32 %0, %0, %2;\n\t"                    \
    "and.b32 t, %3, 32768;\n\tsetp.ne.u32 p, t, 0;\n\tselp.b32 ad, %1, %4, p;\n\t"             \
    "st.shared.f32 [ad], %0;\n\tselp.f32 %0, 0f00000000, %0, p;\n\t"                           \
    "shr.u32 t, t, 8;\n\tadd.u32 %1, %1, t;\n\t}"

// Adds a group's sum s to the lane's running run sum acc; if the group ends the run (x = the
// group's first two entries), stores acc at the run's slot, clears it and steps slot to the
// next one (128 bytes on); otherwise the store goes to the lane's dummy slot.
template <bool MAX>
__device__ __forceinline__ void rw_group_end(float s, uint32_t x, uint32_t dummy, float &acc, uint32_t &slot) {
    if constexpr (MAX) asm volatile(FA_RW_END_PTX("max") : "+f"(acc), "+r"(slot) : "f"(s), "r"(x), "r"(dummy));
    else asm volatile(FA_RW_END_PTX("add") : "+f"(acc), "+r"(slot) : "f"(s), "r"(x), "r"(dummy));
}

// One block per (position, row block): M_t(s, s') for rows s in [r0, r1), row exponent 0.  A
// masked position sums its probabilities over each cell's tokens (papernotes.org key design
// 1: g(x=v | z=e) = 1[v in label(e)] p_t(v), aggregated over the edges s -> s'); a committed
// position counts the edges s -> s' that carry its token.
//
// The probability row is staged in shared memory one vocabulary chunk at a time (the whole
// row when |V| <= FA_REWEIGHT_MAX_CHUNK) by asynchronous copies.  Warp w walks the entry
// streams of units u0 + w, u0 + w + FA_RW_WARPS, ... (UPW at most; see fa_automaton): lane l
// adds the staged probabilities of its entries and, at each run end, stores the run's chunk
// sum into its slot; after each walk the lane folds those slots into the unit's register
// totals, in chunk order.  After the last chunk the totals go to the freed chunk buffer and
// every cell adds its runs' totals in a fixed order, so the result is deterministic; with
// tile != 0 the block's rows are assembled in shared memory and written whole, each with its
// maximum and smallest nonzero entry.  fflag / fmap (non-null for a DFA on the tensor-core
// path): whether the position's M_t is a partial function (a committed position) and that
// function, s -> the target of the edge from s carrying the token (-1: none).
// MAX = true: the max-product variant for greedy decoding, M_t(s, s') = max over the tokens of
// the edges s -> s' of w_t(v) (a committed position: 1 where an edge carries its token).
template <bool MAX, int UPW>
__global__ void __launch_bounds__(32 * FA_RW_WARPS, 2) k_reweight(DevFA fa, int L, const float *__restrict__ probs,
                                                                const int32_t *__restrict__ committed,
                                                                const int4 *__restrict__ rbm, int nrb, int tot_floats,
                                                                    float *mant, int32_t *rho, int32_t *rmax,
                                                                    int32_t *rminc, int32_t *zero, long n_zero,
                                                                    int tile, int32_t *fflag, int32_t *fmap) {
    extern __shared__ float smem_f[];
    const int nthr = blockDim.x;
    // clear the row maxima of the higher tree levels (their products accumulate with atomicMax)
    {
        const long nb = (long)gridDim.x * gridDim.y;
        const long bid = (long)blockIdx.y * gridDim.x + blockIdx.x;
        for (long i = bid * nthr + threadIdx.x; i < n_zero; i += nb * nthr) zero[i] = 0;
    }
    const int S = fa.S, CH = fa.chunk_tokens, nch = fa.n_chunks;
    // shared memory: [0, tot_floats) holds the staged chunk, followed by the pad entries'
    // zero slots [CH, CH + FA_PAD_SLOTS), while the chunks are walked, then every unit's run
    // totals (FA_UNIT_SLOTS per unit) followed by the row maxima and the complemented row
    // minima; after it, one slot array per warp for the run sums of the chunk being walked,
    // then one dummy slot per lane that takes the stores of groups ending no run
    float *utot = smem_f;
    float *slots = smem_f + tot_floats;                    // [FA_RW_WARPS * FA_UNIT_SLOTS]
    const int t = blockIdx.x / nrb, r = blockIdx.x % nrb, b = blockIdx.y;
    const size_t pos = (size_t)b * L + t;
    // the block's metadata and the committed token, loaded together
    const int4 m0 = __ldg(rbm + 2 * r), m1 = __ldg(rbm + 2 * r + 1);
    const int c = committed[pos];
    const int r0 = m0.x, r1 = m0.y, u0 = m0.z, nu = m0.w - m0.z, c0 = m1.x, c1 = m1.y;
    int *smax = (int *)(utot + nu * FA_UNIT_SLOTS);        // [rows] row maxima (bits), once the chunks are done
    int *smin = smax + (r1 - r0);                          // [rows] complemented row minima
    float *M = mant + pos * (size_t)S * S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // a masked position writes every cell of its rows (whole rows when they are assembled in
    // shared memory): the rest of the rows is cleared, all of it unless the cells cover every
    // (s, s') pair of the rows
    if (c >= 0 || (!tile && c1 - c0 < (r1 - r0) * S))
        for (size_t i = (size_t)r0 * S + tid; i < (size_t)r1 * S; i += nthr) M[i] = 0.0f;
    // functional spans (DFA): a committed position's M_t is the partial function s -> the
    // target of the edge from s carrying its token; a masked position's is not functional
    if (fflag && r == 0 && tid == 0) fflag[pos] = c >= 0 ? 1 : 0;
    if (c < 0) {
        const float *prow = probs + pos * (size_t)fa.V;
        const bool aligned = (reinterpret_cast<uintptr_t>(prow) & 15) == 0 && (CH & 3) == 0;
        const uint2 *g4 = reinterpret_cast<const uint2 *>(fa.ru_tok);
        // a run's sum for the current chunk is stored (not added) into the lane's slot at its
        // end; after each walk the lane folds the slots it wrote into register totals, in chunk
        // order.  Warp w walks units w, w + FA_RW_WARPS, ... of the block (UPW at most).
        float *my = slots + warp * FA_UNIT_SLOTS + lane;
        const uint32_t my_addr = (uint32_t)__cvta_generic_to_shared(my);
        // one dummy slot per lane after the warps' slot arrays (shared by the warps; never read)
        const uint32_t dummy_addr =
            (uint32_t)__cvta_generic_to_shared(slots + (blockDim.x >> 5) * FA_UNIT_SLOTS + lane);
        float tot[UPW][FA_RUN_SLOTS];
#pragma unroll
        for (int h = 0; h < UPW; ++h)
#pragma unroll
            for (int q = 0; q < FA_RUN_SLOTS; ++q) tot[h][q] = 0.0f;
        for (int ch = 0; ch < nch; ++ch) {
            const int base = ch * CH, n = min(CH, fa.V - base);
            // the warp's units' stream bounds for this chunk and the first unit's first four
            // groups, loaded before the staging so that their latency overlaps it
            int gbv[UPW], ngv[UPW];
#pragma unroll
            for (int h = 0; h < UPW; ++h) {
                const int uw = warp + FA_RW_WARPS * h;
                ngv[h] = -1;
                gbv[h] = 0;
                if (uw < nu) {
                    const size_t ui = (size_t)(u0 + uw) * nch + ch;
                    gbv[h] = __ldg(fa.ru_goff + ui);
                    ngv[h] = (__ldg(fa.ru_goff + ui + 1) - gbv[h]) >> 5;
                }
            }
            uint2 f0v = __ldg(g4 + gbv[0] + lane), f1v = __ldg(g4 + gbv[0] + lane + 32);
            uint2 f2v = __ldg(g4 + gbv[0] + lane + 64), f3v = __ldg(g4 + gbv[0] + lane + 96);
            __syncthreads();  // every warp is done with the previous chunk
            if (aligned) {
                // asynchronous 16-byte global->shared copies, all in flight before one wait
                const char *src = reinterpret_cast<const char *>(prow + base);
                const unsigned d = (unsigned)__cvta_generic_to_shared(smem_f);
                for (int i = tid; i < (n >> 2); i += nthr)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d + 16u * i), "l"(src + 16 * (size_t)i)
                                 : "memory");
                asm volatile("cp.async.commit_group;\n" ::: "memory");
                for (int i = (n & ~3) + tid; i < n; i += nthr) smem_f[i] = __ldg(prow + base + i);
            } else {
                for (int i = tid; i < n; i += nthr) smem_f[i] = __ldg(prow + base + i);
            }
            if (tid < FA_PAD_SLOTS) smem_f[CH + tid] = 0.0f;  // the pad entries' zero slots
            asm volatile("cp.async.wait_all;\n" ::: "memory");
            __syncthreads();
#pragma unroll
            for (int h = 0; h < UPW; ++h) {
                const int ng = ngv[h];
                if (ng < 0) break;
                const uint2 *gp = g4 + gbv[h] + lane;
                float acc = 0.0f;
                uint32_t slot_addr = my_addr;  // shared address of the current run's slot
                const uint32_t cbase = (uint32_t)__cvta_generic_to_shared(smem_f);
                // whole steps of four groups (their sixteen gathers first, then the run-end
                // stores), the next four loaded (unconditionally: the stream array is padded
                // past its end) while these are summed; then the tail
                uint2 c0v, c1v, c2v, c3v;
                if (h == 0) {
                    c0v = f0v; c1v = f1v; c2v = f2v; c3v = f3v;
                } else {
                    c0v = __ldg(gp); c1v = __ldg(gp + 32); c2v = __ldg(gp + 64); c3v = __ldg(gp + 96);
                }
                int k = 0;
                for (; k + 4 <= ng; k += 4) {
                    gp += 128;
                    const uint2 n0 = __ldg(gp), n1 = __ldg(gp + 32), n2 = __ldg(gp + 64), n3 = __ldg(gp + 96);
                    const float s0 = rw_gather<MAX>(c0v, cbase), s1 = rw_gather<MAX>(c1v, cbase);
                    const float s2 = rw_gather<MAX>(c2v, cbase), s3 = rw_gather<MAX>(c3v, cbase);
                    rw_group_end<MAX>(s0, c0v.x, dummy_addr, acc, slot_addr);
                    rw_group_end<MAX>(s1, c1v.x, dummy_addr, acc, slot_addr);
                    rw_group_end<MAX>(s2, c2v.x, dummy_addr, acc, slot_addr);
                    rw_group_end<MAX>(s3, c3v.x, dummy_addr, acc, slot_addr);
                    c0v = n0; c1v = n1; c2v = n2; c3v = n3;
                }
                if (k < ng) rw_group_end<MAX>(rw_gather<MAX>(c0v, cbase), c0v.x, dummy_addr, acc, slot_addr);
                if (k + 1 < ng) rw_group_end<MAX>(rw_gather<MAX>(c1v, cbase), c1v.x, dummy_addr, acc, slot_addr);
                if (k + 2 < ng) rw_group_end<MAX>(rw_gather<MAX>(c2v, cbase), c2v.x, dummy_addr, acc, slot_addr);
                // the slot stores above are ordered before the reads below
                asm volatile("" ::: "memory");
                // runs of this lane = run ends seen in the walk; fold the slots it wrote (the
                // others may hold the sums of the warp's other unit); every lane reads only its
                // own slots
                const int mine = (int)((slot_addr - my_addr) >> 7);
#pragma unroll
                for (int q = 0; q < FA_RUN_SLOTS; ++q) {
                    const float sv = q < mine ? my[q * 32] : 0.0f;
                    if constexpr (MAX) tot[h][q] = fmaxf(tot[h][q], sv); else tot[h][q] += sv;
                }
                asm volatile("" ::: "memory");
            }
        }
        __syncthreads();  // the chunk buffer is free now: it takes the units' totals
#pragma unroll
        for (int h = 0; h < UPW; ++h) {
            const int uw = warp + FA_RW_WARPS * h;
            if (uw < nu) {
#pragma unroll
                for (int q = 0; q < FA_RUN_SLOTS; ++q) utot[uw * FA_UNIT_SLOTS + q * 32 + lane] = tot[h][q];
            }
        }
        // tile != 0: the block's rows of M_t are assembled in shared memory after the totals
        // (dense, zero where no cell lies) and written out row by row, coalesced, with each
        // row's maximum and smallest nonzero entry; else cells store straight to M_t
        float *mt = utot + nu * FA_UNIT_SLOTS;
        const int nrow = r1 - r0;
        if (tile) {
            for (int i = tid; i < nrow * S; i += nthr) mt[i] = 0.0f;
        } else {
            for (int i = tid; i < nrow; i += nthr) { smax[i] = 0; smin[i] = 0; }
        }
        __syncthreads();
#pragma unroll 4
        for (int cell = c0 + tid; cell < c1; cell += nthr) {
            const int2 rec = __ldg(fa.cell_rec + cell);
            float v = 0.0f;
            if (rec.y >= 0) {
                v = utot[rec.y - u0 * FA_UNIT_SLOTS];   // a cell of one run
            } else {
                const float *sb = utot + (size_t)(fa.row_unit0[rec.x / S] - u0) * FA_UNIT_SLOTS;
                for (int q = fa.crun_off[cell]; q < fa.crun_off[cell + 1]; ++q) {
                    if constexpr (MAX) v = fmaxf(v, sb[fa.crun_slot[q]]); else v += sb[fa.crun_slot[q]];
                }
            }
            if (tile) {
                mt[rec.x - r0 * S] = v;
                continue;
            }
            const int s = rec.x / S;
            M[rec.x] = v;
            // consecutive cells mostly share a row: one atomic per row and warp
            const unsigned act = __activemask();
            const unsigned same = __match_any_sync(act, s);
            const int rowmax = (int)__reduce_max_sync(same, (unsigned)__float_as_int(v));
            const int rowminc = (int)__reduce_max_sync(same, v > 0.0f ? 0x7fffffffu - (unsigned)__float_as_int(v) : 0u);
            if ((threadIdx.x & 31) == __ffs(same) - 1) {
                atomicMax(&smax[s - r0], rowmax);
                atomicMax(&smin[s - r0], rowminc);
            }
        }
        if (tile) {
            __syncthreads();
            // one warp per row (entries are >= 0, so their bit patterns order like the values)
            for (int r = warp; r < nrow; r += nthr >> 5) {
                const float *src = mt + r * S;
                float *dst = M + (size_t)(r0 + r) * S;
                unsigned mx = 0u, mnc = 0u;
                auto see = [&](float v) {
                    const unsigned b = (unsigned)__float_as_int(v);
                    mx = max(mx, b);
                    if (v > 0.0f) mnc = max(mnc, 0x7fffffffu - b);
                };
                if (tile == 2) {  // S % 4 == 0 and M_t 16-byte aligned: float4 rows
                    for (int j = 4 * lane; j < S; j += 128) {
                        const float4 v = *reinterpret_cast<const float4 *>(src + j);
                        *reinterpret_cast<float4 *>(dst + j) = v;
                        see(v.x); see(v.y); see(v.z); see(v.w);
                    }
                } else {
                    for (int j = lane; j < S; j += 32) {
                        const float v = src[j];
                        dst[j] = v;
                        see(v);
                    }
                }
                mx = __reduce_max_sync(0xffffffffu, mx);
                mnc = __reduce_max_sync(0xffffffffu, mnc);
                if (lane == 0) {
                    rho[pos * S + r0 + r] = 0;
                    if (rmax) rmax[pos * S + r0 + r] = (int)mx;
                    if (rminc) rminc[pos * S + r0 + r] = (int)mnc;
                }
            }
            return;
        }
    } else {
        for (int i = tid; i < r1 - r0; i += nthr) {
            smax[i] = 0;
            smin[i] = 0;
            if (fmap) fmap[pos * S + r0 + i] = -1;
        }
        __syncthreads();
        if (c < fa.V) {
            const int64_t a0 = fa.tok_off[c], a1 = fa.tok_off[c + 1];
            for (int64_t j = a0 + tid; j < a1; j += nthr) {
                const int e = fa.tok_edges[j];
                const int s = fa.edge_src[e];
                if (s >= r0 && s < r1) {
                    if constexpr (MAX) M[(size_t)s * S + fa.edge_dst[e]] = 1.0f;
                    else atomicAdd(&M[(size_t)s * S + fa.edge_dst[e]], 1.0f);
                    if (fmap) fmap[pos * S + s] = fa.edge_dst[e];   // one edge per (s, token) in a DFA
                }
            }
            __syncthreads();
            for (int64_t j = a0 + tid; j < a1; j += nthr) {
                const int e = fa.tok_edges[j];
                const int s = fa.edge_src[e];
                if (s >= r0 && s < r1) {
                    const int bits = __float_as_int(M[(size_t)s * S + fa.edge_dst[e]]);  // an edge count >= 1
                    atomicMax(&smax[s - r0], bits);
                    atomicMax(&smin[s - r0], 0x7fffffff - bits);
                }
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < r1 - r0; i += nthr) {
        rho[pos * S + r0 + i] = 0;
        if (rmax) rmax[pos * S + r0 + i] = smax[i];
        if (rminc) rminc[pos * S + r0 + i] = smin[i];
    }
}

// ----------------------------------------------------------------------------- 2. up-sweep

// Row shift for the product C = A_left * A_right at tree level k (paperfeed.app, "The scan
// trick": 2^k-step transitions from two 2^(k-1)-step ones).  For row i,
//   C[i, :] = 2^rhoL[i] * sum_m Ã_L[i, m] 2^rhoR[m] Ã_R[m, :]
// and mu[i] = max over m with Ã_L[i, m] > 0 and a nonzero right row m of
// rhoR[m] + e(rmaxR[m]) + e(Ã_L[i, m]), so the prescaled left row
// Ã_L[i, m] 2^(rhoR[m] - mu[i]) keeps its largest contribution near 1.  Also clears rmax of
// the product.  One warp per row.
__global__ void __launch_bounds__(kThreads) k_rowshift(int S, int L, int k, int nk, const float *__restrict__ mant_c,
                                                     const int32_t *__restrict__ rho_c,
                                                     const int32_t *__restrict__ rmax_c, int nc, int32_t *mu,
                                                     int32_t *rmax_p, const int32_t *__restrict__ fflag_p) {
    const int b = blockIdx.z, j = blockIdx.y;
    const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (i >= S) return;
    const size_t pnode = (size_t)b * nk + j;
    if (lane == 0) rmax_p[pnode * S + i] = 0;
    const bool has_right = ((2 * j + 1) << (k - 1)) < L;
    if (!has_right || (fflag_p && fflag_p[pnode])) return;   // a copy, or a functional span
    const size_t lnode = (size_t)b * nc + 2 * j, rnode = lnode + 1;
    const float *Lrow = mant_c + lnode * (size_t)S * S + (size_t)i * S;
    const int32_t *rhoR = rho_c + rnode * S;
    const int32_t *rmaxR = rmax_c + rnode * S;
    int best = FA_INT_NONE;
    if ((S & 3) == 0) {
        // 16-byte loads, four in flight per lane
        for (int m0 = 4 * lane; m0 < S; m0 += 512) {
            float4 x[4];
            int4 rr[4], rh[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int m = m0 + 128 * u;
                x[u] = m < S ? __ldg(reinterpret_cast<const float4 *>(Lrow + m)) : make_float4(0.f, 0.f, 0.f, 0.f);
                rr[u] = m < S ? __ldg(reinterpret_cast<const int4 *>(rmaxR + m)) : make_int4(0, 0, 0, 0);
                rh[u] = m < S ? __ldg(reinterpret_cast<const int4 *>(rhoR + m)) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                const int rs[4] = {rr[u].x, rr[u].y, rr[u].z, rr[u].w}, hs[4] = {rh[u].x, rh[u].y, rh[u].z, rh[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (xs[e] > 0.0f && rs[e] > 0) best = max(best, hs[e] + fa_exponent(__int_as_float(rs[e])) + fa_exponent(xs[e]));
            }
        }
    } else {
        for (int m = lane; m < S; m += 32) {
            const float x = Lrow[m];
            const int rr = rmaxR[m];
            if (x > 0.0f && rr > 0) best = max(best, rhoR[m] + fa_exponent(__int_as_float(rr)) + fa_exponent(x));
        }
    }
    best = fa_warp_max_int(best);
    if (lane == 0) mu[pnode * S + i] = best;
}

// Functional spans of tree level k (a DFA, tensor-core path): a node is functional when its
// children are (a copy node, whose right child is padding, when its left child is), and its
// partial function composes theirs, f(s) = f_R(f_L(s)).  Such a span is the 0/1 matrix of
// that function with row exponents 0 -- exactly what the product of the two 0/1 matrices
// gives -- so the level's products skip it and write the matrix from the function.  One block
// per node.
__global__ void __launch_bounds__(kThreads) k_func_level(int S, int L, int k, int nk, int nc,
                                                       const int32_t *__restrict__ fflag_c,
                                                       const int32_t *__restrict__ fmap_c, int32_t *fflag_p,
                                                       int32_t *fmap_p) {
    const long pn = blockIdx.x;                    // b * nk + node
    const int node = (int)(pn % nk), b = (int)(pn / nk);
    const size_t lnode = (size_t)b * nc + 2 * node, rnode = lnode + 1;
    const bool has_right = ((2 * node + 1) << (k - 1)) < L;
    const int f = fflag_c[lnode] && (!has_right || fflag_c[rnode]);
    if (threadIdx.x == 0) fflag_p[pn] = f;
    if (!f) return;
    const int32_t *fl = fmap_c + lnode * S, *fr = fmap_c + rnode * S;
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        const int m = fl[i];
        fmap_p[(size_t)pn * S + i] = m < 0 ? -1 : (has_right ? fr[m] : m);
    }
}

// |S| <= 64: a product C = A_L A_R of one node is split into 32x32 output tiles, one block
// each, with the row shift mu (see k_rowshift) recomputed per block from its 32 full rows and
// the row maxima combined across column tiles with atomicMax (cleared by the reweight).
constexpr int SMALL_S = 64;
constexpr int ST = 32;

template <bool MAX>
__global__ void __launch_bounds__(kThreads) k_span_small(int S, int L, int k, int nk, const float *__restrict__ mant_c,
                                                       const int32_t *__restrict__ rho_c,
                                                       const int32_t *__restrict__ rmax_c,
                                                       const int32_t *__restrict__ rminc_c, int nc, float *mant_p,
                                                       int32_t *rho_p, int32_t *rmax_p, int32_t *rminc_p,
                                                       int32_t *range_lost) {
    // the A tile is stored transposed (At[m][row]) and both tiles padded to 16-byte rows, so
    // the inner loop reads two float2 per step
    __shared__ __align__(16) float At[SMALL_S][ST + 4];
    __shared__ __align__(16) float Bs[SMALL_S][ST + 4];
    __shared__ int rhoR_s[SMALL_S], rmaxR_s[SMALL_S], eminR_s[SMALL_S], mu_s[ST];
    const int tpd = (S + ST - 1) / ST;
    const int tile = blockIdx.x % (tpd * tpd);
    const long bn = blockIdx.x / (tpd * tpd);
    const int node = (int)(bn % nk), b = (int)(bn / nk);
    const int i0 = (tile / tpd) * ST, j0 = (tile % tpd) * ST;
    const int tid = threadIdx.x;
    const size_t pnode = (size_t)b * nk + node;
    const size_t lnode = (size_t)b * nc + 2 * node, rnode = lnode + 1;
    const size_t SS = (size_t)S * S;
    const float *A = mant_c + lnode * SS;
    float *C = mant_p + pnode * SS;
    if (((2 * node + 1) << (k - 1)) >= L) {      // right child is padding: C = A_L
        for (int q = tid; q < ST * ST; q += kThreads) {
            const int r = i0 + q / ST, c = j0 + q % ST;
            if (r < S && c < S) C[(size_t)r * S + c] = A[(size_t)r * S + c];
        }
        if (j0 == 0)
            for (int r = i0 + tid; r < min(i0 + ST, S); r += kThreads) {
                rho_p[pnode * S + r] = rho_c[lnode * S + r];
                rmax_p[pnode * S + r] = rmax_c[lnode * S + r];
                rminc_p[pnode * S + r] = rminc_c[lnode * S + r];
            }
        return;
    }
    const float *Bm = mant_c + rnode * SS;
    {
        // all loads of this thread in flight before any shared-memory store
        constexpr int U = ST * SMALL_S / kThreads;  // 8
        float va[U], vb[U];
        int ra = 0, rr = 0, rn = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = tid + u * kThreads;
            const int r = q / SMALL_S, c = q % SMALL_S;                  // A: 32 rows x 64 cols
            va[u] = (i0 + r < S && c < S) ? __ldg(A + (size_t)(i0 + r) * S + c) : 0.0f;
            const int rb = q / ST, cb = q % ST;                          // B: 64 rows x 32 cols
            vb[u] = (rb < S && j0 + cb < S) ? __ldg(Bm + (size_t)rb * S + j0 + cb) : 0.0f;
        }
        if (tid < SMALL_S) {
            ra = tid < S ? rho_c[rnode * S + tid] : 0;
            rr = tid < S ? rmax_c[rnode * S + tid] : 0;
            rn = tid < S ? rminc_c[rnode * S + tid] : 0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = tid + u * kThreads;
            At[q % SMALL_S][q / SMALL_S] = va[u];
            Bs[q / ST][q % ST] = vb[u];
        }
        if (tid < SMALL_S) {
            rhoR_s[tid] = ra;
            rmaxR_s[tid] = rr;
            // exponent of the right row's smallest nonzero entry, capped at 0
            eminR_s[tid] = rn > 0 ? min(0, fa_exponent(__int_as_float(0x7fffffff - rn))) : 0;
        }
    }
    __syncthreads();
    {
        // row shift: eight threads per row, each over every eighth inner index, then three
        // shuffles (all 32 rows at once)
        const int r = tid >> 3, seg = tid & 7;
        int best = FA_INT_NONE;
        for (int m = seg; m < S; m += 8) {
            const float x = At[m][r];
            const int q = rmaxR_s[m];
            if (x > 0.0f && q > 0) best = max(best, rhoR_s[m] + fa_exponent(__int_as_float(q)) + fa_exponent(x));
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
        if (seg == 0) mu_s[r] = best;
    }
    __syncthreads();
    int lost = 0;
    for (int q = tid; q < ST * SMALL_S; q += kThreads) {
        const int m = q / ST, r = q % ST;
        const float x = At[m][r];
        const int mr = mu_s[r];
        const bool live = x > 0.0f && mr != FA_INT_NONE && m < S && rmaxR_s[m] > 0;
        // a nonzero entry prescaled below the normal range, or whose product with the right
        // row's smallest entry would be, may lose its mass
        if (live && fa_exponent(x) + rhoR_s[m] - mr + eminR_s[m] < -126) lost = 1;
        At[m][r] = live ? fa_mul_pow2(x, rhoR_s[m] - mr) : 0.0f;
    }
    if (__syncthreads_or(lost) && tid == 0) atomicOr(range_lost + b, 1);
    const int tx = tid & 15, ty = tid >> 4;          // 2x2 outputs per thread
    float c00 = 0.0f, c01 = 0.0f, c10 = 0.0f, c11 = 0.0f;
    auto step = [&](int m) {
        const float2 a = *reinterpret_cast<const float2 *>(&At[m][2 * ty]);
        const float2 bq = *reinterpret_cast<const float2 *>(&Bs[m][2 * tx]);
        if constexpr (MAX) {
            c00 = fmaxf(c00, a.x * bq.x); c01 = fmaxf(c01, a.x * bq.y);
            c10 = fmaxf(c10, a.y * bq.x); c11 = fmaxf(c11, a.y * bq.y);
        } else {
            c00 = fmaf(a.x, bq.x, c00); c01 = fmaf(a.x, bq.y, c01);
            c10 = fmaf(a.y, bq.x, c10); c11 = fmaf(a.y, bq.y, c11);
        }
    };
    int m = 0;
    for (; m + 8 <= S; m += 8) {
#pragma unroll
        for (int u = 0; u < 8; ++u) step(m + u);
    }
    for (; m < S; ++m) step(m);
    const float cv[2][2] = {{c00, c01}, {c10, c11}};
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int i = i0 + 2 * ty + p;
        float mx = 0.0f, mn = FLT_MAX;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int j = j0 + 2 * tx + q;
            if (i < S && j < S) {
                C[(size_t)i * S + j] = cv[p][q];
                mx = fmaxf(mx, cv[p][q]);
                if (cv[p][q] > 0.0f) mn = fminf(mn, cv[p][q]);
            }
        }
#pragma unroll
        for (int o = 8; o; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        if (tx == 0 && i < S) {
            if (mx > 0.0f) {
                atomicMax(&rmax_p[pnode * S + i], __float_as_int(mx));
                atomicMax(&rminc_p[pnode * S + i], 0x7fffffff - __float_as_int(mn));
            }
            if (j0 == 0) {
                const int mr = mu_s[2 * ty + p];
                rho_p[pnode * S + i] = (mr == FA_INT_NONE) ? 0 : rho_c[lnode * S + i] + mr;
            }
        }
    }
}

constexpr int GBM = 64, GBN = 64, GBK = 16;

// C̃ = (Ã_L prescaled per (row, m)) x Ã_R in fp32 FMA, 64x64 tiles, 4x4 per thread.  A
// product whose right child lies wholly in the padding beyond L is a copy of the left child.
template <bool MAX>
__global__ void __launch_bounds__(kThreads) k_gemm_simt(int S, int L, int k, int nk, const float *__restrict__ mant_c,
                                                      const int32_t *__restrict__ rho_c,
                                                      const int32_t *__restrict__ rmax_c,
                                                      const int32_t *__restrict__ rminc_c, int nc,
                                                      const int32_t *__restrict__ mu, float *mant_p, int32_t *rho_p,
                                                      int32_t *rmax_p, int32_t *rminc_p, int32_t *range_lost) {
    __shared__ float As[GBK][GBM + 4];
    __shared__ float Bs[GBK][GBN + 4];
    __shared__ int mu_s[GBM];
    const int tiles = (S + GBN - 1) / GBN;
    const long flat = blockIdx.x;                       // ((b * nk + node) * tiles + ti) * tiles + tj
    const int tj = (int)(flat % tiles), ti = (int)((flat / tiles) % tiles);
    const long bn = flat / ((long)tiles * tiles);
    const int node = (int)(bn % nk), b = (int)(bn / nk);
    const int i0 = ti * GBM, j0 = tj * GBN;
    const int tid = threadIdx.x;
    const size_t pnode = (size_t)b * nk + node;
    const size_t lnode = (size_t)b * nc + 2 * node, rnode = lnode + 1;
    const float *A = mant_c + lnode * (size_t)S * S;
    float *C = mant_p + pnode * (size_t)S * S;
    const bool has_right = ((2 * node + 1) << (k - 1)) < L;
    if (!has_right) {
        for (int q = tid; q < GBM * GBN; q += kThreads) {
            const int r = q / GBN, c = q % GBN;
            if (i0 + r < S && j0 + c < S) C[(size_t)(i0 + r) * S + j0 + c] = A[(size_t)(i0 + r) * S + j0 + c];
        }
        if (tj == 0)
            for (int r = tid; r < GBM; r += kThreads)
                if (i0 + r < S) {
                    rho_p[pnode * S + i0 + r] = rho_c[lnode * S + i0 + r];
                    rmax_p[pnode * S + i0 + r] = rmax_c[lnode * S + i0 + r];
                    rminc_p[pnode * S + i0 + r] = rminc_c[lnode * S + i0 + r];
                }
        return;
    }
    const float *Bm = mant_c + rnode * (size_t)S * S;
    const int32_t *rhoR = rho_c + rnode * S;
    const int32_t *rmaxR = rmax_c + rnode * S;
    const int32_t *rmincR = rminc_c + rnode * S;
    for (int r = tid; r < GBM; r += kThreads) mu_s[r] = (i0 + r < S) ? mu[pnode * S + i0 + r] : FA_INT_NONE;
    __syncthreads();
    const int tx = tid & 15, ty = tid >> 4;
    float acc[4][4] = {};
    int lost = 0;
    for (int k0 = 0; k0 < S; k0 += GBK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * kThreads;
            const int r = idx / GBK, kk = idx % GBK;
            const int i = i0 + r, m = k0 + kk;
            float v = 0.0f;
            if (i < S && m < S) {
                const float x = A[(size_t)i * S + m];
                const int mr = mu_s[r];
                if (x > 0.0f && mr != FA_INT_NONE && rmaxR[m] > 0) {
                    // below the normal range after the prescale, alone or times the right
                    // row's smallest entry: mass may be lost
                    const int rn = rmincR[m];
                    const int emin = rn > 0 ? min(0, fa_exponent(__int_as_float(0x7fffffff - rn))) : 0;
                    if (fa_exponent(x) + rhoR[m] - mr + emin < -126) lost = 1;
                    v = fa_mul_pow2(x, rhoR[m] - mr);
                }
            }
            As[kk][r] = v;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * kThreads;
            const int kk = idx / GBN, c = idx % GBN;
            const int m = k0 + kk, j = j0 + c;
            Bs[kk][c] = (m < S && j < S) ? Bm[(size_t)m * S + j] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GBK; ++kk) {
            float a[4], bb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) { a[q] = As[kk][ty * 4 + q]; bb[q] = Bs[kk][tx * 4 + q]; }
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (MAX) acc[p][q] = fmaxf(acc[p][q], a[p] * bb[q]);
                    else acc[p][q] = fmaf(a[p], bb[q], acc[p][q]);
                }
        }
        __syncthreads();
    }
    if (__syncthreads_or(lost) && tid == 0) atomicOr(range_lost + b, 1);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int i = i0 + ty * 4 + p;
        float mx = 0.0f, mn = FLT_MAX;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = j0 + tx * 4 + q;
            if (i < S && j < S) {
                C[(size_t)i * S + j] = acc[p][q];
                mx = fmaxf(mx, acc[p][q]);
                if (acc[p][q] > 0.0f) mn = fminf(mn, acc[p][q]);
            }
        }
#pragma unroll
        for (int o = 8; o; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        if (tx == 0 && i < S) {
            if (mx > 0.0f) {
                atomicMax(&rmax_p[pnode * S + i], __float_as_int(mx));
                atomicMax(&rminc_p[pnode * S + i], 0x7fffffff - __float_as_int(mn));
            }
            if (tj == 0) {
                const int mr = mu_s[ty * 4 + p];
                rho_p[pnode * S + i] = (mr == FA_INT_NONE) ? 0 : rho_c[lnode * S + i] + mr;
            }
        }
    }
}

// ----------------------------------------------------------------------------- 3. root

// Z = e_{s0}^T A_root 1_F, the end state z_L ~ A_root[s0, f] over f in F, and the boundary
// messages alpha_0 = e_{s0}, beta_L = 1_F (papernotes.org key design 2: sample the boundary
// states from the joint marginal; the start is pinned to s0).
__global__ void __launch_bounds__(kThreads) k_root(DevFA fa, int L, int K, int nK, const float *__restrict__ mant_root,
                                                 const int32_t *__restrict__ rho_root, uint64_t seed, uint64_t offset,
                                                 int32_t *z, float *am, int32_t *ae, float *bm, int32_t *be,
                                                 float *zsum_ws, int32_t *zexp_ws, double *logZ, int32_t *status,
                                                 const int32_t *__restrict__ tc_err,
                                                 const int32_t *__restrict__ range_lost) {
    const int b = blockIdx.x, S = fa.S, s0 = fa.start;
    const float *row = mant_root + (size_t)b * nK * S * S + (size_t)s0 * S;
    const size_t bnd0 = (size_t)b * (L + 1);
    for (int s = threadIdx.x; s < S; s += kThreads) {
        am[bnd0 * S + s] = (s == s0) ? 1.0f : 0.0f;
        ae[bnd0 * S + s] = 0;
        bm[(bnd0 + L) * S + s] = fa.accept_mask[s] ? 1.0f : 0.0f;
        be[(bnd0 + L) * S + s] = 0;
    }
    if (threadIdx.x >= 32) return;
    const float u = fa_uniform(seed, offset, 0u, (uint32_t)b, FA_RNG_ROOT);
    const int pick = warp_categorical(fa.n_accept, u, [&](int i) { return row[fa.accept[i]]; });
    float tot = 0.0f;
    for (int i = threadIdx.x; i < fa.n_accept; i += 32) tot += row[fa.accept[i]];
    tot = fa_warp_sum(tot);
    if (threadIdx.x == 0) {
        z[bnd0] = s0;
        if (tc_err && *tc_err) {
            status[b] = FA_ROW_TIMEOUT;
            logZ[b] = -INFINITY;
            z[bnd0 + L] = s0;
            zsum_ws[b] = 0.0f;
            zexp_ws[b] = 0;
        } else if (range_lost && range_lost[b]) {
            // the up-sweep dropped nonzero mass below the fp32 range: Z and every draw from
            // these spans may be wrong, so none is reported
            status[b] = FA_ROW_UNDERFLOW;
            logZ[b] = NAN;
            z[bnd0 + L] = s0;
            zsum_ws[b] = 0.0f;
            zexp_ws[b] = 0;
        } else if (pick < 0 || !(tot > 0.0f)) {
            status[b] = FA_ROW_EMPTY;
            logZ[b] = -INFINITY;
            z[bnd0 + L] = s0;
            zsum_ws[b] = 0.0f;
            zexp_ws[b] = 0;
        } else {
            status[b] = FA_ROW_OK;
            const int rr = rho_root[(size_t)b * nK * S + s0];
            logZ[b] = (double)rr * 0.69314718055994530942 + log((double)tot);
            z[bnd0 + L] = fa.accept[pick];
            zsum_ws[b] = tot;
            zexp_ws[b] = rr;
        }
    }
}

// ----------------------------------------------------------------------------- 4. top-down

// One launch per tree level k+1 (K-1 down to 0) does three independent jobs for every node
// [l, r) of that level with midpoint m < L (blocks are split by role):
//  - midpoint: z_m ~ A[l, m)[z_l, s] * A[m, r)[s, z_r] (paperfeed.app, "The scan trick";
//    papernotes.org key design 2: given the segment ends the two halves are conditionally
//    independent given the midpoint), one warp per node;
//  - prefix message alpha_m = alpha_l A[l, m), CB columns x QS row splits per block;
//  - suffix message beta_m = A[m, r) beta_r, one warp per row.
// Messages keep a mantissa in [1, 2) and an exponent per state, so no state is lost to range;
// each sum is formed in two passes (largest term exponent, then terms scaled to it).
struct TopdownArgs {
    int S, B, L, k, nc, np;
    int nA, nB;           // number of alpha and beta blocks
    int CB, QS;           // alpha: columns per block, row splits
    const float *mant;    // level-k spans
    const int32_t *rho, *rmax;
    int vec4;             // |S| % 4 == 0: 16-byte loads in the message passes
    int beta_rows;        // rows per beta block: a multiple of the warps, more for large |S| so
                          // that the staging of beta_r is shared by more rows
    const int32_t *fflag, *fmap;   // functional spans of the level (nullptr: none)
    uint64_t seed, offset;
    int32_t *z, *status;
    float *am, *bm;
    int32_t *ae, *be;
};

__device__ void topdown_midpoint(const TopdownArgs &a, int blk) {
    const int S = a.S, L = a.L, k = a.k;
    const long gw = (long)blk * kWarps + (threadIdx.x >> 5);
    if (gw >= (long)a.B * a.np) return;
    const int b = (int)(gw / a.np), j = (int)(gw % a.np);
    const int l = j << (k + 1), m = l + (1 << k);
    if (m >= L) return;
    const int r = min(l + (1 << (k + 1)), L);
    if (__shfl_sync(0xffffffffu, a.status[b], 0) != FA_ROW_OK) return;
    const int32_t *zb = a.z + (size_t)b * (L + 1);
    const int zl = zb[l], zr = zb[r];
    const size_t lnode = (size_t)b * a.nc + 2 * j, rnode = lnode + 1;
    const float *Lrow = a.mant + lnode * (size_t)S * S + (size_t)zl * S;
    const float *R = a.mant + rnode * (size_t)S * S;
    const int32_t *rhoR = a.rho + rnode * S;
    const int lane = threadIdx.x & 31;
    int emax = FA_INT_NONE;
    for (int s = lane; s < S; s += 32) {
        const float x = Lrow[s], y = R[(size_t)s * S + zr];
        if (x > 0.0f && y > 0.0f) emax = max(emax, rhoR[s] + fa_exponent(x) + fa_exponent(y));
    }
    emax = fa_warp_max_int(emax);
    int pick = -1;
    if (emax != FA_INT_NONE) {
        const float u = fa_uniform(a.seed, a.offset, (uint32_t)m, (uint32_t)b, FA_RNG_MID);
        pick = warp_categorical(S, u, [&](int s) {
            const float x = Lrow[s], y = R[(size_t)s * S + zr];
            if (!(x > 0.0f && y > 0.0f)) return 0.0f;
            float mx, my;
            int ex, ey;
            fa_split(x, mx, ex);
            fa_split(y, my, ey);
            return mx * my * fa_pow2(rhoR[s] + ex + ey - emax);
        });
    }
    if (lane == 0) {
        if (pick < 0) a.status[b] = FA_ROW_UNDERFLOW;
        else a.z[(size_t)b * (L + 1) + m] = pick;
    }
}

// Messages: one scaled pass, the exact two-pass form where it is needed.  Every term of a
// message entry is alpha_l(q) A(q, col) (beta: A(row, q) beta_r(q)), each with its own
// exponent.  The fast pass scales all terms by one power of two, chosen so that the largest
// term any row can give is at most about 4, and keeps the plain fp32 sum when that sum is
// at least 2^-60: the terms that lose precision below the fp32 normal range then add at
// most |S| 2^-126, under 2^-57 of the sum.  A second sum with every scale set to 1 tells an
// exactly zero entry apart (the terms are non-negative, so a positive one never cancels).
// Any other entry -- a state whose weight is far below the largest, such as one a committed
// token reaches only through rare tokens -- takes the exact form: the largest term's
// exponent first, then the sum scaled by it, so no state is lost to range.
constexpr float kMsgFastMin = 8.6736174e-19f;  // 2^-60

__device__ __forceinline__ int fa_block_max_int(int v, int *red) {
    v = fa_warp_max_int(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int r = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = max(r, red[i]);
    __syncthreads();
    return r;
}

__device__ void topdown_alpha(const TopdownArgs &a, int blk, float *sm) {
    const int S = a.S, L = a.L, k = a.k, CB = a.CB, QS = a.QS;
    const int ncb = (S + CB - 1) / CB;
    const int cbk = blk % ncb;
    const long bj = blk / ncb;
    const int j = (int)(bj % a.np), b = (int)(bj / a.np);
    const int l = j << (k + 1), m = l + (1 << k);
    if (m >= L) return;
    float *sa = sm;                          // [S] mantissas of alpha_l
    int *sc = (int *)(sa + S);               // [S] alpha exponent + row exponent of A[l, m)
    float *sf = (float *)(sc + S);           // [S] fast-pass row factors alpha_l(q) 2^(rho(q) - R)
    float *sz = sf + S;                      // [S] 1 where alpha_l(q) > 0
    int *pe = (int *)(sz + S);               // [QS * CB] partial max exponents (exact form)
    float *ps = (float *)(pe + QS * CB);     // [QS * CB] partial sums (exact form)
    // (the fast pass uses [pe, pe + 8 kThreads) for its partial sums first)
    __shared__ int red[kWarps];
    __shared__ int need_exact;
    const size_t lnode = (size_t)b * a.nc + 2 * j;
    const size_t bl = ((size_t)b * (L + 1) + l) * S, bmid = ((size_t)b * (L + 1) + m) * S;
    const int32_t *rho = a.rho + lnode * S, *rmx = a.rmax + lnode * S;
    // R: the exponent of the largest term any row can give (row maxima as bit patterns)
    int w = FA_INT_NONE;
    for (int q = threadIdx.x; q < S; q += kThreads) {
        const float x = a.am[bl + q];
        const int e = a.ae[bl + q] + rho[q], rb = rmx[q];
        sa[q] = x;
        sc[q] = e;
        if (x > 0.0f && rb > 0) w = max(w, e + fa_exponent(x) + max(-126, fa_exponent(__int_as_float(rb))));
    }
    if (threadIdx.x == 0) need_exact = 0;
    const int R = fa_block_max_int(w, red);
    if (a.fflag && a.fflag[lnode]) {
        // a functional span (committed positions of a DFA): alpha_m(d) is the sum of alpha_l(s)
        // over the states s its function maps to d, each term with its own exponent -- the
        // largest exponent first, then the sum scaled by it; the span is not read
        int *fm = reinterpret_cast<int *>(sf);
        for (int q = threadIdx.x; q < S; q += kThreads) fm[q] = a.fmap[lnode * S + q];
        __syncthreads();
        if (threadIdx.x < CB) {
            const int d = cbk * CB + threadIdx.x;
            if (d < S) {
                int E = FA_INT_NONE;
                for (int q = 0; q < S; ++q)
                    if (fm[q] == d && sa[q] > 0.0f) E = max(E, sc[q] + fa_exponent(sa[q]));
                float sum = 0.0f;
                if (E != FA_INT_NONE)
                    for (int q = 0; q < S; ++q)
                        if (fm[q] == d && sa[q] > 0.0f) sum += fa_mul_pow2(sa[q], sc[q] - E);
                float mo = 0.0f;
                int eo = 0;
                if (sum > 0.0f) { fa_split(sum, mo, eo); eo += E; }
                a.am[bmid + d] = mo;
                a.ae[bmid + d] = eo;
            }
        }
        return;
    }
    for (int q = threadIdx.x; q < S; q += kThreads) {
        sf[q] = (sa[q] > 0.0f && R != FA_INT_NONE) ? fa_mul_pow2(sa[q], sc[q] - R) : 0.0f;
        sz[q] = sa[q] > 0.0f ? 1.0f : 0.0f;
    }
    __syncthreads();
    const int c = threadIdx.x % CB, qs = threadIdx.x / CB;
    const int col = cbk * CB + c;
    const float *A = a.mant + lnode * (size_t)S * S;
    constexpr int U = 16;  // loads issued together
    // fast pass partial sums: [nsplit][CB] each (sums, then the exact-zero sums)
    float *fs = reinterpret_cast<float *>(pe), *fz = fs + kThreads * 4;
    int nsplit = QS;
    if (a.vec4 && CB == 64) {
        // |S| % 4 == 0: 16 four-column groups x 16 row splits, 16-byte loads
        nsplit = kThreads / 16;
        const int c4 = threadIdx.x & 15, rs = threadIdx.x >> 4, col4 = cbk * CB + 4 * c4;
        float4 sm4 = make_float4(0.f, 0.f, 0.f, 0.f), sz4 = make_float4(0.f, 0.f, 0.f, 0.f);
        constexpr int U4 = 8;
        if (col4 < S)
            for (int q0 = rs; q0 < S; q0 += U4 * 16) {
                float4 v[U4];
#pragma unroll
                for (int u = 0; u < U4; ++u) {
                    const int q = q0 + 16 * u;
                    v[u] = q < S ? __ldg(reinterpret_cast<const float4 *>(A + (size_t)q * S + col4)) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < U4; ++u) {
                    const int q = min(q0 + 16 * u, S - 1);
                    const float f = sf[q], z = sz[q];
                    sm4.x = fmaf(f, v[u].x, sm4.x); sm4.y = fmaf(f, v[u].y, sm4.y);
                    sm4.z = fmaf(f, v[u].z, sm4.z); sm4.w = fmaf(f, v[u].w, sm4.w);
                    sz4.x = fmaf(z, v[u].x, sz4.x); sz4.y = fmaf(z, v[u].y, sz4.y);
                    sz4.z = fmaf(z, v[u].z, sz4.z); sz4.w = fmaf(z, v[u].w, sz4.w);
                }
            }
        *reinterpret_cast<float4 *>(fs + rs * CB + 4 * c4) = sm4;
        *reinterpret_cast<float4 *>(fz + rs * CB + 4 * c4) = sz4;
    } else {
        float sum = 0.0f, sum1 = 0.0f;
        if (col < S)
            for (int q0 = qs; q0 < S; q0 += U * QS) {
                float v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int q = q0 + u * QS;
                    v[u] = q < S ? __ldg(A + (size_t)q * S + col) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int q = min(q0 + u * QS, S - 1);
                    sum = fmaf(sf[q], v[u], sum);
                    sum1 = fmaf(sz[q], v[u], sum1);
                }
            }
        fs[qs * CB + c] = sum;
        fz[qs * CB + c] = sum1;
    }
    __syncthreads();
    bool exact_col = false;
    if (qs == 0 && col < S) {
        float tot = 0.0f, tot1 = 0.0f;
        for (int t = 0; t < nsplit; ++t) { tot += fs[t * CB + c]; tot1 += fz[t * CB + c]; }
        if (!(tot1 > 0.0f)) {
            a.am[bmid + col] = 0.0f;
            a.ae[bmid + col] = 0;
        } else if (tot >= kMsgFastMin && tot <= 3.0e38f) {
            float mo;
            int eo;
            fa_split(tot, mo, eo);
            a.am[bmid + col] = mo;
            a.ae[bmid + col] = eo + R;
        } else {
            exact_col = true;
            need_exact = 1;
        }
    }
    __syncthreads();
    if (!need_exact) return;
    // the exact form for the block's columns (written only where the fast pass gave up)
    int e = FA_INT_NONE;
    if (col < S)
        for (int q0 = qs; q0 < S; q0 += U * QS) {
            float v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = q0 + u * QS;
                v[u] = q < S ? __ldg(A + (size_t)q * S + col) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = q0 + u * QS;
                if (v[u] > 0.0f && q < S && sa[q] > 0.0f) e = max(e, sc[q] + fa_exponent(v[u]));
            }
        }
    pe[qs * CB + c] = e;
    __syncthreads();
    int E = FA_INT_NONE;
    for (int t = 0; t < QS; ++t) E = max(E, pe[t * CB + c]);
    float esum = 0.0f;
    if (col < S && E != FA_INT_NONE)
        for (int q0 = qs; q0 < S; q0 += U * QS) {
            float v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = q0 + u * QS;
                v[u] = q < S ? __ldg(A + (size_t)q * S + col) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = q0 + u * QS;
                if (v[u] > 0.0f && q < S && sa[q] > 0.0f) {
                    float mv;
                    int ev;
                    fa_split(v[u], mv, ev);
                    esum += sa[q] * mv * fa_pow2(sc[q] + ev - E);
                }
            }
        }
    ps[qs * CB + c] = esum;
    __syncthreads();
    if (exact_col) {
        float tot = 0.0f;
        for (int t = 0; t < QS; ++t) tot += ps[t * CB + c];
        float mo = 0.0f;
        int eo = 0;
        if (tot > 0.0f) { fa_split(tot, mo, eo); eo += E; }
        a.am[bmid + col] = mo;
        a.ae[bmid + col] = eo;
    }
}

__device__ void topdown_beta(const TopdownArgs &a, int blk, float *sm) {
    const int S = a.S, L = a.L, k = a.k;
    const int RB = a.beta_rows;
    const int nrbk = (S + RB - 1) / RB;
    const int rbk = blk % nrbk;
    const long bj = blk / nrbk;
    const int j = (int)(bj % a.np), b = (int)(bj / a.np);
    const int l = j << (k + 1), m = l + (1 << k);
    if (m >= L) return;
    const int r = min(l + (1 << (k + 1)), L);
    float *sb = sm;                  // [S] mantissas of beta_r
    int *se = (int *)(sb + S);       // [S] their exponents
    float *sg = (float *)(se + S);   // [S] fast-pass factors beta_r(q) 2^-R
    float *sz = sg + S;              // [S] 1 where beta_r(q) > 0
    __shared__ int red[kWarps];
    const size_t br = ((size_t)b * (L + 1) + r) * S, bmid = ((size_t)b * (L + 1) + m) * S;
    int w = FA_INT_NONE;
    for (int q = threadIdx.x; q < S; q += kThreads) {
        const float x = a.bm[br + q];
        const int e = a.be[br + q];
        sb[q] = x;
        se[q] = e;
        if (x > 0.0f) w = max(w, e + fa_exponent(x));
    }
    const int R = fa_block_max_int(w, red);
    for (int q = threadIdx.x; q < S; q += kThreads) {
        sg[q] = (sb[q] > 0.0f && R != FA_INT_NONE) ? fa_mul_pow2(sb[q], se[q] - R) : 0.0f;
        sz[q] = sb[q] > 0.0f ? 1.0f : 0.0f;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const size_t rnode_f = (size_t)b * a.nc + 2 * j + 1;
    if (a.fflag && a.fflag[rnode_f]) {
        // a functional span: beta_m(s) = beta_r(f(s)) (row exponents 0); the span is not read
        for (int row = rbk * RB + threadIdx.x; row < min(S, (rbk + 1) * RB); row += kThreads) {
            const int t = a.fmap[rnode_f * S + row];
            a.bm[bmid + row] = t >= 0 ? sb[t] : 0.0f;
            a.be[bmid + row] = t >= 0 ? se[t] : 0;
        }
        return;
    }
    // warp w takes rows rbk * RB + w, + kWarps, ... of the block's RB rows
    for (int row = rbk * RB + (threadIdx.x >> 5); row < min(S, (rbk + 1) * RB); row += kWarps) {
        const size_t rnode = (size_t)b * a.nc + 2 * j + 1;
        const float *Rrow = a.mant + rnode * (size_t)S * S + (size_t)row * S;
        // the row's entries scaled by its largest (their exponents then stay near 0)
        const int rb = a.rmax[rnode * S + row];
        const int er = min(126, max(-126, fa_exponent(__int_as_float(rb))));
        const float rs = __int_as_float((127 - er) << 23);   // 2^-er
        float sum = 0.0f, sum1 = 0.0f;
        if (rb > 0 && a.vec4) {
            constexpr int U4 = 4;  // 16-byte loads issued together
            for (int q0 = 4 * lane; q0 < S; q0 += 128 * U4) {
                float4 v[U4];
    #pragma unroll
                for (int u = 0; u < U4; ++u) {
                    const int q = q0 + 128 * u;
                    v[u] = q < S ? __ldg(reinterpret_cast<const float4 *>(Rrow + q)) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
    #pragma unroll
                for (int u = 0; u < U4; ++u) {
                    const int q = min(q0 + 128 * u, S - 4);
                    const float4 g = *reinterpret_cast<const float4 *>(sg + q), z = *reinterpret_cast<const float4 *>(sz + q);
                    sum = fmaf(v[u].x * rs, g.x, sum); sum = fmaf(v[u].y * rs, g.y, sum);
                    sum = fmaf(v[u].z * rs, g.z, sum); sum = fmaf(v[u].w * rs, g.w, sum);
                    sum1 = fmaf(v[u].x, z.x, sum1); sum1 = fmaf(v[u].y, z.y, sum1);
                    sum1 = fmaf(v[u].z, z.z, sum1); sum1 = fmaf(v[u].w, z.w, sum1);
                }
            }
        } else if (rb > 0) {
            constexpr int U = 8;
            for (int q0 = lane; q0 < S; q0 += 32 * U) {
                float v[U];
    #pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int q = q0 + 32 * u;
                    v[u] = q < S ? __ldg(Rrow + q) : 0.0f;
                }
    #pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int q = min(q0 + 32 * u, S - 1);
                    sum = fmaf(v[u] * rs, sg[q], sum);
                    sum1 = fmaf(v[u], sz[q], sum1);
                }
            }
        }
        sum = fa_warp_sum(sum);
        sum1 = fa_warp_sum(sum1);
        if (!(sum1 > 0.0f)) {
            if (lane == 0) { a.bm[bmid + row] = 0.0f; a.be[bmid + row] = 0; }
            continue;
        }
        if (sum >= kMsgFastMin && sum <= 3.0e38f) {
            if (lane == 0) {
                float mo;
                int eo;
                fa_split(sum, mo, eo);
                a.bm[bmid + row] = mo;
                a.be[bmid + row] = eo + R + er + a.rho[rnode * S + row];
            }
            continue;
        }
        // the exact form for this row
        int e = FA_INT_NONE;
        for (int q = lane; q < S; q += 32) {
            const float v = Rrow[q];
            if (v > 0.0f && sb[q] > 0.0f) e = max(e, se[q] + fa_exponent(v));
        }
        e = fa_warp_max_int(e);
        float esum = 0.0f;
        if (e != FA_INT_NONE)
            for (int q = lane; q < S; q += 32) {
                const float v = Rrow[q];
                if (v > 0.0f && sb[q] > 0.0f) {
                    float mv;
                    int ev;
                    fa_split(v, mv, ev);
                    esum += sb[q] * mv * fa_pow2(se[q] + ev - e);
                }
            }
        esum = fa_warp_sum(esum);
        if (lane == 0) {
            float mo = 0.0f;
            int eo = 0;
            if (esum > 0.0f) { fa_split(esum, mo, eo); eo += e + a.rho[rnode * S + row]; }
            a.bm[bmid + row] = mo;
            a.be[bmid + row] = eo;
        }
    }
}

__global__ void __launch_bounds__(kThreads) k_topdown(TopdownArgs a) {
    extern __shared__ float smem_td[];
    const int blk = blockIdx.x;
    if (blk < a.nA) topdown_alpha(a, blk, smem_td);
    else if (blk < a.nA + a.nB) topdown_beta(a, blk - a.nA, smem_td);
    else topdown_midpoint(a, blk - a.nA - a.nB);
}

// ----------------------------------------------------------------------------- 5. leaves

// Token at each position: committed positions echo their token; a masked position draws
// v ~ w_t(v) over the tokens of the edges z_{t-1} -> z_t (paperfeed.app: all tokens emit in
// parallel at the leaves), then its constrained marginal
//   p(x_t = v) = w_t(v) sum_{e carries v} alpha_{t-1}(src e) beta_t(dst e) / D_t
// (papernotes.org key design 3), D_t = alpha_{t-1}^T M_t beta_t the local normaliser (equal
// to Z, and sharing alpha and beta with the numerator, so their errors cancel).
//
// One block per position.  The three reductions of a masked position (the normaliser over
// the cells of M_t, the draw over the cell's tokens, the numerator over the token's
// incidences) are spread over all threads, so that a position costs a few dependent memory
// round trips instead of hundreds.
constexpr int kLeafThreads = 256;
constexpr int kLeafWarps = kLeafThreads / 32;
constexpr int kLeafStageStates = 2048;  // alpha/beta rows staged in shared memory up to this |S|

struct LeafShared {
    float wm[kLeafWarps];
    int we[kLeafWarps];
    float wsum[kLeafWarps];
    float xm;
    int xe;
    int ra, rb;   // the scales of the normaliser's fast pass
    int cell, pick_thread, last_thread, v, ok;
    int last;
};

// Merge every thread's accumulator; the result lands in sh.xm / sh.xe (mantissa, exponent).
__device__ void block_xacc(fa_xacc x, LeafShared &sh) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    x.warp_reduce();
    if (lane == 0) { sh.wm[w] = x.acc; sh.we[w] = x.E; }
    __syncthreads();
    if (threadIdx.x == 0) {
        fa_xacc y;
        y.init();
        for (int i = 0; i < kLeafWarps; ++i) y.merge(sh.wm[i], sh.we[i]);
        y.normalised(sh.xm, sh.xe);
    }
    __syncthreads();
}

// Inclusive scan of one value per thread over the block (thread order); returns this
// thread's inclusive prefix and the block total in *total.
__device__ float block_scan(float x, LeafShared &sh, float *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sh.wsum[w] = incl;
    __syncthreads();
    float before = 0.0f, all = 0.0f;
    for (int i = 0; i < kLeafWarps; ++i) {
        if (i < w) before += sh.wsum[i];
        all += sh.wsum[i];
    }
    __syncthreads();
    *total = all;
    return before + incl;
}

__device__ bool leaf_position(const DevFA &fa, int b, int t, int L, const float *__restrict__ probs,
                              const int32_t *__restrict__ committed, uint64_t seed, uint64_t offset,
                              const int32_t *__restrict__ z, const float *__restrict__ am,
                              const int32_t *__restrict__ ae, const float *__restrict__ bm,
                              const int32_t *__restrict__ be, int32_t *tokens, float *marg, int32_t *status,
                              const float *__restrict__ leaf, LeafShared &sh, float *stage, int conf_mode,
                              float *conf, float *den_mo, int32_t *den_eo) {
    const int tid = threadIdx.x;
    const size_t pos = (size_t)b * L + t;
    const int c = committed[pos];
    if (c >= 0) {
        if (tid == 0) { tokens[pos] = c; marg[pos] = 1.0f; }
        return true;
    }
    // one read of the status for the whole block (another block of the sequence may change it)
    if (tid == 0) { sh.cell = -1; sh.pick_thread = INT_MAX; sh.last_thread = -1; sh.v = -1; sh.ok = status[b] == FA_ROW_OK; }
    __syncthreads();
    if (!sh.ok) {
        if (tid == 0) { tokens[pos] = -1; marg[pos] = 0.0f; }
        return true;
    }
    const int S = fa.S;
    const int32_t *zb = z + (size_t)b * (L + 1);
    const int zp = zb[t], zn = zb[t + 1];
    const size_t ba = ((size_t)b * (L + 1) + t) * S, bb = ((size_t)b * (L + 1) + t + 1) * S;
    // the cell z_{t-1} -> z_t (one pass over the source's cells) and the two messages
    const float *a_m = am + ba, *b_m = bm + bb;
    const int32_t *a_e = ae + ba, *b_e = be + bb;
    // staged: the messages, and for the normaliser's fast pass the messages scaled by one
    // power of two each (alpha_{t-1}(s) 2^-Ra, beta_t(d) 2^-Rb, at most 2)
    float *sa2 = nullptr, *sb2 = nullptr;
    if (stage) {
        float *sam = stage, *sbm = stage + S;
        int32_t *sae = (int32_t *)(stage + 2 * S), *sbe = (int32_t *)(stage + 3 * S);
        sa2 = stage + 4 * S;
        sb2 = stage + 5 * S;
        int ra = FA_INT_NONE, rb = FA_INT_NONE;
        for (int s = tid; s < S; s += kLeafThreads) {
            const float x = a_m[s], y = b_m[s];
            const int ex = a_e[s], ey = b_e[s];
            sam[s] = x; sae[s] = ex; sbm[s] = y; sbe[s] = ey;
            if (x > 0.0f) ra = max(ra, ex + fa_exponent(x));
            if (y > 0.0f) rb = max(rb, ey + fa_exponent(y));
        }
        ra = fa_warp_max_int(ra);
        rb = fa_warp_max_int(rb);
        if ((tid & 31) == 0) { sh.we[tid >> 5] = ra; reinterpret_cast<int *>(sh.wsum)[tid >> 5] = rb; }
        __syncthreads();
        if (tid == 0) {
            int A = FA_INT_NONE, Bv = FA_INT_NONE;
            for (int i = 0; i < kLeafWarps; ++i) { A = max(A, sh.we[i]); Bv = max(Bv, reinterpret_cast<int *>(sh.wsum)[i]); }
            sh.ra = A;
            sh.rb = Bv;
        }
        __syncthreads();
        const int RA = sh.ra, RB = sh.rb;
        for (int s = tid; s < S; s += kLeafThreads) {
            sa2[s] = (sam[s] > 0.0f && RA != FA_INT_NONE) ? fa_mul_pow2(sam[s], sae[s] - RA) : 0.0f;
            sb2[s] = (sbm[s] > 0.0f && RB != FA_INT_NONE) ? fa_mul_pow2(sbm[s], sbe[s] - RB) : 0.0f;
        }
        a_m = sam; b_m = sbm; a_e = sae; b_e = sbe;
    }
    __syncthreads();
    for (int i = fa.row_cell_off[zp] + tid; i < fa.row_cell_off[zp + 1]; i += kLeafThreads)
        if (fa.cell_dst[i] == zn) sh.cell = i;  // at most one cell per (src, dst)
    __syncthreads();
    const int cell = sh.cell;

    // the draw, first half: this thread's share of the cell's tokens (i = tid, tid + T, ...),
    // taken in thread order for the inverse CDF
    const float *prow = probs + pos * (size_t)fa.V;
    int64_t a0 = 0;
    int n = 0;
    if (cell >= 0) { a0 = fa.cell_off[cell]; n = (int)(fa.cell_off[cell + 1] - a0); }
    float own = 0.0f;
    for (int i = tid; i < n; i += kLeafThreads) own += __ldg(prow + fa.cell_tok[a0 + i]);

    // the normaliser over the cells of M_t (zero everywhere else): through the cell lists, or,
    // when the cells cover a quarter of the (s, s') pairs or more, over M_t read whole as
    // float4s in address order (coalesced, no index traffic).  Thread tid takes the float4s
    // tid, tid + T, ...; its (row, column) advances by a fixed step, without divisions.
    const float *Mt = leaf + pos * (size_t)S * S;
    fa_xacc dx;
    dx.init();
    auto term = [&](float a, int ea, float mv, int d) {
        const float bv = b_m[d];
        if (bv > 0.0f && mv > 0.0f) {
            float mm;
            int em;
            fa_split(mv, mm, em);
            dx.add(a * bv * mm, ea + b_e[d] + em);
        }
    };
    const bool dense = (long)fa.n_cells * 4 >= (long)S * S && (S & 3) == 0 && (reinterpret_cast<uintptr_t>(Mt) & 15) == 0;
    // fast pass of a dense normaliser: plain fp32 sum of sa2(s) M_t(s, d) sb2(d) (terms at most
    // 4), kept when it is at least 2^-60 (the terms lost below the fp32 normal range then add
    // under 2^-57 of it); otherwise the exact form below
    bool exact_den = true;
    float den_m = 0.0f;
    int den_e = 0;
    if (dense && sa2) {
        const int S4 = S >> 2, n4 = S * S4;
        const int dr = kLeafThreads / S4, dc = kLeafThreads % S4;
        int r = tid / S4, c4 = tid % S4;
        const float4 *M4 = reinterpret_cast<const float4 *>(Mt);
        float fsum = 0.0f;
#pragma unroll 8
        for (int i = tid; i < n4; i += kLeafThreads) {
            const float4 mv = __ldg(M4 + i);
            const float4 bv = *reinterpret_cast<const float4 *>(sb2 + 4 * c4);
            fsum = fmaf(sa2[r], mv.x * bv.x + mv.y * bv.y + mv.z * bv.z + mv.w * bv.w, fsum);
            r += dr;
            c4 += dc;
            if (c4 >= S4) { c4 -= S4; ++r; }
        }
        fsum = fa_warp_sum(fsum);
        __syncthreads();   // the scale reductions above are read
        if ((tid & 31) == 0) sh.wsum[tid >> 5] = fsum;
        __syncthreads();
        float D = 0.0f;
        for (int i = 0; i < kLeafWarps; ++i) D += sh.wsum[i];
        __syncthreads();
        if (D >= 8.6736174e-19f && D <= 3.0e38f) {
            exact_den = false;
            fa_split(D, den_m, den_e);
            den_e += sh.ra + sh.rb;
        }
    }
    if (!exact_den) {
    } else if (dense) {
        const int S4 = S >> 2, n4 = S * S4;
        const int dr = kLeafThreads / S4, dc = kLeafThreads % S4;
        int r = tid / S4, c4 = tid % S4;
        const float4 *M4 = reinterpret_cast<const float4 *>(Mt);
#pragma unroll 4
        for (int i = tid; i < n4; i += kLeafThreads) {
            const float4 mv = __ldg(M4 + i);
            const float a = a_m[r];
            if (a > 0.0f) {
                const int ea = a_e[r], d = 4 * c4;
                term(a, ea, mv.x, d);
                term(a, ea, mv.y, d + 1);
                term(a, ea, mv.z, d + 2);
                term(a, ea, mv.w, d + 3);
            }
            r += dr;
            c4 += dc;
            if (c4 >= S4) { c4 -= S4; ++r; }
        }
    } else {
#pragma unroll 4
        for (int q = tid; q < fa.n_cells; q += kLeafThreads) {
            const int s = fa.cell_src[q], d = fa.cell_dst[q];
            const float a = a_m[s], bv = b_m[d], mv = __ldg(Mt + (size_t)s * S + d);
            if (a > 0.0f && bv > 0.0f && mv > 0.0f) {
                float mm;
                int em;
                fa_split(mv, mm, em);
                dx.add(a * bv * mm, a_e[s] + b_e[d] + em);
            }
        }
    }

    float total;
    const float incl = block_scan(own, sh, &total);
    if (exact_den) {
        block_xacc(dx, sh);
        den_m = sh.xm;
        den_e = sh.xe;
    }
    if (!(total > 0.0f)) {
        if (tid == 0) { status[b] = FA_ROW_UNDERFLOW; tokens[pos] = -1; marg[pos] = 0.0f; }
        return false;
    }
    const float u = fa_uniform(seed, offset, (uint32_t)t, (uint32_t)b, FA_RNG_LEAF);
    const float target = u * total;
    if (own > 0.0f) {
        if (incl > target) atomicMin(&sh.pick_thread, tid);
        atomicMax(&sh.last_thread, tid);
    }
    __syncthreads();
    // the draw, second half: the first thread whose prefix passes the target walks its share
    // (a rounding shortfall falls back to the last positive token)
    const int who = sh.pick_thread != INT_MAX ? sh.pick_thread : sh.last_thread;
    if (tid == who) {
        float run = incl - own;
        int pick = -1, lastpos = -1;
        for (int i = tid; i < n; i += kLeafThreads) {
            const float w = __ldg(prow + fa.cell_tok[a0 + i]);
            if (w > 0.0f) {
                lastpos = i;
                run += w;
                if (run > target) { pick = i; break; }
            }
        }
        if (pick < 0) pick = lastpos;
        sh.v = pick >= 0 ? fa.cell_tok[a0 + pick] : -1;
    }
    __syncthreads();
    const int v = sh.v;
    if (v < 0) {
        if (tid == 0) { status[b] = FA_ROW_UNDERFLOW; tokens[pos] = -1; marg[pos] = 0.0f; }
        return false;
    }
    // numerator: sum over the edges carrying v of alpha_{t-1}(src) beta_t(dst)
    fa_xacc x;
    x.init();
    for (int64_t j = fa.tok_off[v] + tid; j < fa.tok_off[v + 1]; j += kLeafThreads) {
        const int e = fa.tok_edges[j];
        const int s = fa.edge_src[e], d = fa.edge_dst[e];
        const float a = a_m[s], bv = b_m[d];
        if (a > 0.0f && bv > 0.0f) x.add(a * bv, a_e[s] + b_e[d]);
    }
    block_xacc(x, sh);
    if (tid == 0) {
        tokens[pos] = v;
        double mval = 0.0;
        if (sh.xm > 0.0f && den_m > 0.0f)
            mval = ldexp((double)__ldg(prow + v) * (double)sh.xm / (double)den_m, sh.xe - den_e);
        marg[pos] = (float)mval;
        den_mo[pos] = den_m;
        den_eo[pos] = den_e;
        // the commit's ranking score (the entropy score is written by k_tm_finish)
        if (conf_mode == FA_CONF_MARGINAL) conf[pos] = (float)mval;
        else if (conf_mode == FA_CONF_UNCONSTRAINED) conf[pos] = __ldg(prow + v);
    }
    return true;
}

__device__ void topk_row(int b, int L, int k, int lo, int hi, float *marg, const float *conf,
                         const int32_t *__restrict__ committed, const int32_t *status, int32_t *out, int32_t *tokens,
                         unsigned long long *skey);

// Leaves, then the commit: every block takes its sequence's ticket after its position is
// written; the last block of a sequence sees all of its marginals and runs its top-k.
__global__ void __launch_bounds__(kLeafThreads, 1) k_leaf_commit(DevFA fa, int B, int L, const float *__restrict__ probs,
                                                            const int32_t *__restrict__ committed, uint64_t seed,
                                                            uint64_t offset, const int32_t *__restrict__ z,
                                                            const float *__restrict__ am,
                                                            const int32_t *__restrict__ ae,
                                                            const float *__restrict__ bm,
                                                            const int32_t *__restrict__ be, int32_t *tokens,
                                                            float *marg, int32_t *status, int k, int lo, int hi,
                                                            int32_t *commit_idx, unsigned long long *keys,
                                                            int32_t *done, const float *__restrict__ leaf,
                                                            int conf_mode, float *conf, float *den_mo,
                                                            int32_t *den_eo, int do_commit) {
    extern __shared__ float leaf_stage[];
    __shared__ LeafShared sh;
    const int b = (int)(blockIdx.x / (unsigned)L), t = (int)(blockIdx.x % (unsigned)L);
    leaf_position(fa, b, t, L, probs, committed, seed, offset, z, am, ae, bm, be, tokens, marg, status, leaf, sh,
                  fa.S <= kLeafStageStates ? leaf_stage : nullptr, conf_mode, conf, den_mo, den_eo);
    if (!do_commit) return;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        sh.last = atomicAdd(done + b, 1) == L - 1;
    }
    __syncthreads();
    if (!sh.last) return;
    __threadfence();
    topk_row(b, L, k, lo, hi, marg, conf, committed, status, commit_idx, tokens, keys + (size_t)b * L);
}

// ----------------------------------------------------------------------------- 5b. all-token marginals

// Full constrained marginal of a masked position t (papernotes.org key design 3):
//   p(x_t = v) = w_t(v) sum_{e carries v} alpha_{t-1}(src e) beta_t(dst e) / D_t,
// D_t = alpha_{t-1}^T M_t beta_t the local normaliser the leaves computed (the same sum taken
// over the cells), and the entropy H_t = -sum_v p ln p.  One block per (position, chunk of
// `chunk_tokens` tokens, a multiple of 32); token v is summed by one thread over its
// incidences (interleaved by groups of 32 tokens, see fa_automaton), the block's sum of
// p ln p lands in a per-chunk slot, and k_tm_finish adds the slots in chunk order, so the
// result is deterministic.
constexpr int kTmThreads = 256;
constexpr int kTmWarps = kTmThreads / 32;

__global__ void __launch_bounds__(kTmThreads) k_tm_partial(DevFA fa, int L, int n_chunks, int chunk_tokens,
                                                          const float *__restrict__ probs,
                                                          const int32_t *__restrict__ committed,
                                                          const int32_t *__restrict__ status,
                                                          const float *__restrict__ am, const int32_t *__restrict__ ae,
                                                          const float *__restrict__ bm, const int32_t *__restrict__ be,
                                                          const float *__restrict__ den_m,
                                                          const int32_t *__restrict__ den_e, float *marg_all,
                                                          double *part) {
    // shared memory: fast form [S + 1] alpha', [S + 1] beta' (fp32, scaled, zero at index S);
    // exact form [S + 1] + [S + 1] (mantissa, exponent bits) pairs
    extern __shared__ float2 tm_s[];
    __shared__ double red[kTmWarps];
    __shared__ int ired[2 * kTmWarps];
    const int S = fa.S, V = fa.V;
    const size_t pos = blockIdx.x / (unsigned)n_chunks;
    const int chunk = (int)(blockIdx.x % (unsigned)n_chunks);
    const int b = (int)(pos / (size_t)L), t = (int)(pos % (size_t)L);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v0 = chunk * chunk_tokens, v1 = min(V, v0 + chunk_tokens);
    const int c = committed[pos];
    float *out = marg_all ? marg_all + pos * (size_t)V : nullptr;
    const float dm = (c >= 0 || status[b] != FA_ROW_OK) ? 0.0f : den_m[pos];
    if (!(dm > 0.0f)) {
        if (out)
            for (int v = v0 + tid; v < v1; v += kTmThreads) out[v] = (c >= 0 && v == c) ? 1.0f : 0.0f;
        if (tid == 0) part[blockIdx.x] = 0.0;
        return;
    }
    const int E = den_e[pos];
    const float inv = 1.0f / dm;
    const size_t ba = ((size_t)b * (L + 1) + t) * S, bb = ba + S;
    // the fast form scales alpha and beta by one power of two each (at most 2 after it), and a
    // token's sum by 2^X, X = Ea + Eb - E; it is taken when X <= 60, so the products lost
    // below the fp32 normal range weigh under |S| 2^-66 in a marginal
    int ea = FA_INT_NONE, eb = FA_INT_NONE;
    for (int s = tid; s < S; s += kTmThreads) {
        const float x = am[ba + s], y = bm[bb + s];
        if (x > 0.0f) ea = max(ea, ae[ba + s] + fa_exponent(x));
        if (y > 0.0f) eb = max(eb, be[bb + s] + fa_exponent(y));
    }
    ea = fa_warp_max_int(ea);
    eb = fa_warp_max_int(eb);
    if (lane == 0) { ired[warp] = ea; ired[kTmWarps + warp] = eb; }
    __syncthreads();
    int Ea = FA_INT_NONE, Eb = FA_INT_NONE;
    for (int w = 0; w < kTmWarps; ++w) { Ea = max(Ea, ired[w]); Eb = max(Eb, ired[kTmWarps + w]); }
    const bool fast = Ea != FA_INT_NONE && Eb != FA_INT_NONE && Ea + Eb - E <= 60;
    const int X = fast ? Ea + Eb - E : 0;
    float *fa1 = reinterpret_cast<float *>(tm_s), *fb1 = fa1 + S + 1;
    float2 *sa = tm_s, *sb = tm_s + S + 1;
    if (fast) {
        for (int s = tid; s <= S; s += kTmThreads) {
            const float x = s < S ? am[ba + s] : 0.0f, y = s < S ? bm[bb + s] : 0.0f;
            fa1[s] = x > 0.0f ? fa_mul_pow2(x, ae[ba + s] - Ea) : 0.0f;
            fb1[s] = y > 0.0f ? fa_mul_pow2(y, be[bb + s] - Eb) : 0.0f;
        }
    } else {
        for (int s = tid; s <= S; s += kTmThreads) {
            sa[s] = s < S ? make_float2(am[ba + s], __int_as_float(ae[ba + s])) : make_float2(0.0f, 0.0f);
            sb[s] = s < S ? make_float2(bm[bb + s], __int_as_float(be[bb + s])) : make_float2(0.0f, 0.0f);
        }
    }
    __syncthreads();
    const uint32_t pad = ((uint32_t)S << 16) | (uint32_t)S;   // the streams' padding: index S (zero)
    const float *prow = probs + pos * (size_t)V;
    float sl = 0.0f, cl = 0.0f;  // compensated sum of p ln p
    // the block's range [v0, v1) is in the tok_perm order; warp w takes the token groups
    // g0 + w, g0 + w + kTmWarps, ...; lane l the token tok_perm[32 g + l], reading row k of
    // the group's interleaved incidences (one 128-byte line per warp)
    for (int g = v0 / 32 + warp; g < (v1 + 31) / 32; g += kTmWarps) {
        const int i = 32 * g + lane;
        const int v = i < v1 ? __ldg(fa.tok_perm + i) : 0;
        const float w = i < v1 ? __ldg(prow + v) : 0.0f;
        const int64_t r0 = fa.tok_goff[g], nr = fa.tok_goff[g + 1] - r0;
        const uint32_t *col = fa.tok_sd + (size_t)r0 * 32 + lane;
        float acc = 0.0f;
        if (fast) {
            // whole steps of eight rows (their loads in flight before any is used), then the rest
            const uint32_t *p = col;
            int64_t k0 = 0;
            for (; k0 + 8 <= nr; k0 += 8, p += 256) {
                uint32_t sdv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) sdv[u] = __ldg(p + 32 * u);
#pragma unroll
                for (int u = 0; u < 8; ++u) acc = fmaf(fa1[sdv[u] >> 16], fb1[sdv[u] & 0xffffu], acc);
            }
            for (; k0 < nr; ++k0, p += 32) {
                const uint32_t sd = __ldg(p);
                acc = fmaf(fa1[sd >> 16], fb1[sd & 0xffffu], acc);
            }
        } else {
            for (int64_t k0 = 0; k0 < nr; k0 += 8) {
                uint32_t sdv[8];  // eight rows' loads in flight before any is used
#pragma unroll
                for (int u = 0; u < 8; ++u) sdv[u] = k0 + u < nr ? __ldg(col + (size_t)(k0 + u) * 32) : pad;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t sd = sdv[u];
                    const float2 a = sa[sd >> 16], bq = sb[sd & 0xffffu];
                    if (a.x > 0.0f && bq.x > 0.0f) acc += a.x * bq.x * fa_pow2(__float_as_int(a.y) + __float_as_int(bq.y) - E);
                }
            }
        }
        if (i >= v1) continue;
        const float pv = w > 0.0f ? w * fa_mul_pow2(acc, X) * inv : 0.0f;
        if (out) out[v] = pv;
        if (pv > 0.0f) {
            const float y = pv * logf(pv) - cl, tt = sl + y;
            cl = (tt - sl) - y;
            sl = tt;
        }
    }
    double dl = (double)sl - (double)cl;
#pragma unroll
    for (int o = 16; o; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
    if (lane == 0) red[warp] = dl;
    __syncthreads();
    if (tid == 0) {
        double tot = 0.0;
        for (int w = 0; w < kTmWarps; ++w) tot += red[w];
        part[blockIdx.x] = tot;
    }
}

// H_t = -(sum of the chunk slots, in chunk order); the commit score is -H_t.
__global__ void k_tm_finish(long n_pos, int n_chunks, const double *__restrict__ part, float *entropy, float *conf) {
    const long pos = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (pos >= n_pos) return;
    double tot = 0.0;
    for (int q = 0; q < n_chunks; ++q) tot += part[pos * n_chunks + q];
    const float H = (float)(tot == 0.0 ? 0.0 : -tot);
    if (entropy) entropy[pos] = H;
    if (conf) conf[pos] = -H;
}

// The commit of every sequence as its own block (when it must wait for the entropies).
__global__ void __launch_bounds__(kThreads) k_commit_rows(int L, int k, int lo, int hi, float *marg,
                                                        const float *conf, const int32_t *__restrict__ committed,
                                                        const int32_t *status, int32_t *commit_idx, int32_t *tokens,
                                                        unsigned long long *keys) {
    const int b = blockIdx.x;
    topk_row(b, L, k, lo, hi, marg, conf, committed, status, commit_idx, tokens, keys + (size_t)b * L);
}

// ----------------------------------------------------------------------------- chain variant

// The chain form of the same computation (paperfeed.app summary, "The scan trick": the O(L)
// chain that the tree shortens to O(log L) depth): forward messages alpha_t = alpha_{t-1} M_t
// for t = 1..L, then backward messages beta_{t-1} = M_t beta_t together with forward-filtering
// backward-sampling of the states, z_L ~ alpha_L restricted to F and
// z_{t-1} ~ alpha_{t-1}(s) M_t(s, z_t).  One block per sequence.  The vectors keep the tree
// messages' format (mantissa in [1, 2) and an exponent per state) and land in the same
// workspace arrays, so leaves, marginals and the commit are the tree path's kernels.  Every
// sum is one pass with a running exponent (fa_xacc).
constexpr int kChThreads = 512;
constexpr int kChWarps = kChThreads / 32;

__device__ __forceinline__ int chain_cb(int S) { return S >= 64 ? 64 : 32; }

// Shared memory: two (mantissa, exponent) vectors, and in the forward kernel the partials of
// the row splits (one mantissa and one exponent per thread).
size_t chain_smem(int S, bool forward) { return (size_t)S * 16 + (forward ? (size_t)kChThreads * 8 : 0); }

__global__ void __launch_bounds__(kChThreads) k_chain_forward(DevFA fa, int L, const float *__restrict__ leaf,
                                                             float *am, int32_t *ae) {
    extern __shared__ float ch_s[];
    const int S = fa.S, b = blockIdx.x, tid = threadIdx.x;
    float *va[2] = {ch_s, ch_s + S};
    int *ve[2] = {reinterpret_cast<int *>(ch_s + 2 * S), reinterpret_cast<int *>(ch_s + 3 * S)};
    const int CB = chain_cb(S), QS = kChThreads / CB;
    float *pm = ch_s + 4 * S;
    int *pe = reinterpret_cast<int *>(pm + kChThreads);
    const size_t base = (size_t)b * (L + 1) * S;
    for (int q = tid; q < S; q += kChThreads) {
        const float a0 = q == fa.start ? 1.0f : 0.0f;
        am[base + q] = a0; ae[base + q] = 0;
        va[0][q] = a0; ve[0][q] = 0;
    }
    __syncthreads();
    const int c = tid % CB, qs = tid / CB;
    for (int t = 1; t <= L; ++t) {
        const int in = (t - 1) & 1, out = t & 1;
        const float *M = leaf + ((size_t)b * L + (t - 1)) * (size_t)S * S;
        for (int c0 = 0; c0 < S; c0 += CB) {
            const int col = c0 + c;
            fa_xacc x;
            x.init();
            if (col < S)
                for (int q = qs; q < S; q += QS) {
                    const float a = va[in][q], v = __ldg(M + (size_t)q * S + col);
                    if (a > 0.0f && v > 0.0f) {
                        float mv;
                        int ev;
                        fa_split(v, mv, ev);
                        x.add(a * mv, ve[in][q] + ev);
                    }
                }
            pm[qs * CB + c] = x.acc;
            pe[qs * CB + c] = x.E;
            __syncthreads();
            if (qs == 0 && col < S) {
                fa_xacc y;
                y.init();
                for (int r = 0; r < QS; ++r) y.merge(pm[r * CB + c], pe[r * CB + c]);
                float mo;
                int eo;
                y.normalised(mo, eo);
                va[out][col] = mo; ve[out][col] = eo;
                am[base + (size_t)t * S + col] = mo; ae[base + (size_t)t * S + col] = eo;
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kChThreads) k_chain_backward(DevFA fa, int L, const float *__restrict__ leaf,
                                                              const float *__restrict__ am,
                                                              const int32_t *__restrict__ ae, float *bm, int32_t *be,
                                                              int32_t *z, uint64_t seed, uint64_t offset, double *logZ,
                                                              int32_t *status, float *zsum_ws, int32_t *zexp_ws) {
    extern __shared__ float ch_s[];
    __shared__ int zcur, alive;
    const int S = fa.S, b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *vb[2] = {ch_s, ch_s + S};
    int *vbe[2] = {reinterpret_cast<int *>(ch_s + 2 * S), reinterpret_cast<int *>(ch_s + 3 * S)};
    const size_t base = (size_t)b * (L + 1) * S;
    int32_t *zb = z + (size_t)b * (L + 1);
    for (int q = tid; q < S; q += kChThreads) {
        const float b0 = fa.accept_mask[q] ? 1.0f : 0.0f;
        bm[base + (size_t)L * S + q] = b0; be[base + (size_t)L * S + q] = 0;
        vb[L & 1][q] = b0; vbe[L & 1][q] = 0;
    }
    // the end state and logZ from alpha_L over the accepting states
    if (warp == 0) {
        const float *aL = am + base + (size_t)L * S;
        const int32_t *eL = ae + base + (size_t)L * S;
        int emax = FA_INT_NONE;
        for (int i = lane; i < fa.n_accept; i += 32) {
            const int f = fa.accept[i];
            if (aL[f] > 0.0f) emax = max(emax, eL[f]);
        }
        emax = fa_warp_max_int(emax);
        int pick = -1;
        float tot = 0.0f;
        if (emax != FA_INT_NONE) {
            auto w = [&](int i) { const int f = fa.accept[i]; return aL[f] > 0.0f ? aL[f] * fa_pow2(eL[f] - emax) : 0.0f; };
            const float u = fa_uniform(seed, offset, 0u, (uint32_t)b, FA_RNG_ROOT);
            pick = warp_categorical(fa.n_accept, u, w);
            for (int i = lane; i < fa.n_accept; i += 32) tot += w(i);
            tot = fa_warp_sum(tot);
        }
        if (lane == 0) {
            zb[0] = fa.start;
            if (pick < 0 || !(tot > 0.0f)) {
                status[b] = FA_ROW_EMPTY;
                logZ[b] = -INFINITY;
                zsum_ws[b] = 0.0f;
                zexp_ws[b] = 0;
                alive = 0;
            } else {
                status[b] = FA_ROW_OK;
                logZ[b] = (double)emax * 0.69314718055994530942 + log((double)tot);
                zsum_ws[b] = tot;
                zexp_ws[b] = emax;
                zcur = fa.accept[pick];
                zb[L] = zcur;
                alive = 1;
            }
        }
    }
    __syncthreads();
    if (!alive) {
        for (int t = tid; t <= L; t += kChThreads) zb[t] = fa.start;   // keep every state in range
        return;
    }
    for (int t = L; t >= 1; --t) {
        const int in = t & 1, out = (t - 1) & 1;
        const float *M = leaf + ((size_t)b * L + (t - 1)) * (size_t)S * S;
        // beta_{t-1}(s) = sum_d M_t(s, d) beta_t(d), one warp per row
        for (int r = warp; r < S; r += kChWarps) {
            fa_xacc x;
            x.init();
            for (int d = lane; d < S; d += 32) {
                const float v = __ldg(M + (size_t)r * S + d), bq = vb[in][d];
                if (v > 0.0f && bq > 0.0f) {
                    float mv;
                    int ev;
                    fa_split(v, mv, ev);
                    x.add(bq * mv, vbe[in][d] + ev);
                }
            }
            x.warp_reduce();
            if (lane == 0) {
                float mo;
                int eo;
                x.normalised(mo, eo);
                vb[out][r] = mo; vbe[out][r] = eo;
                bm[base + (size_t)(t - 1) * S + r] = mo; be[base + (size_t)(t - 1) * S + r] = eo;
            }
        }
        // z_{t-1} ~ alpha_{t-1}(s) M_t(s, z_t) (warp 0; the other warps' rows do not need it)
        if (warp == 0 && t > 1) {
            const int zt = zcur;
            const float *a = am + base + (size_t)(t - 1) * S;
            const int32_t *ea = ae + base + (size_t)(t - 1) * S;
            int emax = FA_INT_NONE;
            for (int q = lane; q < S; q += 32) {
                const float v = __ldg(M + (size_t)q * S + zt);
                if (a[q] > 0.0f && v > 0.0f) emax = max(emax, ea[q] + fa_exponent(v));
            }
            emax = fa_warp_max_int(emax);
            int pick = -1;
            if (emax != FA_INT_NONE) {
                const float u = fa_uniform(seed, offset, (uint32_t)(t - 1), (uint32_t)b, FA_RNG_MID);
                pick = warp_categorical(S, u, [&](int q) {
                    const float v = __ldg(M + (size_t)q * S + zt);
                    if (!(a[q] > 0.0f && v > 0.0f)) return 0.0f;
                    float mv;
                    int ev;
                    fa_split(v, mv, ev);
                    return a[q] * mv * fa_pow2(ea[q] + ev - emax);
                });
            }
            if (lane == 0) {
                if (pick < 0) { status[b] = FA_ROW_UNDERFLOW; pick = fa.start; }
                zb[t - 1] = pick;
                zcur = pick;
            }
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------- greedy (MAP) decoding

// Greedy (T = 0) decoding by max-product over the same tree (the max-product reweight and span
// products above; paperfeed.app summary, greedy decoding under the constraint): the root takes
// the best accepting end state, every midpoint the best state given its segment's ends, every
// leaf the best token of the chosen edge set.  Ties go to the lowest index everywhere.

// Warp argmax of w(i) > 0 over i < n, the lowest index among equal values; -1 if none is
// positive.  *best gets the maximum.
template <class WF>
__device__ int warp_argmax(int n, WF w, float *best) {
    float bv = 0.0f;
    int bi = -1;
    for (int i = (threadIdx.x & 31); i < n; i += 32) {
        const float x = w(i);
        if (x > bv) { bv = x; bi = i; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) { bv = ov; bi = oi; }
    }
    *best = bv;
    return bi;
}

__global__ void __launch_bounds__(32) k_map_root(DevFA fa, int L, int nK, const float *__restrict__ mant_root,
                                                 const int32_t *__restrict__ rho_root, int32_t *z, double *score,
                                                 int32_t *status, const int32_t *__restrict__ range_lost) {
    const int b = blockIdx.x, S = fa.S, s0 = fa.start;
    const float *row = mant_root + (size_t)b * nK * S * S + (size_t)s0 * S;
    float best;
    const int pick = warp_argmax(fa.n_accept, [&](int i) { return row[fa.accept[i]]; }, &best);
    if (threadIdx.x == 0) {
        const size_t bnd0 = (size_t)b * (L + 1);
        z[bnd0] = s0;
        if (range_lost[b]) {            // a max-product lost a candidate below the fp32 range
            status[b] = FA_ROW_UNDERFLOW;
            score[b] = NAN;
            z[bnd0 + L] = s0;
        } else if (pick < 0) {
            status[b] = FA_ROW_EMPTY;
            score[b] = -INFINITY;
            z[bnd0 + L] = s0;
        } else {
            status[b] = FA_ROW_OK;
            score[b] = (double)rho_root[(size_t)b * nK * S + s0] * 0.69314718055994530942 + log((double)best);
            z[bnd0 + L] = fa.accept[pick];
        }
    }
}

// Level k: the midpoint m of every node [l, r) takes argmax_s A[l, m)[z_l, s] A[m, r)[s, z_r].
__global__ void __launch_bounds__(kThreads) k_map_midpoints(int S, int B, int L, int k, int nc, int np,
                                                          const float *__restrict__ mant,
                                                          const int32_t *__restrict__ rho, int32_t *z,
                                                          int32_t *status) {
    const long gw = (long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (gw >= (long)B * np) return;
    const int b = (int)(gw / np), j = (int)(gw % np);
    const int l = j << (k + 1), m = l + (1 << k);
    if (m >= L) return;
    const int r = min(l + (1 << (k + 1)), L);
    if (__shfl_sync(0xffffffffu, status[b], 0) != FA_ROW_OK) return;
    const int32_t *zb = z + (size_t)b * (L + 1);
    const int zl = zb[l], zr = zb[r];
    const size_t lnode = (size_t)b * nc + 2 * j, rnode = lnode + 1;
    const float *Lrow = mant + lnode * (size_t)S * S + (size_t)zl * S;
    const float *R = mant + rnode * (size_t)S * S;
    const int32_t *rhoR = rho + rnode * S;
    const int lane = threadIdx.x & 31;
    int emax = FA_INT_NONE;
    for (int q = lane; q < S; q += 32) {
        const float x = Lrow[q], y = R[(size_t)q * S + zr];
        if (x > 0.0f && y > 0.0f) emax = max(emax, rhoR[q] + fa_exponent(x) + fa_exponent(y));
    }
    emax = fa_warp_max_int(emax);
    int pick = -1;
    if (emax != FA_INT_NONE) {
        float best;
        pick = warp_argmax(S, [&](int q) {
            const float x = Lrow[q], y = R[(size_t)q * S + zr];
            if (!(x > 0.0f && y > 0.0f)) return 0.0f;
            float mx, my;
            int ex, ey;
            fa_split(x, mx, ex);
            fa_split(y, my, ey);
            return mx * my * fa_pow2(rhoR[q] + ex + ey - emax);
        }, &best);
    }
    if (lane == 0) {
        if (pick < 0) status[b] = FA_ROW_UNDERFLOW;
        else z[(size_t)b * (L + 1) + m] = pick;
    }
}

// Leaves: the best token of the cell z_{t-1} -> z_t (committed positions echo their token).
__global__ void __launch_bounds__(kThreads) k_map_leaf(DevFA fa, int B, int L, const float *__restrict__ probs,
                                                     const int32_t *__restrict__ committed,
                                                     const int32_t *__restrict__ z, int32_t *tokens,
                                                     int32_t *status) {
    const long gw = (long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (gw >= (long)B * L) return;
    const int b = (int)(gw / L), t = (int)(gw % L), lane = threadIdx.x & 31;
    const size_t pos = (size_t)b * L + t;
    const int c = committed[pos];
    if (c >= 0) {
        if (lane == 0) tokens[pos] = c;
        return;
    }
    if (__shfl_sync(0xffffffffu, status[b], 0) != FA_ROW_OK) {
        if (lane == 0) tokens[pos] = -1;
        return;
    }
    const int32_t *zb = z + (size_t)b * (L + 1);
    const int zp = zb[t], zn = zb[t + 1];
    int lo = fa.row_cell_off[zp], hi = fa.row_cell_off[zp + 1];
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (fa.cell_dst[mid] < zn) lo = mid + 1; else hi = mid;
    }
    int v = -1;
    if (lo < fa.row_cell_off[zp + 1] && fa.cell_dst[lo] == zn) {
        const int64_t a0 = fa.cell_off[lo];
        const int n = (int)(fa.cell_off[lo + 1] - a0);
        const float *prow = probs + pos * (size_t)fa.V;
        float best;
        const int pick = warp_argmax(n, [&](int i) { return __ldg(prow + fa.cell_tok[a0 + i]); }, &best);
        if (pick >= 0) v = fa.cell_tok[a0 + pick];
    }
    if (lane == 0) {
        tokens[pos] = v;
        if (v < 0) status[b] = FA_ROW_UNDERFLOW;
    }
}

// Sequences that failed: -1 at every masked position and a score of -inf.
__global__ void k_map_fix(int B, int L, const int32_t *__restrict__ committed, const int32_t *__restrict__ status,
                          int32_t *tokens, double *score) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)B * L) return;
    const int b = (int)(i / L), t = (int)(i % L);
    if (status[b] == FA_ROW_OK) return;
    if (committed[i] < 0) tokens[i] = -1;
    if (t == 0) score[b] = -INFINITY;
}

// ----------------------------------------------------------------------------- 6. commit

// Per sequence, the k masked positions of [lo, hi) with the largest marginal, descending,
// ties to the lower position (papernotes.org key design 3, the "Mar" confidence; LLaDA's
// highest-probability rule in the paperfeed.app summary).  Rank by counting larger keys.
// A sequence whose status is not OK gets no commits and -1 tokens / 0 marginals at every
// masked position (some leaves may have been drawn before the failure was recorded).
// Executed by one whole block; skey holds hi - lo keys.
// Order-preserving bits of a float (any sign): larger float, larger key.
__device__ __forceinline__ uint32_t fa_order_bits(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ void topk_row(int b, int L, int k, int lo, int hi, float *marg, const float *conf,
                         const int32_t *__restrict__ committed, const int32_t *status, int32_t *out, int32_t *tokens,
                         unsigned long long *skey) {
    int32_t *o = out + (size_t)b * k;
    for (int i = threadIdx.x; i < k; i += blockDim.x) o[i] = -1;
    if (status[b] != FA_ROW_OK) {
        for (int t = threadIdx.x; t < L; t += blockDim.x)
            if (committed[(size_t)b * L + t] < 0) { tokens[(size_t)b * L + t] = -1; marg[(size_t)b * L + t] = 0.0f; }
        return;
    }
    const float *cf = conf + (size_t)b * L;
    const int32_t *cm = committed + (size_t)b * L;
    const int t0 = max(lo, 0), t1 = min(hi, L), n = t1 - t0;
    // key = (confidence bits, ~t): larger confidence first, then lower position; 0 = not eligible
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int t = t0 + i;
        skey[i] = (cm[t] >= 0) ? 0ull
                               : (((unsigned long long)fa_order_bits(cf[t]) << 32) |
                                  (unsigned long long)(0xFFFFFFFFu - (unsigned)t));
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const unsigned long long kt = skey[i];
        if (!kt) continue;
        int rank = 0;
        for (int q = 0; q < n && rank < k; ++q) rank += skey[q] > kt;
        if (rank < k) o[rank] = t0 + i;
    }
}

// committed[b, idx] = tokens[b, idx] for every idx >= 0 in commit_idx[b, :].
__global__ void k_apply_commits(int B, int L, int k, const int32_t *__restrict__ commit_idx,
                                const int32_t *__restrict__ tokens, int32_t *committed) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)B * k) return;
    const int b = (int)(i / k);
    const int t = commit_idx[i];
    if (t >= 0 && t < L) committed[(size_t)b * L + t] = tokens[(size_t)b * L + t];
}

// L = 0: the empty string is the only candidate.
__global__ void k_empty_length(int start, const int32_t *accept_mask, int B, int k, double *logZ, int32_t *status,
                               int32_t *commit_idx) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const bool ok = accept_mask[start] != 0;
    logZ[b] = ok ? 0.0 : -INFINITY;
    status[b] = ok ? FA_ROW_OK : FA_ROW_EMPTY;
    for (int i = 0; i < k; ++i) commit_idx[(size_t)b * k + i] = -1;
}

// ----------------------------------------------------------------------------- host glue

std::atomic<unsigned long long> g_launches{0};

fa_status launch_check(const char *what) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        fa_set_error(std::string(what) + ": " + cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

// Stage-boundary timing events (per host thread): when enabled, every step records
// FA_N_STAGES + 1 events on its stream, as graph nodes if the stream is being captured.
struct StageEvents {
    bool enabled = false;
    bool created = false;
    cudaEvent_t ev[FA_N_STAGES + 1];
};
thread_local StageEvents g_stage;

void stage_mark(int i, cudaStream_t s) {
    if (!g_stage.enabled) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(g_stage.ev[i], s, cudaEventRecordExternal);
    else cudaEventRecord(g_stage.ev[i], s);
}

int pick_partition(const fa_automaton *a, long positions) {
    // the first partition giving about three blocks per SM over all positions: every extra
    // block re-stages its probability row and repeats its metadata round trips
    int p = 0;
    while (p + 1 < (int)a->part_count.size() && positions * a->part_count[p] < 152L * 3) ++p;
    return p;
}

fa_status check_device(const fa_automaton *a, const char *fn) {
    int dev = -1;
    cudaGetDevice(&dev);
    if (dev != a->device) {
        fa_set_error(std::string(fn) + ": current device differs from the automaton's device");
        return FA_ERR_INVALID_ARG;
    }
    return FA_OK;
}

fa_status launch_reweight(const fa_automaton *a, int B, int L, const float *probs, const int32_t *committed,
                          float *mant, int32_t *rho, int32_t *rmax, int32_t *rminc, cudaStream_t st,
                          int32_t *zero = nullptr, long n_zero = 0, bool use_max = false,
                          int32_t *fflag = nullptr, int32_t *fmap = nullptr, long layout_positions = -1) {
    // the row-block layout is chosen by the whole batch's positions (layout_positions when a
    // batch is reweighted in pieces, so every piece sums its cells exactly as the whole would)
    const int p = pick_partition(a, layout_positions >= 0 ? layout_positions : (long)B * L);
    const int nrb = a->part_count[p];
    const int4 *rbm = reinterpret_cast<const int4 *>(a->rb_meta) + 2 * a->part_first[p];
    const int max_units = a->part_max_units[p];
    const int threads = std::min(32 * FA_RW_WARPS, std::max(256, 32 * max_units));
    // the staged chunk, whose space takes the units' run totals and the row maxima and minima
    // at the end, then one run-slot array per warp
    int tot_floats = (int)std::max((size_t)((a->chunk_tokens + FA_PAD_SLOTS + 3) & ~3),
                                   (size_t)max_units * FA_UNIT_SLOTS + 2 * (size_t)a->part_max_rows[p]);
    // the rows of M_t are assembled in shared memory when the largest block's totals and rows
    // fit beside the chunk without costing the second block per SM (227 KB per block, 228 KB
    // per SM with 1 KB reserved per block)
    const long per_block_floats = (233472L / 2 - 1024) / 4 - (long)(threads / 32) * FA_UNIT_SLOTS - 32;
    int tile = 0;
    if ((long)a->part_tile_floats[p] <= std::max<long>(tot_floats, per_block_floats)) {
        tot_floats = std::max(tot_floats, (int)((a->part_tile_floats[p] + 3) & ~3L));
        tile = ((a->S & 3) == 0 && (reinterpret_cast<uintptr_t>(mant) & 15) == 0) ? 2 : 1;
    }
    const size_t smem = sizeof(float) * ((size_t)tot_floats + (size_t)(threads / 32) * FA_UNIT_SLOTS + 32);
    // units per warp: the register totals of a third unit cost the smaller layouts ~10%
    const int upw = (max_units + FA_RW_WARPS - 1) / FA_RW_WARPS;
    using K = void (*)(DevFA, int, const float *, const int32_t *, const int4 *, int, int, float *, int32_t *, int32_t *,
                       int32_t *, int32_t *, long, int, int32_t *, int32_t *);
    K kern = upw <= 1 ? (use_max ? (K)k_reweight<true, 1> : (K)k_reweight<false, 1>)
             : upw == 2 ? (use_max ? (K)k_reweight<true, 2> : (K)k_reweight<false, 2>)
                        : (use_max ? (K)k_reweight<true, 3> : (K)k_reweight<false, 3>);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) { fa_set_error(std::string("reweight smem: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    }
    dim3 grid((unsigned)((long)L * nrb), (unsigned)B);
    kern<<<grid, threads, smem, st>>>(dev_view(a), L, probs, committed, rbm, nrb, tot_floats, mant, rho, rmax, rminc,
                                      zero, n_zero, tile, fflag, fmap);
    return launch_check("reweight");
}

fa_status launch_token_marginals(const fa_automaton *aut, int B, int L, const float *probs, const int32_t *committed,
                                 const Plan &p, const char *ws, const int32_t *row_status, float *marg_all,
                                 float *entropy, float *conf, cudaStream_t st) {
    const size_t smem = ((size_t)aut->S + 1) * 16;
    if (smem > 44 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_tm_partial, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) { fa_set_error(std::string("token marginals smem: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    }
    auto F = [&](size_t off) { return (const float *)(ws + off); };
    auto I = [&](size_t off) { return (const int32_t *)(ws + off); };
    double *part = (double *)(ws + p.tm_part);
    const long n_pos = (long)B * L;
    k_tm_partial<<<(unsigned)(n_pos * p.tm_chunks), kTmThreads, smem, st>>>(
        dev_view(aut), L, p.tm_chunks, p.tm_chunk, probs, committed, row_status, F(p.am), I(p.ae), F(p.bm), I(p.be), F(p.den_m),
        I(p.den_e), marg_all, part);
    fa_status s = launch_check("token marginals");
    if (s != FA_OK) return s;
    if (entropy || conf) {
        k_tm_finish<<<(unsigned)((n_pos + 255) / 256), 256, 0, st>>>(n_pos, p.tm_chunks, part, entropy, conf);
        s = launch_check("entropies");
    }
    return s;
}

}  // namespace

extern "C" fa_status fa_token_marginals(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                        const int32_t *committed, const void *workspace, size_t ws_bytes,
                                        const int32_t *row_status, float *marg_all, float *entropy,
                                        fa_stream stream) {
    if (!aut) { fa_set_error("fa_token_marginals: NULL automaton"); return FA_ERR_INVALID_ARG; }
    if (B < 0 || B > 65535 || L < 0 || L > FA_MAX_LENGTH) {
        fa_set_error("fa_token_marginals: B or L out of range"); return FA_ERR_INVALID_ARG;
    }
    if ((long)B * L == 0 || (!marg_all && !entropy)) return FA_OK;
    if (!probs || !committed || !workspace || !row_status) {
        fa_set_error("fa_token_marginals: NULL buffer"); return FA_ERR_INVALID_ARG;
    }
    fa_status st = check_device(aut, "fa_token_marginals");
    if (st != FA_OK) return st;
    const Plan p = make_plan(aut, B, L);
    if (ws_bytes < p.total) {
        fa_set_error("fa_token_marginals: workspace needs " + std::to_string(p.total) + " bytes");
        return FA_ERR_WORKSPACE_TOO_SMALL;
    }
    if (((uintptr_t)workspace & 255) != 0) { fa_set_error("fa_token_marginals: workspace not 256-byte aligned"); return FA_ERR_INVALID_ARG; }
    return launch_token_marginals(aut, B, L, probs, committed, p, (const char *)workspace, row_status, marg_all, entropy,
                                  nullptr, (cudaStream_t)stream);
}

extern "C" fa_status fa_map_step(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                 const int32_t *committed, void *workspace, size_t ws_bytes, int32_t *tokens,
                                 double *score, int32_t *row_status, fa_stream stream) {
    if (!aut) { fa_set_error("fa_map_step: NULL automaton"); return FA_ERR_INVALID_ARG; }
    if (B < 0 || B > 65535 || L < 0 || L > FA_MAX_LENGTH) { fa_set_error("fa_map_step: B or L out of range"); return FA_ERR_INVALID_ARG; }
    if (B == 0) return FA_OK;
    if (!score || !row_status || (L > 0 && (!probs || !committed || !tokens))) {
        fa_set_error("fa_map_step: NULL buffer"); return FA_ERR_INVALID_ARG;
    }
    fa_status st = check_device(aut, "fa_map_step");
    if (st != FA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (L == 0) {
        k_empty_length<<<(B + 255) / 256, 256, 0, s>>>(aut->start, aut->accept_mask, B, 0, score, row_status, nullptr);
        return launch_check("empty length");
    }
    const Plan p = make_plan(aut, B, L);
    if (!workspace || ws_bytes < p.total) {
        fa_set_error("fa_map_step: workspace needs " + std::to_string(p.total) + " bytes");
        return FA_ERR_WORKSPACE_TOO_SMALL;
    }
    if (((uintptr_t)workspace & 255) != 0) { fa_set_error("fa_map_step: workspace not 256-byte aligned"); return FA_ERR_INVALID_ARG; }
    char *ws = (char *)workspace;
    auto F = [&](size_t off) { return (float *)(ws + off); };
    auto I = [&](size_t off) { return (int32_t *)(ws + off); };
    const int S = aut->S;
    stage_mark(0, s);
    st = launch_reweight(aut, B, L, probs, committed, F(p.mant[0]), I(p.rho[0]), I(p.rmax[0]), I(p.rminc[0]), s,
                         I(p.rmax_hi), (long)(p.rmax_hi_bytes / sizeof(int32_t)), true);
    if (st != FA_OK) return st;
    stage_mark(1, s);
    for (int kk = 1; kk <= p.K; ++kk) {
        if (S <= SMALL_S) {
            const long tpd = (S + ST - 1) / ST;
            k_span_small<true><<<(unsigned)((long)B * p.nk[kk] * tpd * tpd), kThreads, 0, s>>>(
                S, L, kk, p.nk[kk], F(p.mant[kk - 1]), I(p.rho[kk - 1]), I(p.rmax[kk - 1]), I(p.rminc[kk - 1]),
                p.nk[kk - 1], F(p.mant[kk]), I(p.rho[kk]), I(p.rmax[kk]), I(p.rminc[kk]), I(p.range_lost));
            if ((st = launch_check("span product (small, max)")) != FA_OK) return st;
            continue;
        }
        dim3 g1((S + kWarps - 1) / kWarps, p.nk[kk], B);
        k_rowshift<<<g1, kThreads, 0, s>>>(S, L, kk, p.nk[kk], F(p.mant[kk - 1]), I(p.rho[kk - 1]), I(p.rmax[kk - 1]),
                                           p.nk[kk - 1], I(p.mu[kk]), I(p.rmax[kk]), nullptr);
        if ((st = launch_check("rowshift")) != FA_OK) return st;
        const long tiles = (S + GBN - 1) / GBN;
        k_gemm_simt<true><<<(unsigned)((long)B * p.nk[kk] * tiles * tiles), kThreads, 0, s>>>(
            S, L, kk, p.nk[kk], F(p.mant[kk - 1]), I(p.rho[kk - 1]), I(p.rmax[kk - 1]), I(p.rminc[kk - 1]),
            p.nk[kk - 1], I(p.mu[kk]), F(p.mant[kk]), I(p.rho[kk]), I(p.rmax[kk]), I(p.rminc[kk]), I(p.range_lost));
        if ((st = launch_check("span product (max)")) != FA_OK) return st;
    }
    stage_mark(2, s);
    k_map_root<<<B, 32, 0, s>>>(dev_view(aut), L, p.nk[p.K], F(p.mant[p.K]), I(p.rho[p.K]), I(p.z), score, row_status,
                                I(p.range_lost));
    if ((st = launch_check("greedy root")) != FA_OK) return st;
    for (int kk = p.K - 1; kk >= 0; --kk) {
        const int np = p.nk[kk + 1];
        k_map_midpoints<<<(unsigned)(((long)B * np + kWarps - 1) / kWarps), kThreads, 0, s>>>(
            S, B, L, kk, p.nk[kk], np, F(p.mant[kk]), I(p.rho[kk]), I(p.z), row_status);
        if ((st = launch_check("greedy midpoints")) != FA_OK) return st;
    }
    stage_mark(3, s);
    k_map_leaf<<<(unsigned)(((long)B * L + kWarps - 1) / kWarps), kThreads, 0, s>>>(dev_view(aut), B, L, probs, committed,
                                                                              I(p.z), tokens, row_status);
    if ((st = launch_check("greedy leaves")) != FA_OK) return st;
    k_map_fix<<<(unsigned)(((long)B * L + 255) / 256), 256, 0, s>>>(B, L, committed, row_status, tokens, score);
    st = launch_check("greedy fix-up");
    stage_mark(4, s);
    return st;
}

extern "C" fa_status fa_step_workspace_bytes(const fa_automaton *aut, int32_t B, int32_t L, size_t *bytes) {
    if (!aut || !bytes) { fa_set_error("fa_step_workspace_bytes: NULL argument"); return FA_ERR_INVALID_ARG; }
    if (B < 0 || L < 0 || L > FA_MAX_LENGTH) { fa_set_error("fa_step_workspace_bytes: B or L out of range"); return FA_ERR_INVALID_ARG; }
    *bytes = make_plan(aut, B, L).total;
    return FA_OK;
}

extern "C" fa_status fa_transition_matrices(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                            const int32_t *committed, float *mant, int32_t *row_exp,
                                            fa_stream stream) {
    if (!aut) { fa_set_error("fa_transition_matrices: NULL automaton"); return FA_ERR_INVALID_ARG; }
    if (B < 0 || L < 0 || B > 65535) { fa_set_error("fa_transition_matrices: B or L out of range"); return FA_ERR_INVALID_ARG; }
    if ((long)B * L == 0) return FA_OK;
    if (!probs || !committed || !mant || !row_exp) { fa_set_error("fa_transition_matrices: NULL buffer"); return FA_ERR_INVALID_ARG; }
    fa_status st = check_device(aut, "fa_transition_matrices");
    if (st != FA_OK) return st;
    return launch_reweight(aut, B, L, probs, committed, mant, row_exp, nullptr, nullptr, (cudaStream_t)stream);
}

extern "C" fa_status fa_constrained_step(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                         const int32_t *committed, uint64_t philox_seed, uint64_t philox_offset,
                                         int32_t k, int32_t commit_lo, int32_t commit_hi, void *workspace,
                                         size_t ws_bytes, int32_t *tokens, double *logZ, float *marg,
                                         int32_t *commit_idx, int32_t *row_status, fa_stream stream) {
    return fa_constrained_step_ex(aut, B, L, probs, committed, philox_seed, philox_offset, k, commit_lo, commit_hi,
                                  FA_CONF_MARGINAL, workspace, ws_bytes, tokens, logZ, marg, nullptr, commit_idx,
                                  row_status, stream);
}

namespace {
// Inputs still in host memory (fa_constrained_step_host): copied into the device buffers
// probs / committed in pieces of positions, each piece's reweighting started once it has
// landed.
struct HostInput {
    const float *probs;
    const int32_t *committed;
};

fa_status step_impl(const fa_automaton *aut, int32_t B, int32_t L, const float *probs, const int32_t *committed,
                    uint64_t philox_seed, uint64_t philox_offset, int32_t k, int32_t commit_lo, int32_t commit_hi,
                    int32_t confidence, void *workspace, size_t ws_bytes, int32_t *tokens, double *logZ, float *marg,
                    float *entropy, int32_t *commit_idx, int32_t *row_status, fa_stream stream, bool chain,
                    const HostInput *hin = nullptr);
}

extern "C" fa_status fa_constrained_step_ex(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                            const int32_t *committed, uint64_t philox_seed, uint64_t philox_offset,
                                            int32_t k, int32_t commit_lo, int32_t commit_hi, int32_t confidence,
                                            void *workspace, size_t ws_bytes, int32_t *tokens, double *logZ,
                                            float *marg, float *entropy, int32_t *commit_idx, int32_t *row_status,
                                            fa_stream stream) {
    return step_impl(aut, B, L, probs, committed, philox_seed, philox_offset, k, commit_lo, commit_hi, confidence,
                     workspace, ws_bytes, tokens, logZ, marg, entropy, commit_idx, row_status, stream, false);
}

extern "C" fa_status fa_constrained_step_host(const fa_automaton *aut, int32_t B, int32_t L, const float *h_probs,
                                              const int32_t *h_committed, float *d_probs, int32_t *d_committed,
                                              uint64_t philox_seed, uint64_t philox_offset, int32_t k,
                                              int32_t commit_lo, int32_t commit_hi, void *workspace, size_t ws_bytes,
                                              int32_t *tokens, double *logZ, float *marg, int32_t *commit_idx,
                                              int32_t *row_status, fa_stream stream) {
    if (B > 0 && L > 0 && (!h_probs || !h_committed || !d_probs || !d_committed)) {
        fa_set_error("fa_constrained_step_host: NULL input buffer");
        return FA_ERR_INVALID_ARG;
    }
    const HostInput hin{h_probs, h_committed};
    return step_impl(aut, B, L, d_probs, d_committed, philox_seed, philox_offset, k, commit_lo, commit_hi,
                     FA_CONF_MARGINAL, workspace, ws_bytes, tokens, logZ, marg, nullptr, commit_idx, row_status, stream,
                     false, &hin);
}

extern "C" fa_status fa_constrained_step_chain(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                               const int32_t *committed, uint64_t philox_seed,
                                               uint64_t philox_offset, int32_t k, int32_t commit_lo,
                                               int32_t commit_hi, int32_t confidence, void *workspace,
                                               size_t ws_bytes, int32_t *tokens, double *logZ, float *marg,
                                               float *entropy, int32_t *commit_idx, int32_t *row_status,
                                               fa_stream stream) {
    return step_impl(aut, B, L, probs, committed, philox_seed, philox_offset, k, commit_lo, commit_hi, confidence,
                     workspace, ws_bytes, tokens, logZ, marg, entropy, commit_idx, row_status, stream, true);
}

namespace {
// The copy stream and events of fa_constrained_step_host, per host thread and device.
struct CopyContext {
    cudaStream_t cs = nullptr;
    cudaEvent_t start = nullptr, com = nullptr;
    cudaEvent_t chunk[kHostChunks] = {};
};

fa_status copy_context(CopyContext *&out) {
    static thread_local std::vector<CopyContext> ctx;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { fa_set_error(std::string("host inputs: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    if ((int)ctx.size() <= dev) ctx.resize(dev + 1);
    CopyContext &c = ctx[dev];
    if (!c.cs) {
        e = cudaStreamCreateWithFlags(&c.cs, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.start, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.com, cudaEventDisableTiming);
        for (int i = 0; i < kHostChunks && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&c.chunk[i], cudaEventDisableTiming);
        if (e != cudaSuccess) { c.cs = nullptr; fa_set_error(std::string("host inputs: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    }
    out = &c;
    return FA_OK;
}

// Emission reweighting from host inputs: the committed tokens and then the probabilities are
// copied on the copy stream (after the work already on `s`) in up to kHostChunks pieces of
// consecutive positions, and the reweighting of each piece runs on `s` once its rows are in,
// so the copies of later pieces overlap the reweighting of earlier ones.
fa_status reweight_from_host(const fa_automaton *a, int B, int L, const HostInput &hin, float *d_probs,
                             int32_t *d_committed, float *mant, int32_t *rho, int32_t *rmax, int32_t *rminc,
                             cudaStream_t s, int32_t *zero, long n_zero, int32_t *fflag, int32_t *fmap) {
    CopyContext *c = nullptr;
    fa_status st = copy_context(c);
    if (st != FA_OK) return st;
    const size_t S = (size_t)a->S, V = (size_t)a->V, P = (size_t)B * (size_t)L;
    size_t bound[kHostChunks + 1];
    const int nch = fa_host_pieces(P, bound);
    cudaError_t e = cudaEventRecord(c->start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->cs, c->start, 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(d_committed, hin.committed, P * sizeof(int32_t), cudaMemcpyHostToDevice, c->cs);
    if (e == cudaSuccess) e = cudaEventRecord(c->com, c->cs);
    for (int i = 0; i < nch && e == cudaSuccess; ++i) {
        e = cudaMemcpyAsync(d_probs + bound[i] * V, hin.probs + bound[i] * V,
                            (bound[i + 1] - bound[i]) * V * sizeof(float), cudaMemcpyHostToDevice, c->cs);
        if (e == cudaSuccess) e = cudaEventRecord(c->chunk[i], c->cs);
    }
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c->com, 0);
    if (e != cudaSuccess) { fa_set_error(std::string("host inputs: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    for (int i = 0; i < nch; ++i) {
        e = cudaStreamWaitEvent(s, c->chunk[i], 0);
        if (e != cudaSuccess) { fa_set_error(std::string("host inputs: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
        const size_t p0 = bound[i];
        st = launch_reweight(a, 1, (int)(bound[i + 1] - p0), d_probs + p0 * V, d_committed + p0, mant + p0 * S * S,
                             rho + p0 * S, rmax + p0 * S, rminc + p0 * S, s, i == 0 ? zero : nullptr,
                             i == 0 ? n_zero : 0, false, fflag ? fflag + p0 : nullptr, fmap ? fmap + p0 * S : nullptr,
                             (long)P);
        if (st != FA_OK) return st;
    }
    return FA_OK;
}

fa_status step_impl(const fa_automaton *aut, int32_t B, int32_t L, const float *probs, const int32_t *committed,
                    uint64_t philox_seed, uint64_t philox_offset, int32_t k, int32_t commit_lo, int32_t commit_hi,
                    int32_t confidence, void *workspace, size_t ws_bytes, int32_t *tokens, double *logZ, float *marg,
                    float *entropy, int32_t *commit_idx, int32_t *row_status, fa_stream stream, bool chain,
                    const HostInput *hin) {
    if (!aut) { fa_set_error("fa_constrained_step: NULL automaton"); return FA_ERR_INVALID_ARG; }
    if (confidence != FA_CONF_MARGINAL && confidence != FA_CONF_NEG_ENTROPY && confidence != FA_CONF_UNCONSTRAINED) {
        fa_set_error("fa_constrained_step: unknown confidence"); return FA_ERR_INVALID_ARG;
    }
    if (B < 0 || B > 65535 || L < 0 || L > FA_MAX_LENGTH || k < 0) {
        fa_set_error("fa_constrained_step: B, L or k out of range"); return FA_ERR_INVALID_ARG;
    }
    if (commit_lo < 0 || commit_hi < commit_lo || commit_hi > L) {
        fa_set_error("fa_constrained_step: commit window must satisfy 0 <= lo <= hi <= L"); return FA_ERR_INVALID_ARG;
    }
    if (B == 0) return FA_OK;
    if (!logZ || !row_status || (k > 0 && !commit_idx)) { fa_set_error("fa_constrained_step: NULL output"); return FA_ERR_INVALID_ARG; }
    if (L > 0 && (!probs || !committed || !tokens || !marg)) { fa_set_error("fa_constrained_step: NULL buffer"); return FA_ERR_INVALID_ARG; }
    fa_status st = check_device(aut, "fa_constrained_step");
    if (st != FA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (L == 0) {
        k_empty_length<<<(B + 255) / 256, 256, 0, s>>>(aut->start, aut->accept_mask, B, k, logZ, row_status, commit_idx);
        return launch_check("empty length");
    }
    const Plan p = make_plan(aut, B, L);
    if (!workspace || ws_bytes < p.total) {
        fa_set_error("fa_constrained_step: workspace needs " + std::to_string(p.total) + " bytes");
        return FA_ERR_WORKSPACE_TOO_SMALL;
    }
    if (((uintptr_t)workspace & 255) != 0) { fa_set_error("fa_constrained_step: workspace not 256-byte aligned"); return FA_ERR_INVALID_ARG; }
    char *ws = (char *)workspace;
    auto F = [&](size_t off) { return (float *)(ws + off); };
    auto I = [&](size_t off) { return (int32_t *)(ws + off); };
    const int S = aut->S;

    // 1. emission reweighting -> level-0 spans (also clears the row maxima of levels >= 1)
    stage_mark(0, s);
    if (hin)
        st = reweight_from_host(aut, B, L, *hin, const_cast<float *>(probs), const_cast<int32_t *>(committed),
                                F(p.mant[0]), I(p.rho[0]), I(p.rmax[0]), I(p.rminc[0]), s, I(p.rmax_hi),
                                (long)(p.rmax_hi_bytes / sizeof(int32_t)), p.functional ? I(p.fflag[0]) : nullptr,
                                p.functional ? I(p.fmap[0]) : nullptr);
    else
        st = launch_reweight(aut, B, L, probs, committed, F(p.mant[0]), I(p.rho[0]), I(p.rmax[0]), I(p.rminc[0]), s,
                             I(p.rmax_hi), (long)(p.rmax_hi_bytes / sizeof(int32_t)), false,
                             p.functional ? I(p.fflag[0]) : nullptr, p.functional ? I(p.fmap[0]) : nullptr);
    if (st != FA_OK) return st;

    if (chain) {
        // 2-4, chain form: forward messages, then backward messages with the state draws
        stage_mark(1, s);
        const size_t fsm = chain_smem(S, true), bsm = chain_smem(S, false);
        if (fsm > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(k_chain_forward, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(k_chain_backward, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bsm);
            if (e != cudaSuccess) { fa_set_error(std::string("chain smem: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
        }
        k_chain_forward<<<B, kChThreads, fsm, s>>>(dev_view(aut), L, F(p.mant[0]), F(p.am), I(p.ae));
        if ((st = launch_check("chain forward")) != FA_OK) return st;
        stage_mark(2, s);
        k_chain_backward<<<B, kChThreads, bsm, s>>>(dev_view(aut), L, F(p.mant[0]), F(p.am), I(p.ae), F(p.bm),
                                                    I(p.be), I(p.z), philox_seed, philox_offset, logZ, row_status,
                                                    F(p.zsum), I(p.zexp));
        if ((st = launch_check("chain backward")) != FA_OK) return st;
    }

    // 2. up-sweep: level k from level k-1
    if (!chain) stage_mark(1, s);
    for (int kk = 1; kk <= p.K && !chain; ++kk) {
        if (S <= SMALL_S) {
            const long tpd = (S + ST - 1) / ST;
            k_span_small<false><<<(unsigned)((long)B * p.nk[kk] * tpd * tpd), kThreads, 0, s>>>(
                S, L, kk, p.nk[kk], F(p.mant[kk - 1]), I(p.rho[kk - 1]), I(p.rmax[kk - 1]), I(p.rminc[kk - 1]),
                p.nk[kk - 1], F(p.mant[kk]), I(p.rho[kk]), I(p.rmax[kk]), I(p.rminc[kk]), I(p.range_lost));
            if ((st = launch_check("span product (small)")) != FA_OK) return st;
            continue;
        }
        // functional spans of this level (a DFA on the tensor-core path), before its products
        int32_t *fflag_k = nullptr, *fmap_k = nullptr;
        if (p.functional) {
            fflag_k = I(p.fflag[kk]);
            fmap_k = I(p.fmap[kk]);
            k_func_level<<<(unsigned)((long)B * p.nk[kk]), kThreads, 0, s>>>(S, L, kk, p.nk[kk], p.nk[kk - 1],
                                                                             I(p.fflag[kk - 1]), I(p.fmap[kk - 1]),
                                                                             fflag_k, fmap_k);
            if ((st = launch_check("functional spans")) != FA_OK) return st;
        }
        dim3 g1((S + kWarps - 1) / kWarps, p.nk[kk], B);
        k_rowshift<<<g1, kThreads, 0, s>>>(S, L, kk, p.nk[kk], F(p.mant[kk - 1]), I(p.rho[kk - 1]), I(p.rmax[kk - 1]),
                                           p.nk[kk - 1], I(p.mu[kk]), I(p.rmax[kk]), fflag_k);
        if ((st = launch_check("rowshift")) != FA_OK) return st;
        if (fa_span_tc_supported(S)) {
            g_launches.fetch_add(2, std::memory_order_relaxed);
            st = fa_span_tc_level(S, B, L, kk, p.nk[kk], F(p.mant[kk - 1]), I(p.rho[kk - 1]), I(p.rmax[kk - 1]),
                                  I(p.rminc[kk - 1]), p.nk[kk - 1], I(p.mu[kk]), F(p.mant[kk]), I(p.rho[kk]),
                                  I(p.rmax[kk]), I(p.rminc[kk]), I(p.tc_err), I(p.range_lost), ws + p.img, s, fflag_k,
                                  fmap_k);
            if (st != FA_OK) return st;
            continue;
        }
        const long tiles = (S + GBN - 1) / GBN;
        const long g2 = (long)B * p.nk[kk] * tiles * tiles;
        k_gemm_simt<false><<<(unsigned)g2, kThreads, 0, s>>>(S, L, kk, p.nk[kk], F(p.mant[kk - 1]), I(p.rho[kk - 1]), I(p.rmax[kk - 1]),
                                            I(p.rminc[kk - 1]), p.nk[kk - 1], I(p.mu[kk]), F(p.mant[kk]), I(p.rho[kk]),
                                            I(p.rmax[kk]), I(p.rminc[kk]), I(p.range_lost));
        if ((st = launch_check("span product")) != FA_OK) return st;
    }

    // 3. root: logZ, end state, boundary messages
    if (!chain) stage_mark(2, s);
    if (!chain) k_root<<<B, kThreads, 0, s>>>(dev_view(aut), L, p.K, p.nk[p.K], F(p.mant[p.K]), I(p.rho[p.K]), philox_seed,
                                  philox_offset, I(p.z), F(p.am), I(p.ae), F(p.bm), I(p.be), F(p.zsum), I(p.zexp),
                                  logZ, row_status, I(p.tc_err), I(p.range_lost));
    if (!chain && (st = launch_check("root")) != FA_OK) return st;

    // 4. top-down: midpoints and prefix/suffix messages, level K-1 .. 0
    for (int kk = p.K - 1; kk >= 0 && !chain; --kk) {
        TopdownArgs ta;
        ta.S = S; ta.B = B; ta.L = L; ta.k = kk; ta.nc = p.nk[kk]; ta.np = p.nk[kk + 1];
        ta.CB = S >= 64 ? 64 : ((S + 31) / 32) * 32;
        ta.QS = kThreads / ta.CB;
        ta.nA = B * ta.np * ((S + ta.CB - 1) / ta.CB);
        ta.beta_rows = S >= 256 ? 4 * kWarps : kWarps;
        ta.fflag = p.functional ? I(p.fflag[kk]) : nullptr;
        ta.fmap = p.functional ? I(p.fmap[kk]) : nullptr;
        ta.nB = B * ta.np * ((S + ta.beta_rows - 1) / ta.beta_rows);
        const int nM = (B * ta.np + kWarps - 1) / kWarps;
        ta.mant = F(p.mant[kk]); ta.rho = I(p.rho[kk]); ta.rmax = I(p.rmax[kk]);
        ta.vec4 = (S & 3) == 0;
        ta.seed = philox_seed; ta.offset = philox_offset;
        ta.z = I(p.z); ta.status = row_status;
        ta.am = F(p.am); ta.ae = I(p.ae); ta.bm = F(p.bm); ta.be = I(p.be);
        const size_t smem = (size_t)S * 16 + (size_t)kThreads * 32;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(k_topdown, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) { fa_set_error(std::string("top-down smem: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
        }
        k_topdown<<<(unsigned)(ta.nA + ta.nB + nM), kThreads, smem, s>>>(ta);
        if ((st = launch_check("top-down level")) != FA_OK) return st;
    }

    // 5. leaves: tokens and marginals, then the commit (one launch); before them, when asked,
    //    the entropy of every position's full constrained distribution
    stage_mark(3, s);
    const bool entropies = confidence == FA_CONF_NEG_ENTROPY || entropy;
    const size_t leaf_smem = S <= kLeafStageStates ? (size_t)S * 24 : 0;
    if (leaf_smem + sizeof(LeafShared) > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_leaf_commit, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)leaf_smem);
        if (e != cudaSuccess) { fa_set_error(std::string("leaf smem: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    }
    k_leaf_commit<<<(unsigned)((long)B * L), kLeafThreads, leaf_smem, s>>>(
        dev_view(aut), B, L, probs, committed, philox_seed, philox_offset, I(p.z), F(p.am), I(p.ae), F(p.bm), I(p.be),
        tokens, marg, row_status, k, commit_lo, commit_hi, commit_idx, (unsigned long long *)(ws + p.keys),
        I(p.leaf_done), F(p.mant[0]), confidence, F(p.conf), F(p.den_m), I(p.den_e), entropies ? 0 : 1);
    st = launch_check("leaf and commit");
    if (st == FA_OK && entropies) {
        // the entropies need every leaf's normaliser; the commit waits for them
        st = launch_token_marginals(aut, B, L, probs, committed, p, ws, row_status, nullptr, entropy,
                                    confidence == FA_CONF_NEG_ENTROPY ? F(p.conf) : nullptr, s);
        if (st == FA_OK) {
            k_commit_rows<<<B, kThreads, 0, s>>>(L, k, commit_lo, commit_hi, marg, F(p.conf), committed, row_status,
                                                 commit_idx, tokens, (unsigned long long *)(ws + p.keys));
            st = launch_check("commit");
        }
    }
    stage_mark(4, s);
    return st;
}
}  // namespace

extern "C" fa_status fa_profile_enable(int32_t enable) {
    if (enable && !g_stage.created) {
        for (int i = 0; i <= FA_N_STAGES; ++i) {
            cudaError_t e = cudaEventCreate(&g_stage.ev[i]);
            if (e != cudaSuccess) { fa_set_error(std::string("fa_profile_enable: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
        }
        g_stage.created = true;
    }
    g_stage.enabled = enable != 0;
    return FA_OK;
}

extern "C" fa_status fa_profile_read(float *ms) {
    if (!ms) { fa_set_error("fa_profile_read: NULL argument"); return FA_ERR_INVALID_ARG; }
    if (!g_stage.created) { fa_set_error("fa_profile_read: profiling never enabled"); return FA_ERR_INVALID_ARG; }
    cudaError_t e = cudaEventSynchronize(g_stage.ev[FA_N_STAGES]);
    if (e != cudaSuccess) { fa_set_error(std::string("fa_profile_read: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    for (int i = 0; i < FA_N_STAGES; ++i) {
        e = cudaEventElapsedTime(&ms[i], g_stage.ev[i], g_stage.ev[i + 1]);
        if (e != cudaSuccess) { fa_set_error(std::string("fa_profile_read: ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    }
    return FA_OK;
}

extern "C" fa_status fa_launch_count(uint64_t *n) {
    if (!n) { fa_set_error("fa_launch_count: NULL argument"); return FA_ERR_INVALID_ARG; }
    *n = g_launches.load(std::memory_order_relaxed);
    return FA_OK;
}

extern "C" fa_status fa_apply_commits(int32_t B, int32_t L, int32_t k, const int32_t *commit_idx, const int32_t *tokens,
                                      int32_t *committed, fa_stream stream) {
    if (B < 0 || L < 0 || k < 0) { fa_set_error("fa_apply_commits: B, L or k negative"); return FA_ERR_INVALID_ARG; }
    if ((long)B * k == 0) return FA_OK;
    if (!commit_idx || !tokens || !committed) { fa_set_error("fa_apply_commits: NULL buffer"); return FA_ERR_INVALID_ARG; }
    const long n = (long)B * k;
    k_apply_commits<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(B, L, k, commit_idx, tokens, committed);
    return launch_check("apply commits");
}
