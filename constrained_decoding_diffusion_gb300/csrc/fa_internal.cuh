// Internal definitions shared by the compile and step translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstring>
#include <string>
#include <vector>

#include "../../include/fa.h"

// ----------------------------------------------------------------------------- host side

// A compiled automaton: the canonical arrays (exported bit-exact by fa_export_csr) plus
// the kernel-facing "cell" layout.  A cell is a distinct (src, dst) pair; its token list is
// the sorted multiset union of the label sets of all edges src -> dst, so the cell's sum of
// token weights is exactly M_t(src, dst) (parallel edges add, as NFA path counting needs).
struct fa_automaton {
    int32_t S = 0, V = 0, E = 0, start = 0, n_accept = 0, is_dfa = 0, device = 0;
    int64_t I = 0;
    int32_t n_cells = 0;
    int32_t max_cell_len = 0;
    // canonical arrays (device)
    int64_t *lab_off = nullptr;
    int32_t *lab_tok = nullptr;
    int32_t *src_off = nullptr, *src_edges = nullptr;
    int32_t *dst_off = nullptr, *dst_edges = nullptr;
    int64_t *tok_off = nullptr;
    int32_t *tok_edges = nullptr;
    int32_t *accept = nullptr;       // [n_accept] ascending
    int32_t *accept_mask = nullptr;  // [S] 0/1
    int32_t *edge_src = nullptr, *edge_dst = nullptr;
    // (src << 16) | dst of every incidence, token-major: tokens in the order tok_perm (by
    // incidence count, ties by id), interleaved by groups of 32: row k of group g (rows
    // tok_goff[g] .. tok_goff[g + 1]) holds incidence k of token tok_perm[32 g + lane] at
    // tok_sd[32 * row + lane], (|S|, |S|) past a token's count, so a warp reading one row
    // reads 128 contiguous bytes
    uint32_t *tok_sd = nullptr;
    int64_t *tok_goff = nullptr;     // [ceil(V / 32) + 1]
    int32_t *tok_perm = nullptr;     // [V]
    // cells (device), sorted by (src, dst)
    int32_t *row_cell_off = nullptr;  // [S+1]
    int32_t *cell_dst = nullptr;      // [n_cells]
    int32_t *cell_src = nullptr;      // [n_cells]
    int64_t *cell_off = nullptr;      // [n_cells+1]
    int32_t *cell_tok = nullptr;      // [I]
    // reweight layout ("runs", built in fa_compile).  The vocabulary is read in chunks of
    // chunk_tokens tokens staged in shared memory.  Every cell's sorted token list is cut
    // into runs (run q of nr takes tokens q, q + nr, ...); a run belongs to one lane of one
    // warp unit and owns one accumulator slot.  Unit u's entries for chunk c are 8-byte
    // groups of FA_GROUP_ENTRIES uint16 entries at ru_goff[u*n_chunks+c] + 32 k + lane
    // (k = 0, 1, ...): bits 0-14 give the in-chunk token index (chunk_tokens + j for j <
    // FA_PAD_SLOTS = a zero pad slot, one per shared-memory bank, so the lanes of one step
    // read distinct banks or one shared pad address); a run's entries fill whole groups, and
    // bit 15 of a group's first entry says that the group ends the lane's current run (every
    // run ends exactly once per chunk, so slot j of a lane is its j-th run).  A lane's slot j is at FA_UNIT_SLOTS * (unit - row_unit0[row]) + 32 j + lane
    // relative to the first unit of the row's group; cell x adds the slots
    // crun_slot[crun_off[x] .. crun_off[x+1]] in order.
    int32_t chunk_tokens = 0, n_chunks = 1, n_units = 0;
    uint16_t *ru_tok = nullptr;
    int32_t *ru_goff = nullptr, *row_unit0 = nullptr, *crun_off = nullptr;
    uint16_t *crun_slot = nullptr;
    // per cell {s * |S| + dst, its slot relative to the unit array (FA_UNIT_SLOTS * row_unit0[s]
    // + crun_slot) when the cell is one run, else -1}: one coalesced load per cell
    int2 *cell_rec = nullptr;
    // row blocks for the reweight grid: partition p holds part_count[p] blocks of whole rows
    // (at most FA_RW_MAX_UNITS, 32, 16, ..., 1 units each for p = 0, 1, 2, ..., unless one row
    // group needs more); block i of partition p is rb_meta[8 * (part_first[p] + i) ..] =
    // {r0, r1, u0, u1, c0, c1, 0, 0}, launched with min(32 FA_RW_WARPS, max(256,
    // 32 part_max_units[p])) threads, a warp walking up to three units.
    int32_t *rb_meta = nullptr;
    std::vector<int32_t> part_first, part_count, part_max_units, part_max_rows;
    // per partition, the largest block's unit totals plus its rows of M_t, in floats
    std::vector<int64_t> part_tile_floats;
    void *blob = nullptr;  // one device allocation holding every array above
    size_t blob_bytes = 0;
};

void fa_set_error(const std::string &msg);

// ----------------------------------------------------------------------------- device side

#define FA_INT_NONE (-2147483647 - 1)
#ifndef FA_REWEIGHT_MAX_CHUNK
#define FA_REWEIGHT_MAX_CHUNK 24576  // tokens per staged vocabulary chunk
#endif
#define FA_RUN_END 0x8000u           // flag on a group's first entry: the group ends the lane's run
#define FA_GROUP_ENTRIES 4           // entries per 8-byte group; runs end only at group ends
#define FA_PAD_SLOTS 32              // zero slots after a staged chunk, one per shared-memory bank
#ifndef FA_RUN_SLOTS
#define FA_RUN_SLOTS 8               // runs (accumulator slots) per lane
#endif
#define FA_UNIT_SLOTS (32 * FA_RUN_SLOTS)
#define FA_RW_WARPS 16               // warps per reweight block (two blocks per SM)
#define FA_RW_MAX_UNITS 48           // warp units per reweight block: a warp walks up to three

// floor(log2 x) of a positive normal float from its exponent field (subnormals give -127).
__device__ __forceinline__ int fa_exponent(float x) {
    return ((__float_as_int(x) >> 23) & 0xff) - 127;
}

// x * 2^d exactly (up to flush of results below the fp32 subnormal range).
__device__ __forceinline__ float fa_scale_pow2(float x, int d) {
    if (d < -300) return 0.0f;
    if (d > 254) d = 254;
    return ldexpf(x, d);
}

// 2^d for an integer d <= 127 (0 below the subnormal range).
__device__ __forceinline__ float fa_pow2(int d) {
    if (d >= -126) return __int_as_float((d + 127) << 23);
    if (d >= -149) return __int_as_float(1 << (d + 149));
    return 0.0f;
}

// x * 2^d for any integer d (the common case |d| <= 126 is one multiply).
__device__ __forceinline__ float fa_mul_pow2(float x, int d) {
    if (d >= -126 && d <= 127) return x * __int_as_float((d + 127) << 23);
    return ldexpf(x, max(min(d, 300), -300));
}

// Split x > 0 into m in [1, 2) and integer e with x = m * 2^e (normal or subnormal x).
__device__ __forceinline__ void fa_split(float x, float &m, int &e) {
    int bits = __float_as_int(x);
    int ex = (bits >> 23) & 0xff;
    if (ex == 0) {  // subnormal: renormalise
        x *= 16777216.0f;  // 2^24
        bits = __float_as_int(x);
        ex = ((bits >> 23) & 0xff) - 24;
    }
    e = ex - 127;
    m = __int_as_float((bits & 0x807fffff) | 0x3f800000);
}

// The bit pattern of a float and back (host and device).
__host__ __device__ __forceinline__ uint32_t fa_f32_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return u;
}
__host__ __device__ __forceinline__ float fa_bits_f32(uint32_t u) {
    float x;
    memcpy(&x, &u, sizeof x);
    return x;
}

// The operand split of the tensor-core span products: x = p1 + p2 + p3 with bf16 parts (each
// the upper 16 bits of a float).  p1 keeps x's leading 8 significant bits, p2 the leading 8 of
// the remainder r = x - p1 and p3 = r - p2, which has at most 8 significant bits left; both
// subtractions are exact in fp32, so the parts sum to x exactly (a subnormal p3 keeps its top
// bits only, a loss below 2^-133).  Returns the three bf16 bit patterns in the low halves.
__host__ __device__ __forceinline__ void fa_split_bf16x3(float x, uint32_t &b1, uint32_t &b2, uint32_t &b3) {
    const uint32_t u = fa_f32_bits(x);
    const float r = x - fa_bits_f32(u & 0xFFFF0000u);
    const uint32_t ur = fa_f32_bits(r);
    const float r2 = r - fa_bits_f32(ur & 0xFFFF0000u);
    b1 = u >> 16;
    b2 = ur >> 16;
    b3 = fa_f32_bits(r2) >> 16;
}

// Pieces of the host-input copies of fa_constrained_step_host: bounds bound[0] = 0 <
// bound[1] < ... < bound[n] = P over the batch's P positions, n <= FA_HOST_PIECES (n = 0 for
// P = 0).  The first piece is P / 32 positions (at least one), each next one 1.4 times the
// last, so that a piece's copy lands while the previous piece is reweighted (for a copy up
// to 1.4 times slower per position than the reweighting), and the last piece is the rest.
#define FA_HOST_PIECES 8
inline int fa_host_pieces(size_t P, size_t (&bound)[FA_HOST_PIECES + 1]) {
    int n = 0;
    bound[0] = 0;
    double len = (double)(P / 32 > 0 ? P / 32 : 1);
    while (bound[n] < P) {
        const size_t next = bound[n] + (size_t)len;
        bound[n + 1] = (n == FA_HOST_PIECES - 1 || next > P) ? P : next;
        ++n;
        len *= 1.4;
    }
    return n;
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): a counter-based generator; one call
// maps (counter, key) to four independent 32-bit words.
struct fa_u4 { uint32_t x, y, z, w; };

__device__ __forceinline__ fa_u4 fa_philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                           uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    return fa_u4{c0, c1, c2, c3};
}

// Uniform in [0, 1) with 24 random bits for draw `idx` of sequence b and purpose p.
// The counter is (idx, b, offset<<2 | p, offset>>30): distinct for every draw of one step and
// for every offset below 2^62.
enum { FA_RNG_ROOT = 0, FA_RNG_MID = 1, FA_RNG_LEAF = 2 };

__device__ __forceinline__ float fa_uniform(uint64_t seed, uint64_t offset, uint32_t idx, uint32_t b,
                                            uint32_t purpose) {
    fa_u4 r = fa_philox(idx, b, (uint32_t)(offset << 2) | purpose, (uint32_t)(offset >> 30),
                        (uint32_t)seed, (uint32_t)(seed >> 32));
    return (float)(r.x >> 8) * (1.0f / 16777216.0f);
}

__device__ __forceinline__ float fa_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int fa_warp_max_int(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// An extended-range non-negative number acc * 2^E accumulated term by term (acc is kept
// near [1, 2^24) so no term below the fp32 range of the running maximum is lost).
struct fa_xacc {
    float acc;
    int E;
    __device__ __forceinline__ void init() { acc = 0.0f; E = FA_INT_NONE; }
    // add m * 2^e with m in [0.5, 4)
    __device__ __forceinline__ void add(float m, int e) {
        if (m <= 0.0f) return;
        if (E == FA_INT_NONE) { acc = m; E = e; return; }
        if (e > E) { acc = fa_scale_pow2(acc, E - e) + m; E = e; }
        else acc += fa_scale_pow2(m, e - E);
    }
    __device__ __forceinline__ void merge(float m2, int e2) {
        if (e2 == FA_INT_NONE || m2 <= 0.0f) return;
        if (E == FA_INT_NONE) { acc = m2; E = e2; return; }
        if (e2 > E) { acc = fa_scale_pow2(acc, E - e2) + m2; E = e2; }
        else acc += fa_scale_pow2(m2, e2 - E);
    }
    __device__ __forceinline__ void warp_reduce() {
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            float m2 = __shfl_xor_sync(0xffffffffu, acc, o);
            int e2 = __shfl_xor_sync(0xffffffffu, E, o);
            merge(m2, e2);
        }
    }
    // normalise to mantissa in [1, 2) (or 0 with exponent 0)
    __device__ __forceinline__ void normalised(float &m, int &e) const {
        if (E == FA_INT_NONE || acc <= 0.0f) { m = 0.0f; e = 0; return; }
        int ee;
        float mm;
        fa_split(acc, mm, ee);
        m = mm;
        e = E + ee;
    }
};

// Tensor-core span products (fa_span_tc.cu).
bool fa_span_tc_supported(int S);
size_t fa_span_tc_image_bytes(int S, long products);
fa_status fa_span_tc_level(int S, int B, int L, int k, int nk, const float *mant_c, const int32_t *rho_c,
                           const int32_t *rmax_c, const int32_t *rminc_c, int nc, const int32_t *mu, float *mant_p,
                           int32_t *rho_p, int32_t *rmax_p, int32_t *rminc_p, int32_t *err, int32_t *range_lost,
                           void *img, cudaStream_t stream, const int32_t *fflag_p = nullptr,
                           const int32_t *fmap_p = nullptr);
