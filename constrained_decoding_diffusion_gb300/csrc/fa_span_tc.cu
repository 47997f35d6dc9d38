// Span products on the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// One tree level of the up-sweep of the paperfeed.app summary of "Constrained Decoding for
// Diffusion Language Models via Efficient Inference over Finite Automata" ("The scan trick":
// 2^k-step transition matrices from two 2^(k-1)-step ones by batched matrix products; the
// papernotes.org notes, key design 2): C = A_L * A_R for every node, in the per-row exponent
// format of fa_step.cu.  The left operand is prescaled per (row, m) by 2^(rhoR[m] - mu[row])
// (mu from the row-shift kernel) and both operands are split into three bf16 parts,
// x = p1 + p2 + p3 exactly (p1 the leading 8 significant bits, p2 the next 8 of the remainder,
// p3 the rest), so the six products p1q1, p1q2, p2q1, p1q3, p2q2, p3q1 on the bf16 tensor
// cores (fp32 accumulation) keep fp32 accuracy; the three dropped terms are below 2^-22 of
// the product.  Against a two-part TF32 split (hi*hi + hi*lo + lo*hi at half the bf16 rate)
// the tensor work is the same and the operand images are 6 instead of 8 bytes per element.
//
// Two kernels per tree level.  k_tc_prep converts every operand once: the left child, row
// prescaled, and the right child are split into their parts and written as the exact images
// of the shared-memory tiles the MMAs read (canonical K-major no-swizzle layout: 8-row x
// 16-byte core matrices of 8 bf16, K-direction core stride 128 B, row-group stride 256 B;
// 128x16 left tiles, 256x16 right tiles, the three parts one after the other).  k_span_tc is
// persistent (one CTA per SM, walking the level's 128x256 output tiles) and warp-specialised:
// one producer thread streams the tile images of each K step (36 KB) into one of six
// shared-memory stages, tracked by the stage's "full" mbarrier; one thread issues the six
// MMAs (M=128, N=256, K=16) and commits them to the stage's "empty" mbarrier, which releases
// the stage to the producer; sixteen epilogue warps empty the accumulators.  K steps
// alternate between two tensor-memory accumulators (128 lanes x 256 fp32 columns each): the
// tensor cores' fp32 accumulation truncates, so each chain of additions is kept half as long
// and the two are added with round-to-nearest in the epilogue, which reads them into
// registers and hands tensor memory back to the MMA thread before it writes the tile
// row-major with its row maxima.  The stages keep loading across tile boundaries, so a
// tile's pipeline fill and the previous tile's stores overlap its MMAs.
//
// Every mbarrier wait is bounded (about a second); a wait that runs out records
// FA_ROW_TIMEOUT in the error word, tensor memory is released and the CTA returns.  The
// pipeline waits also give up as soon as the other role has failed, while the waits that
// drain work already issued (the producer's last bulk copies, the MMAs before the final
// commit) keep the long limit: that work completes on its own, and no CTA may leave while a
// copy can still land in its shared memory or an MMA still reads it.
#include <stdint.h>

#include <atomic>
#include <cfloat>

#include "fa_internal.cuh"

namespace {

constexpr int TM = 128, TN = 256, TK = 16, NTHR = 256;
constexpr int NEPI = 16;                    // epilogue warps of the product kernel (64 columns each)
constexpr int NTHR_P = 32 * (2 + NEPI);     // producer warp, MMA warp, epilogue warps
constexpr uint32_t TMEM_COLS = 512;   // two 256-column accumulators
constexpr long long kSpinCycles = 2000000000LL;
constexpr long long kInjectCycles = 1LL << 20;   // the injected wait of a failure test (~0.5 ms)
constexpr int PREP_KT = 256 / TK;           // K steps converted per k_tc_prep block (256 columns)

// Operand format of the products: each operand is split into three bf16 parts,
// x = p1 + p2 + p3 exactly, and a product takes six kind::f16 MMAs (K = 16, both operands
// bf16) per 16 K-columns: p1q1 + p1q2 + p2q1 + p1q3 + p2q2 + p3q1, the dropped terms below
// 2^-22 of the product.  A K step's image holds the three parts one after the other.
constexpr int PARTS = 3;
constexpr int A_PART = TM * TK * 2;         // one bf16 part of a 128x16 left tile (4 KB)
constexpr int B_PART = TN * TK * 2;         // one bf16 part of a 256x16 right tile (8 KB)
constexpr int A_IMG = PARTS * A_PART, B_IMG = PARTS * B_PART;
constexpr int STAGE_BYTES = A_IMG + B_IMG;  // 36 KB
constexpr int NSTAGE = 6;                   // five stages in flight while one is multiplied
constexpr uint32_t KGRP = TK * 2 * 8;       // bytes of one 8-row group (8 rows x 16 bf16)

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// tcgen05 shared-memory matrix descriptor: start address, leading (K-direction) and stride
// (8-row group) byte offsets, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
    d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B both bf16 (format 1), both K-major,
// M = 128, N = 256.
__host__ __device__ constexpr uint32_t umma_idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait (about a second of SM clock by default); false when the limit ran out or,
// given abort, when another thread of the CTA has flagged a failure
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit = kSpinCycles,
                                          const volatile int *abort = nullptr) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (abort && *abort) return false;
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// one-dimensional bulk copy global -> shared, completing bytes on the mbarrier
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
        "[%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// byte offset of element (row, k) in one part of a K-major no-swizzle tile with TK K-columns
// (8-row x 16-byte core matrices of 8 bf16, K-direction core stride 128 B, row-group stride KGRP)
__device__ __forceinline__ uint32_t kmaj_off(int row, int k) {
    return (uint32_t)((row >> 3) * KGRP + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// the three bf16 parts of eight consecutive K-columns as one 16-byte core-matrix row per part
__device__ __forceinline__ void pack_bf16x3(const float (&x)[8], uint4 &q1, uint4 &q2, uint4 &q3) {
    uint32_t w1[4], w2[4], w3[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a1, a2, a3, c1, c2, c3;
        fa_split_bf16x3(x[2 * j], a1, a2, a3);
        fa_split_bf16x3(x[2 * j + 1], c1, c2, c3);
        w1[j] = a1 | (c1 << 16);
        w2[j] = a2 | (c2 << 16);
        w3[j] = a3 | (c3 << 16);
    }
    q1 = make_uint4(w1[0], w1[1], w1[2], w1[3]);
    q2 = make_uint4(w2[0], w2[1], w2[2], w2[3]);
    q3 = make_uint4(w3[0], w3[1], w3[2], w3[3]);
}

// Operand images for one level.  Blocks: (product, side, tile, chunk of PREP_KT K steps);
// side 0 = left operand (prescaled by 2^(rhoR[m] - mu[row]), 128-row tiles), side 1 = right
// operand (256-column tiles, transposed to K-major).
__global__ void __launch_bounds__(NTHR) k_tc_prep(int S, int L, int k, int nk, const float *__restrict__ mant_c,
                                                const int32_t *__restrict__ rho_c,
                                                const int32_t *__restrict__ rmax_c,
                                                const int32_t *__restrict__ rminc_c, int nc,
                                                const int32_t *__restrict__ mu, unsigned char *img,
                                                int32_t *range_lost, const int32_t *__restrict__ fflag_p) {
    const int tid = threadIdx.x;
    const int tiles_m = (S + TM - 1) / TM, tiles_n = (S + TN - 1) / TN, nkt = (S + TK - 1) / TK;
    const int per = tiles_m + tiles_n;
    const int kch = (nkt + PREP_KT - 1) / PREP_KT;                 // K-step chunks per tile
    const int kc = blockIdx.x % kch;
    const long flat = blockIdx.x / kch;
    const int w = (int)(flat % per);
    const long bn = flat / per;
    const int kt0 = kc * PREP_KT, kt1 = min(nkt, kt0 + PREP_KT);
    const int node = (int)(bn % nk), b = (int)(bn / nk);
    if (((2 * node + 1) << (k - 1)) >= L) return;     // a copy, no product
    if (fflag_p && fflag_p[bn]) return;               // a functional span: no product either
    const size_t SS = (size_t)S * S;
    const size_t pnode = (size_t)b * nk + node;
    const size_t lnode = (size_t)b * nc + 2 * node, rnode = lnode + 1;
    const size_t per_prod_a = (size_t)tiles_m * nkt * A_IMG, per_prod_b = (size_t)tiles_n * nkt * B_IMG;
    const size_t total_a = (size_t)gridDim.x / ((size_t)per * kch) * per_prod_a;  // left images come first
    if (w < tiles_m) {
        // two threads per row, eight consecutive K-columns each
        const int tm = w, row = tid >> 1, gi = tm * TM + row, kk0 = (tid & 1) * (TK / 2);
        const float *A = mant_c + lnode * SS;
        const int32_t *rhoR = rho_c + rnode * S, *rmaxR = rmax_c + rnode * S, *rmincR = rminc_c + rnode * S;
        const int mrow = gi < S ? mu[pnode * S + gi] : FA_INT_NONE;
        unsigned char *base = img + (size_t)bn * per_prod_a + (size_t)tm * nkt * A_IMG;
        int lost = 0;
        for (int kt = kt0; kt < kt1; ++kt) {
            unsigned char *t = base + (size_t)kt * A_IMG;
            float y[TK / 2];
#pragma unroll
            for (int q = 0; q < TK / 8; ++q) {
                const int m0 = kt * TK + kk0 + 4 * q;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (gi < S && m0 < S) v = __ldg(reinterpret_cast<const float4 *>(A + (size_t)gi * S + m0));
                const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = m0 + e;
                    float yy = 0.0f;
                    if (x[e] > 0.0f && mrow != FA_INT_NONE && m < S && __ldg(rmaxR + m) > 0) {
                        const int d = __ldg(rhoR + m) - mrow;
                        // below the normal range after the prescale, alone or times the right
                        // row's smallest entry: mass may be lost
                        const int rn = __ldg(rmincR + m);
                        const int emin = rn > 0 ? min(0, fa_exponent(__int_as_float(0x7fffffff - rn))) : 0;
                        if (fa_exponent(x[e]) + d + emin < -126) lost = 1;
                        yy = fa_mul_pow2(x[e], d);
                    }
                    y[4 * q + e] = yy;
                }
            }
            uint4 q1, q2, q3;
            pack_bf16x3(y, q1, q2, q3);
            const uint32_t off = kmaj_off(row, kk0);
            *reinterpret_cast<uint4 *>(t + off) = q1;
            *reinterpret_cast<uint4 *>(t + A_PART + off) = q2;
            *reinterpret_cast<uint4 *>(t + 2 * A_PART + off) = q3;
        }
        if (__any_sync(0xffffffffu, lost) && (tid & 31) == 0) atomicOr(range_lost + b, 1);
    } else {
        // one thread per column, the K step's 16 rows of the right operand
        const int tn = w - tiles_m, n = tid, gj = tn * TN + n;
        const float *Bm = mant_c + rnode * SS;
        unsigned char *base = img + total_a + (size_t)bn * per_prod_b + (size_t)tn * nkt * B_IMG;
        for (int kt = kt0; kt < kt1; ++kt) {
            unsigned char *t = base + (size_t)kt * B_IMG;
            float x[TK];
#pragma unroll
            for (int e = 0; e < TK; ++e) {
                const int m = kt * TK + e;
                x[e] = (gj < S && m < S) ? __ldg(Bm + (size_t)m * S + gj) : 0.0f;
            }
#pragma unroll
            for (int h = 0; h < TK / 8; ++h) {
                float xx[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) xx[e] = x[8 * h + e];
                uint4 q1, q2, q3;
                pack_bf16x3(xx, q1, q2, q3);
                const uint32_t off = kmaj_off(n, 8 * h);
                *reinterpret_cast<uint4 *>(t + off) = q1;
                *reinterpret_cast<uint4 *>(t + B_PART + off) = q2;
                *reinterpret_cast<uint4 *>(t + 2 * B_PART + off) = q3;
            }
        }
    }
}

// Persistent product kernel: one CTA per SM walks the level's output tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... with three roles.  Warp 0 (one thread) streams the
// tile images of every K step into the shared-memory stages ("full" barriers); warp 1 (one
// thread) waits for the accumulators to be free ("acc_empty"), issues the MMAs of a tile,
// releases each stage with a commit to its "empty" barrier and, after the tile's last K step,
// commits to "acc_full"; warps 2-17 (the epilogue, four per tensor-memory lane quarter, 64
// columns each) wait for "acc_full", read both accumulators into registers, add them, arrive
// on "acc_empty" and only then store the tile and its row maxima, so the stores and the next
// tile's first loads overlap the next tile's MMAs.  Copy tiles (right child padding) and
// functional tiles take no MMAs: the epilogue warps write them.  The stage and accumulator
// phases run on across tiles.  Eighteen warps leave 96 registers a thread (five warps on
// some of the four sub-partitions, 16 K registers each).
__global__ void __launch_bounds__(NTHR_P, 1) k_span_tc(int S, int L, int k, int nk, const float *__restrict__ mant_c,
                                           const int32_t *__restrict__ rho_c, const int32_t *__restrict__ rmax_c,
                                           const int32_t *__restrict__ rminc_c, int nc,
                                           const int32_t *__restrict__ mu, const unsigned char *__restrict__ img,
                                           float *mant_p, int32_t *rho_p, int32_t *rmax_p, int32_t *rminc_p,
                                           int32_t *err, int inject_timeout, const int32_t *__restrict__ fflag_p,
                                           const int32_t *__restrict__ fmap_p, long n_prod) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint64_t full[NSTAGE], empty[NSTAGE], acc_full, acc_empty, done, never;
    __shared__ uint32_t tmem_base_s;
    __shared__ int fail_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles_m = (S + TM - 1) / TM, tiles_n = (S + TN - 1) / TN, nkt = (S + TK - 1) / TK;
    const long n_tiles = n_prod * tiles_m * tiles_n;
    const size_t SS = (size_t)S * S;
    const size_t per_prod_a = (size_t)tiles_m * nkt * A_IMG, per_prod_b = (size_t)tiles_n * nkt * B_IMG;
    // what a tile is: 0 = product, 1 = copy of the left child, 2 = functional span
    auto tile_kind = [&](long t, long &bn, int &node, int &b, int &tm, int &tn) {
        tn = (int)(t % tiles_n);
        tm = (int)((t / tiles_n) % tiles_m);
        bn = t / ((long)tiles_n * tiles_m);
        node = (int)(bn % nk);
        b = (int)(bn / nk);
        if (((2 * node + 1) << (k - 1)) >= L) return 1;
        if (fflag_p && fflag_p[bn]) return 2;
        return 0;
    };
    if (tid == 0) {
        for (int s2 = 0; s2 < NSTAGE; ++s2) { mbar_init(&full[s2], 1); mbar_init(&empty[s2], 1); }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, NEPI * 32);
        mbar_init(&done, 1);
        mbar_init(&never, 1);   // nothing ever arrives here: the target of an injected wait
        fail_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    if (tid == 0) {
        // producer: the operand images of every K step of every product tile, in order
        long it = 0, issued = 0;
        for (long t = blockIdx.x; t < n_tiles && !fail_s; t += gridDim.x) {
            long bn;
            int node, b, tm, tn;
            if (tile_kind(t, bn, node, b, tm, tn) != 0) continue;
            const unsigned char *a_img = img + (size_t)bn * per_prod_a + (size_t)tm * nkt * A_IMG;
            const unsigned char *b_img = img + n_prod * per_prod_a + (size_t)bn * per_prod_b + (size_t)tn * nkt * B_IMG;
            for (int kt = 0; kt < nkt; ++kt, ++it) {
                const int st = (int)(it % NSTAGE);
                if (it >= NSTAGE && !mbar_wait(&empty[st], (uint32_t)((it / NSTAGE) - 1) & 1, kSpinCycles, &fail_s)) {
                    atomicExch(&fail_s, 1);
                    break;
                }
                unsigned char *stage = smem + st * STAGE_BYTES;
                mbar_expect_tx(&full[st], STAGE_BYTES);
                bulk_g2s(stage, a_img + (size_t)kt * A_IMG, A_IMG, &full[st]);
                bulk_g2s(stage + A_IMG, b_img + (size_t)kt * B_IMG, B_IMG, &full[st]);
                issued = it + 1;
            }
        }
        // the last phase issued on each stage has landed before the CTA may leave (already
        // true unless a wait failed; the copies complete on their own, so the long limit)
        for (long q = issued > NSTAGE ? issued - NSTAGE : 0; q < issued; ++q)
            (void)mbar_wait(&full[q % NSTAGE], (uint32_t)(q / NSTAGE) & 1);
    } else if (tid == 32) {
        // MMA issuer
        const uint32_t idesc = umma_idesc_bf16();
        // failure test: a short wait on a barrier nothing completes runs out
        if (inject_timeout && !mbar_wait(&never, 0, kInjectCycles)) atomicExch(&fail_s, 1);
        long it = 0, tcount = 0;
        for (long t = blockIdx.x; t < n_tiles && !fail_s; t += gridDim.x) {
            long bn;
            int node, b, tm, tn;
            if (tile_kind(t, bn, node, b, tm, tn) != 0) continue;
            // the epilogue has read the previous tile's accumulators
            if (tcount > 0 && !mbar_wait(&acc_empty, (uint32_t)(tcount - 1) & 1, kSpinCycles, &fail_s)) {
                atomicExch(&fail_s, 1);
                break;
            }
            tc_fence_after();
            bool ok = true;
            for (int kt = 0; kt < nkt; ++kt, ++it) {
                const int st = (int)(it % NSTAGE);
                if (!mbar_wait(&full[st], (uint32_t)(it / NSTAGE) & 1, kSpinCycles, &fail_s)) {
                    atomicExch(&fail_s, 1);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a1 = smem_u32(smem + st * STAGE_BYTES), b1 = a1 + A_IMG;
                const uint32_t dacc = tmem + (uint32_t)(kt & 1) * TN;
                // 16 K-columns = two 128-byte core matrices per 8-row group: one MMA per term
                const uint32_t a2 = a1 + A_PART, a3 = a2 + A_PART;
                const uint32_t b2 = b1 + B_PART, b3 = b2 + B_PART;
                auto da = [](uint32_t x) { return umma_desc(x, 128, KGRP); };
                umma_bf16(dacc, da(a1), da(b1), idesc, kt < 2 ? 0u : 1u);
                umma_bf16(dacc, da(a1), da(b2), idesc, 1u);
                umma_bf16(dacc, da(a2), da(b1), idesc, 1u);
                umma_bf16(dacc, da(a1), da(b3), idesc, 1u);
                umma_bf16(dacc, da(a2), da(b2), idesc, 1u);
                umma_bf16(dacc, da(a3), da(b1), idesc, 1u);
                umma_commit(&empty[st]);
            }
            if (!ok) break;
            umma_commit(&acc_full);
            ++tcount;
        }
        umma_commit(&done);   // completes once every MMA issued above has
    } else if (warp >= 2) {
        // epilogue: warp w reads tensor-memory lanes 32 * (w % 4) ... (its row quarter) and one
        // 64-column quarter of each accumulator
        const int et = tid - 64, q = warp & 3, cq = (warp - 2) >> 2;
        long tcount = 0;
        for (long t = blockIdx.x; t < n_tiles && !fail_s; t += gridDim.x) {
            long bn;
            int node, b, tm, tn;
            const int kind = tile_kind(t, bn, node, b, tm, tn);
            const int i0 = tm * TM, j0 = tn * TN;
            const size_t pnode = (size_t)b * nk + node;
            const size_t lnode = (size_t)b * nc + 2 * node;
            float *C = mant_p + pnode * SS;
            if (kind == 1) {                                  // right child is padding: C = A_L
                const float *A = mant_c + lnode * SS;
                for (int qq = et; qq < TM * TN; qq += NEPI * 32) {
                    const int r = i0 + qq / TN, c = j0 + qq % TN;
                    if (r < S && c < S) C[(size_t)r * S + c] = A[(size_t)r * S + c];
                }
                if (tn == 0)
                    for (int r = i0 + et; r < min(i0 + TM, S); r += NEPI * 32) {
                        rho_p[pnode * S + r] = rho_c[lnode * S + r];
                        rmax_p[pnode * S + r] = rmax_c[lnode * S + r];
                        rminc_p[pnode * S + r] = rminc_c[lnode * S + r];
                    }
                continue;
            }
            if (kind == 2) {
                // a functional span: the 0/1 matrix of its partial function, row exponents 0 --
                // what the product of the two 0/1 matrices gives -- written without the MMAs
                const int32_t *fm = fmap_p + pnode * S;
                for (int qq = et; qq < TM * TN; qq += NEPI * 32) {
                    const int r = i0 + qq / TN, c = j0 + qq % TN;
                    if (r < S && c < S) C[(size_t)r * S + c] = fm[r] == c ? 1.0f : 0.0f;
                }
                if (tn == 0)
                    for (int r = i0 + et; r < min(i0 + TM, S); r += NEPI * 32) {
                        const bool one = fm[r] >= 0;
                        rho_p[pnode * S + r] = 0;
                        rmax_p[pnode * S + r] = one ? __float_as_int(1.0f) : 0;
                        rminc_p[pnode * S + r] = one ? 0x7fffffff - __float_as_int(1.0f) : 0;
                    }
                continue;
            }
            if (!mbar_wait(&acc_full, (uint32_t)tcount & 1, kSpinCycles, &fail_s)) {
                atomicExch(&fail_s, 1);
                break;
            }
            tc_fence_after();
            // both accumulators of the thread's row and 64 columns, added, into registers
            float v[4][16];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * cq + 16 * c4);
                float v2[16];
                tmem_ld16(ta, v[c4]);
                tmem_ld16(ta + TN, v2);
#pragma unroll
                for (int e = 0; e < 16; ++e) v[c4][e] += v2[e];
            }
            tc_fence_before();
            mbar_arrive(&acc_empty);
            ++tcount;
            const int row = 32 * q + lane, gi = i0 + row;
            if (gi < S) {
                float mx = 0.0f, mn = FLT_MAX;
                const int col = 64 * cq;
                float *dst = C + (size_t)gi * S + j0 + col;
                const bool whole = j0 + col + 64 <= S;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const int c = 16 * c4 + e;
                        if (whole) {
                            *reinterpret_cast<float4 *>(dst + c) =
                                make_float4(v[c4][e], v[c4][e + 1], v[c4][e + 2], v[c4][e + 3]);
                        } else {
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                if (j0 + col + c + u < S) dst[c + u] = v[c4][e + u];
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float x = (whole || j0 + col + c + u < S) ? v[c4][e + u] : 0.0f;
                            mx = fmaxf(mx, x);
                            if (x > 0.0f) mn = fminf(mn, x);
                        }
                    }
                if (mx > 0.0f) {
                    atomicMax(&rmax_p[pnode * S + gi], __float_as_int(mx));
                    atomicMax(&rminc_p[pnode * S + gi], 0x7fffffff - __float_as_int(mn));
                }
                if (tn == 0 && cq == 0) {
                    const int mr = mu[pnode * S + gi];
                    rho_p[pnode * S + gi] = (mr == FA_INT_NONE) ? 0 : rho_c[lnode * S + gi] + mr;
                }
            }
        }
    }
    // everyone: the MMAs issued are complete (they complete on their own: the long limit)
    // before tensor memory is released
    if (!mbar_wait(&done, 0)) atomicExch(&fail_s, 1);
    tc_fence_after();
    __syncthreads();
    if (fail_s && tid == 0) atomicExch(err, FA_ROW_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace

size_t span_tc_smem() { return (size_t)NSTAGE * STAGE_BYTES; }

// Launches of k_span_tc still to take the injected wait (failure tests only).
static std::atomic<int> g_inject_timeouts{0};

extern "C" fa_status fa_debug_inject_wait_timeouts(int32_t n_launches) {
    if (n_launches < 0) { fa_set_error("fa_debug_inject_wait_timeouts: negative count"); return FA_ERR_INVALID_ARG; }
    g_inject_timeouts.store(n_launches);
    return FA_OK;
}

bool fa_span_tc_supported(int S) { return S >= 128 && (S % 4) == 0; }

size_t fa_span_tc_image_bytes(int S, long products) {
    const size_t tiles_m = (S + TM - 1) / TM, tiles_n = (S + TN - 1) / TN, nkt = (S + TK - 1) / TK;
    return (size_t)products * nkt * (tiles_m * A_IMG + tiles_n * B_IMG);
}

fa_status fa_span_tc_level(int S, int B, int L, int k, int nk, const float *mant_c, const int32_t *rho_c,
                           const int32_t *rmax_c, const int32_t *rminc_c, int nc, const int32_t *mu, float *mant_p,
                           int32_t *rho_p, int32_t *rmax_p, int32_t *rminc_p, int32_t *err, int32_t *range_lost,
                           void *img, cudaStream_t stream, const int32_t *fflag_p, const int32_t *fmap_p) {
    const size_t smem = span_tc_smem();
    cudaError_t e = cudaFuncSetAttribute(k_span_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) { fa_set_error(std::string("span product (tensor cores): ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    const long tiles_m = (S + TM - 1) / TM, tiles_n = (S + TN - 1) / TN;
    const long kch = ((S + TK - 1) / TK + PREP_KT - 1) / PREP_KT;
    k_tc_prep<<<(unsigned)((long)B * nk * (tiles_m + tiles_n) * kch), NTHR, 0, stream>>>(
        S, L, k, nk, mant_c, rho_c, rmax_c, rminc_c, nc, mu, (unsigned char *)img, range_lost, fflag_p);
    e = cudaGetLastError();
    if (e != cudaSuccess) { fa_set_error(std::string("operand images (tensor cores): ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    const long n_prod = (long)B * nk, n_tiles = n_prod * tiles_m * tiles_n;
    int dev = 0, n_sm = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || n_sm <= 0) { fa_set_error(std::string("span product (tensor cores): ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    const long grid = std::min<long>(n_tiles, n_sm);   // persistent: one CTA per SM
    int inject = 0;
    for (int n = g_inject_timeouts.load(); n > 0 && !inject;)
        if (g_inject_timeouts.compare_exchange_weak(n, n - 1)) inject = 1;
    k_span_tc<<<(unsigned)grid, NTHR_P, smem, stream>>>(S, L, k, nk, mant_c, rho_c, rmax_c, rminc_c, nc, mu,
                                                        (const unsigned char *)img, mant_p, rho_p, rmax_p, rminc_p,
                                                        err, inject, fflag_p, fmap_p, n_prod);
    e = cudaGetLastError();
    if (e != cudaSuccess) { fa_set_error(std::string("span product (tensor cores): ") + cudaGetErrorString(e)); return FA_ERR_CUDA; }
    return FA_OK;
}

