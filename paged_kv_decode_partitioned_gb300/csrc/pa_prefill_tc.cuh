// pa_prefill_tc.cuh -- paged prefix-prefill attention on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory) for GB300 (sm_103a).
//
// The operation (page: project_6 commit cd0d9e1, "qwen3_6_scripts", the
// prefix-prefill part of the paged_attn.py rewrite): a chunk of new tokens of
// each sequence attends to the sequence's whole cached context and, causally,
// to the chunk itself.  The chunk's K/V are already in the paged cache, so
// chunk row i of sequence s (n chunk tokens, L cached tokens) sits at
// position p = L - n + i and attends to cache tokens 0..p.  The pages' tile
// loop (matmul, softmax, matmul per key tile with the running max and sum of
// the online softmax) is what each Q tile of a CTA runs below.
//
// One CTA = NQ Q tiles of 128 query rows of one (sequence, KV head): row =
// chunk token x query head of the GQA group, so every row of the CTA uses
// every K/V tile it loads, and with two Q tiles each loaded K/V byte feeds
// 256 rows.  Warp roles (96 + 128 kSplit NQ threads):
//   warp 0     TMA producer of Q (once: a 4-D map whose box is the group's
//              heads x the CTA's chunk tokens) and of the K tiles of the
//              context (128 tokens, 192 at head_dim 64) through NK shared-
//              memory stages, one (16-row box, 64-element piece) per copy; the
//              last warp is the V producer, through its own NV stages, one
//              16-row box with all its pieces per copy (a cache map with the
//              row ahead of the piece), and zeroes the tail tile's rows past
//              the context.  Each lane looks up the block of one copy and
//              issues it, so a tile's copies go out in parallel.  Each CTA
//              starts its walk at its own tile and wraps around;
//   warp 1     tensor-memory owner and MMA issuer: for each Q tile, S_j =
//              Q K_j^T into the tile's S buffer in tensor memory and O += P_j
//              V_j with P read from tensor memory (the S buffer it was written
//              over) and O accumulating in tensor memory; the whole warp runs
//              a fixed issue sequence (the two tiles take turns, so each tile's
//              MMAs fill the gap of the other's softmax), each step waiting on
//              the one barrier it needs, and one elected lane issues each MMA;
//              a K (V) stage is released once every Q tile's QK (PV) has used it;
//   warps 2..  kSplit softmax warpgroups per Q tile (one by default: a thread
//              per row, on the row's tensor-memory lane; with two, each takes
//              half of the S columns of every row and the halves swap their
//              row maxima through shared memory): S -> causal mask -> scale ->
//              row max -> exp2 -> P (bf16 or f16) written back over the first
//              half of the thread's own S columns (on column pairs: three-input
//              max, packed f32x2 fma and add; at head_dim 128 the row's S stays
//              in registers between the max and the P pass); O is rescaled in
//              tensor memory only when a row's max grows by more than 2^8
//              (exponents stay below 2^8 in between and the final division by
//              the running sum is exact either way); finally O / l -> out.
// Every mbarrier wait is bounded; a role that gives up raises
// PA_DEV_WAIT_TIMEOUT and leaves its loop, in-flight copies and MMAs are
// waited for (bounded) and tensor memory is freed before the CTA exits.
#pragma once

#include "pa_launch.cuh"
#include "pa_tc05.cuh"

namespace pa {

// Softmax warpgroups per Q tile: 2 = each row's S columns split between two
// threads (which swap row maxima and sums), 1 = one thread per whole row.
// One is faster at both head_dims (10 warps instead of 18: the MMA warp shares
// its scheduler with two softmax warps instead of four, no max exchange, and
// 168 registers a thread instead of 96).
#ifndef PA_PREFILL_SPLIT_D64
#define PA_PREFILL_SPLIT_D64 1
#endif
#ifndef PA_PREFILL_SPLIT_D128
#define PA_PREFILL_SPLIT_D128 1
#endif
// Shared-memory stages of K and of V tiles per head_dim.
#ifndef PA_PREFILL_KSTAGES_D64
#define PA_PREFILL_KSTAGES_D64 3
#endif
#ifndef PA_PREFILL_VSTAGES_D64
#define PA_PREFILL_VSTAGES_D64 3
#endif
#ifndef PA_PREFILL_KSTAGES_D128
#define PA_PREFILL_KSTAGES_D128 2
#endif
#ifndef PA_PREFILL_VSTAGES_D128
#define PA_PREFILL_VSTAGES_D128 2
#endif
// P handed to the MMA warp in two halves, per head_dim.
#ifndef PA_PREFILL_HALFP_D64
#define PA_PREFILL_HALFP_D64 1
#endif
#ifndef PA_PREFILL_HALFP_D128
#define PA_PREFILL_HALFP_D128 0
#endif
// K/V tile width per head_dim.
#ifndef PA_PREFILL_N_D64
#define PA_PREFILL_N_D64 192
#endif
#ifndef PA_PREFILL_N_D128
#define PA_PREFILL_N_D128 128
#endif
// S buffers in tensor memory per Q tile, per head_dim (with two, a Q tile's
// next QK runs under its softmax; 2 x (2 N + head_dim) columns must fit 512).
#ifndef PA_PREFILL_SBUFS_D64
#define PA_PREFILL_SBUFS_D64 1
#endif
#ifndef PA_PREFILL_SBUFS_D128
#define PA_PREFILL_SBUFS_D128 1
#endif
// A CTA with one Q tile of rows takes the idle tile's tensor memory as a second
// S buffer when its (sequence, KV head) has at most DUAL_MAX_CTAS CTAs: one query
// head per KV head with 128-token chunks over 32K ran 750 -> 850 TFLOP/s; where
// the CTA shares its (sequence, KV head) with full ones (GQA 6, 128-token chunks)
// the faster walk cost the others more than it saved (1010 -> 775).
#ifndef PA_PREFILL_DUAL
#define PA_PREFILL_DUAL 1
#endif
#ifndef PA_PREFILL_DUAL_MAX_CTAS
#define PA_PREFILL_DUAL_MAX_CTAS 1
#endif
// The CTAs of one (sequence, KV head) start their context walk ROT_STEP tiles
// apart (per head_dim; 0: all at tile 0) when there are at least ROT_MIN_CTAS.
// At head_dim 128 the walks in step share each K/V tile's fetch through L2
// (+1-6 % over walks 37 tiles apart); at head_dim 64 the spread walks measured
// 3 % faster, and on CTA pairs the two are alike.
#ifndef PA_PREFILL_ROT_STEP_D64
#define PA_PREFILL_ROT_STEP_D64 37
#endif
#ifndef PA_PREFILL_ROT_STEP_D128
#define PA_PREFILL_ROT_STEP_D128 0
#endif
#ifndef PA_PREFILL_ROT_STEP_PAIR
#define PA_PREFILL_ROT_STEP_PAIR 37
#endif
#ifndef PA_PREFILL_ROT_MIN_CTAS
#define PA_PREFILL_ROT_MIN_CTAS 0
#endif
// Whole rows of at most 128 columns hold their S in registers between the passes.
#ifndef PA_PREFILL_REGROW
#define PA_PREFILL_REGROW 1
#endif

// Tile plan per head_dim.  A tcgen05.mma with M = 128 and K = 16 takes the
// tensor pipe 65 cycles at N = 128, 129 at N = 256 and 49 at N = 64 (bound by
// the 6 KB of shared-memory operands it reads: 0.65 of the peak rate), and
// every MMA costs the issuing warp the same, so the MMAs are kept wide:
// 128-token K/V tiles, 192 at head_dim 64 (its O is only 64 columns, so two Q
// tiles of S + O still fit 512 columns, and each MMA group does 1.5x the work
// for the same issue overhead: 736 -> 825 TFLOP/s when measured).  head_dim 64 / 128 run
// two Q tiles per CTA, each with one S buffer in tensor memory (the two tiles
// take turns on the tensor pipe).  head_dim 256 (its O alone takes 256
// columns) runs on CTA pairs (pa_prefill_pair.cuh); the one-Q-tile layout with
// two S buffers below is what it ran on single CTAs.
template <int D>
struct PrefillTcCfg {
    static constexpr int kQTiles = D <= 128 ? 2 : 1;
    static constexpr int kRows = 128 * kQTiles;                  // query rows per CTA
    static constexpr int kN = D <= 64 ? PA_PREFILL_N_D64 : (D <= 128 ? PA_PREFILL_N_D128 : 128);   // cache tokens per tile
    static constexpr int kSBufs =
        kQTiles == 2 ? (D <= 64 ? PA_PREFILL_SBUFS_D64 : PA_PREFILL_SBUFS_D128) : 2;   // S buffers per Q tile
    // K and V stages (their own producers and barriers; a third K stage at
    // head_dim 128 or a fourth at head_dim 64 measured no faster)
    static constexpr int kKStages = D <= 64 ? PA_PREFILL_KSTAGES_D64 : (D <= 128 ? PA_PREFILL_KSTAGES_D128 : 1);
    static constexpr int kVStages = D <= 64 ? PA_PREFILL_VSTAGES_D64 : (D <= 128 ? PA_PREFILL_VSTAGES_D128 : 1);
    static constexpr int kPieces = D / 64;
    static constexpr int kQPiece = kRows * 128;                  // bytes of one Q piece
    static constexpr int kQTileBytes = 128 * 128;                // one Q tile's rows in a piece
    static constexpr int kQBytes = kPieces * kQPiece;
    // K and V land one 16-token box per copy, all its pieces, as 8-token
    // groups: [group][piece][8 rows][128 B] (128-byte swizzled), a uniform
    // group stride of kPieces KB for both operands (K read K-major, V MN-major)
    static constexpr int kBoxBytes = kPieces * 2048;
    static constexpr int kTileBytes = (kN / 16) * kBoxBytes;     // K (or V) of one stage
    static constexpr int kKOffset = kQBytes;                          // K stages
    static constexpr int kVOffset = kKOffset + kKStages * kTileBytes;   // V stages
    static constexpr int kBarOffset = kVOffset + kVStages * kTileBytes;
    // barriers: q_full, vtail, mma_done, k_full[NK], k_empty[NK], v_full[NV],
    // v_empty[NV]; per Q tile s_full[2], p_full[2], s_free[2], o_full (the
    // first kSBufs of each pair in use), p_half; then the tensor-memory slot
    static constexpr int kTileBars = 8;
    static constexpr int kTileBarBytes = kTileBars * 8;
    static constexpr int kNumBars = 3 + 2 * kKStages + 2 * kVStages + kTileBars * kQTiles;
    static constexpr int kSlotOffset = kBarOffset + kNumBars * 8;
    // each Q tile's softmax runs in kSplit warpgroups, one per 1 / kSplit of
    // the S columns of every row; with two, they swap row maxima (two buffers
    // by tile parity) and, at the end, row sums through shared memory,
    // synchronised by mbarriers (xbar[2] and xend per Q tile, one arrive per
    // warp)
    static constexpr int kSplit = D <= 64 ? PA_PREFILL_SPLIT_D64 : PA_PREFILL_SPLIT_D128;
    static_assert(kSplit == 1 || kSplit == 2, "one or two softmax warpgroups per Q tile");
    static constexpr int kHalfCols = kN / kSplit;
    // With one S buffer and one softmax warpgroup, P can be handed over in two
    // halves (p_half after the P of the tile's first N / 2 tokens), so the
    // first half of the PV runs under the second half's exponentials: 4 %
    // faster at head_dim 64 (192-column rows), 1.6 % slower at head_dim 128
    // (the mid-pass store wait costs more than the overlap gains there).
    static constexpr bool kHalfP =
        kSBufs == 1 && kSplit == 1 && (D <= 64 ? PA_PREFILL_HALFP_D64 : PA_PREFILL_HALFP_D128);
    static constexpr int kXBarOffset = kSlotOffset + 16;
    static constexpr int kXOffset = kXBarOffset + kQTiles * 3 * 8 + 8;
    static constexpr int kXBytes = kSplit > 1 ? kQTiles * 3 * 2 * 128 * 4 : 0;   // [tile][max0, max1, sum][half][row]
    static constexpr int kLaunchBytes = kXOffset + kXBytes + 1024;
    // warp 0 Q and K producer, warp 1 MMA, then the softmax warps, then the V producer
    static constexpr int kVWarp = 2 + 4 * kSplit * kQTiles;
    static constexpr int kThreads = 32 * (kVWarp + 1);
    // tensor memory per Q tile: S buffers [0, kSBufs N), O [kSBufs N, kSBufs N + D)
    static constexpr int kOCol = kSBufs * kN;
    static constexpr int kTileCols = kSBufs * kN + D;
    static constexpr int kTmemCols = 512;
    static_assert(kLaunchBytes <= 227 * 1024, "shared memory plan too large");
    static_assert(kTileCols * kQTiles <= kTmemCols, "tensor memory plan too large");
};

template <typename T> struct TcType;
template <int V> struct IntTag { static constexpr int value = V; };
template <> struct TcType<__nv_bfloat16> { static constexpr int code = 1; };
template <> struct TcType<__half> { static constexpr int code = 0; };

__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Non-blocking test of phase `parity` of an mbarrier.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier; false after ~1e9 SM cycles (0.5 s
// at 2 GHz).  The pipeline here waits several times per tile, so the limit
// is kept with the SM's own cycle counter, which is cheap to read, not with
// the global timer.
__device__ __forceinline__ bool mbar_wait_cycles(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u && clock64() - t0 > 1000000000ll) return false;
    }
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two fp32 lanes in one 64-bit register, for the packed f32x2 arithmetic.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Hand over the P of a tile's first half: its tensor-memory stores complete,
// ordered before the warp's arrive (one per warp) on `bar`.
__device__ __forceinline__ void p_half_arrive(uint32_t bar, bool leader) {
    tc05::wait_st();
    tc05::fence_before_sync();
    __syncwarp();
    if (leader) mbar_arrive_cta(bar);
}

// Row max of one S tile in tensor memory (raw logits, columns c <= lim only
// when MASK), read in 32-column chunks with the next chunk's load in flight
// while the current one is reduced.  Unmasked and PACKED, each step folds two
// values into one of eight chains with a three-input max.
template <int N, bool MASK, bool PACKED>
__device__ __forceinline__ float tile_row_max(uint32_t sb, int lim) {
    uint32_t rr[2][32];
    float mt = -INFINITY;
    tc05::ld32_async(sb, rr[0]);
#pragma unroll
    for (int h = 0; h < N / 32; ++h) {
        tc05::wait_ld(rr[h & 1]);
        if (h + 1 < N / 32) tc05::ld32_async(sb + (h + 1) * 32, rr[(h + 1) & 1]);
        float mx[8];   // eight independent max chains
        if constexpr (PACKED && !MASK) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float v0 = __uint_as_float(rr[h & 1][2 * k]);
                const float v1 = __uint_as_float(rr[h & 1][2 * k + 1]);
                mx[k & 7] = k < 8 ? fmaxf(v0, v1) : fmax3(mx[k & 7], v0, v1);
            }
            mt = fmax3(mt, fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float v = __uint_as_float(rr[h & 1][c]);
                const float u = (!MASK || h * 32 + c <= lim) ? v : -INFINITY;
                mx[c & 7] = c < 8 ? u : fmaxf(mx[c & 7], u);
            }
            mt = fmaxf(mt, fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))));
        }
    }
    return mt;
}

// P = exp2(s * sl2 - mu) of one S tile (0 past lim when MASK), written as
// 16-bit pairs over the first N / 2 columns of the tile (chunk h's S has been
// read before its P lands on columns [16h, 16h + 16)); returns the row sum.
//
// Unmasked and PACKED, the arithmetic runs on column pairs: one packed fma
// forms both exponents (s * sl2 - mu), one packed add folds both values into
// one of four pair-sum chains (A/B on GB300: +2 % at head_dim 128 and 256; at
// head_dim 64 the pairs spill registers of the 576-thread CTA, so it keeps the
// scalar form).
template <typename T, int N, bool MASK, bool PACKED>
__device__ __forceinline__ float tile_row_p(uint32_t sb, int lim, float sl2, float mu,
                                            uint32_t half_bar, bool leader) {
    uint32_t rr[2][32];
    tc05::ld32_async(sb, rr[0]);
    if constexpr (PACKED && !MASK) {
        uint64_t sp[4];   // four pair-sum chains
        const uint64_t scale2 = f2(sl2, sl2), neg_mu2 = f2(-mu, -mu);
#pragma unroll
        for (int h = 0; h < N / 32; ++h) {
            tc05::wait_ld(rr[h & 1]);
            if (h + 1 < N / 32) tc05::ld32_async(sb + (h + 1) * 32, rr[(h + 1) & 1]);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 x = f2_split(ffma2(
                    f2(__uint_as_float(rr[h & 1][2 * i]), __uint_as_float(rr[h & 1][2 * i + 1])),
                    scale2, neg_mu2));
                const float e0 = ex2(x.x), e1 = ex2(x.y);
                const uint64_t e = f2(e0, e1);
                sp[i & 3] = (h == 0 && i < 4) ? e : fadd2(sp[i & 3], e);
                pk[i] = Mma<T>::pack(e0, e1);
            }
            tc05::st16(sb + h * 16, pk);
            if (half_bar != 0 && h == N / 64 - 1) p_half_arrive(half_bar, leader);
        }
        const float2 a = f2_split(fadd2(fadd2(sp[0], sp[1]), fadd2(sp[2], sp[3])));
        return a.x + a.y;
    } else {
        float sm[8];   // eight independent sum chains
#pragma unroll
        for (int h = 0; h < N / 32; ++h) {
            tc05::wait_ld(rr[h & 1]);
            if (h + 1 < N / 32) tc05::ld32_async(sb + (h + 1) * 32, rr[(h + 1) & 1]);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = h * 32 + 2 * i;
                float e0 = ex2(__uint_as_float(rr[h & 1][2 * i]) * sl2 - mu);
                float e1 = ex2(__uint_as_float(rr[h & 1][2 * i + 1]) * sl2 - mu);
                if (MASK) {
                    e0 = c <= lim ? e0 : 0.f;
                    e1 = c + 1 <= lim ? e1 : 0.f;
                }
                sm[i & 7] = (h == 0 && i < 8) ? e0 + e1 : sm[i & 7] + (e0 + e1);
                pk[i] = Mma<T>::pack(e0, e1);
            }
            tc05::st16(sb + h * 16, pk);
            if (half_bar != 0 && h == N / 64 - 1) p_half_arrive(half_bar, leader);
        }
        return ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
    }
}

// Register-resident form of the two passes, for one thread per whole row
// with registers to spare: the row's S is read from tensor memory once (all
// chunks' reads in flight together; reading chunk by chunk with the next one
// in flight measured the same) and the P pass works from the registers.
template <int N, bool MASK>
__device__ __forceinline__ float row_load_max(uint32_t (&sr)[N / 32][32], uint32_t sb, int lim) {
    float mt = -INFINITY;
    // every chunk's read in flight at once, then one wait
#pragma unroll
    for (int h = 0; h < N / 32; ++h) tc05::ld32_async(sb + h * 32, sr[h]);
#pragma unroll
    for (int h = 0; h < N / 32; ++h) tc05::wait_ld(sr[h]);
#pragma unroll
    for (int h = 0; h < N / 32; ++h) {
        float mx[8];
        if constexpr (!MASK) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float v0 = __uint_as_float(sr[h][2 * k]), v1 = __uint_as_float(sr[h][2 * k + 1]);
                mx[k & 7] = k < 8 ? fmaxf(v0, v1) : fmax3(mx[k & 7], v0, v1);
            }
            mt = fmax3(mt, fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float u = h * 32 + c <= lim ? __uint_as_float(sr[h][c]) : -INFINITY;
                mx[c & 7] = c < 8 ? u : fmaxf(mx[c & 7], u);
            }
            mt = fmaxf(mt, fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))));
        }
    }
    return mt;
}

template <typename T, int N, bool MASK>
__device__ __forceinline__ float row_p_regs(const uint32_t (&sr)[N / 32][32], uint32_t sb, int lim,
                                            float sl2, float mu, uint32_t half_bar, bool leader) {
    uint64_t sp[4];   // four pair-sum chains
    const uint64_t scale2 = f2(sl2, sl2), neg_mu2 = f2(-mu, -mu);
#pragma unroll
    for (int h = 0; h < N / 32; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 x = f2_split(ffma2(
                f2(__uint_as_float(sr[h][2 * i]), __uint_as_float(sr[h][2 * i + 1])), scale2, neg_mu2));
            float e0 = ex2(x.x), e1 = ex2(x.y);
            if (MASK) {
                const int c = h * 32 + 2 * i;
                e0 = c <= lim ? e0 : 0.f;
                e1 = c + 1 <= lim ? e1 : 0.f;
            }
            const uint64_t e = f2(e0, e1);
            sp[i & 3] = (h == 0 && i < 4) ? e : fadd2(sp[i & 3], e);
            pk[i] = Mma<T>::pack(e0, e1);
        }
        tc05::st16(sb + h * 16, pk);
        if (half_bar != 0 && h == N / 64 - 1) p_half_arrive(half_bar, leader);
    }
    const float2 a = f2_split(fadd2(fadd2(sp[0], sp[1]), fadd2(sp[2], sp[3])));
    return a.x + a.y;
}

template <typename T, int D>
__global__ void __launch_bounds__(PrefillTcCfg<D>::kThreads, 1)
    pa_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    using C = PrefillTcCfg<D>;
    constexpr int N = C::kN, NK = C::kKStages, NV = C::kVStages, NQ = C::kQTiles, SB = C::kSBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t base = smem_u32(smem);
    const uint32_t q_smem = base;
    const uint32_t kstage0 = base + C::kKOffset, vstage0 = base + C::kVOffset;
    const uint32_t bars = base + C::kBarOffset;
    const uint32_t q_full = bars, vtail = bars + 8, mma_done = bars + 16;
    const uint32_t k_full = bars + 24, k_empty = k_full + NK * 8;
    const uint32_t v_full = k_empty + NK * 8, v_empty = v_full + NV * 8;
    const uint32_t tile_bars = v_empty + NV * 8;   // + t * kTileBarBytes: s_full, p_full, s_free, o_full, p_half
    const uint32_t slot = base + C::kSlotOffset;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = gridDim.x - 1 - blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
    const int g = p.group;

    // ---- which rows and which context this CTA covers (uniform over the CTA) ----
    const int cap = p.max_blocks * p.block_size;
    const int L = clamp_len(p.seq_lens, s, cap, p.status);
    const int row0 = __ldg(p.q_start + s), row1 = __ldg(p.q_start + s + 1);
    const bool first = blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0;
    if (row0 < 0 || row1 < row0 || row1 > p.num_rows) {   // rows outside the query
        if (first) atomicOr(p.status, kBadRows);
        return;
    }
    const int n = row1 - row0;
    if (n > L) {   // a chunk longer than its whole context: the sequence is skipped
        if (first) atomicOr(p.status, kBadRows);
        return;
    }
    if (first && n > static_cast<int>(gridDim.x) * p.tokens_per_cta)
        atomicOr(p.status, kLenClamped);   // chunk longer than max_q_len: its tail is not written
    const int tok0 = qt * p.tokens_per_cta;
    if (tok0 >= n) return;
    const int ntok = min(p.tokens_per_cta, n - tok0);
    const int pos_first = L - n + tok0;   // position of the CTA's first chunk token
    const int kv_end = pos_first + ntok;  // cache tokens any row of the CTA sees
    const int ntiles = (kv_end + N - 1) / N;
    // Where the CTAs of one (sequence, KV head) start their walk over the
    // context (PA_PREFILL_ROT_STEP_*).  The online softmax does not depend on
    // the order.
    const int rot = static_cast<int>(gridDim.x) >= PA_PREFILL_ROT_MIN_CTAS
                        ? static_cast<int>((static_cast<unsigned>(qt) *
                                            (D <= 64 ? PA_PREFILL_ROT_STEP_D64 : PA_PREFILL_ROT_STEP_D128)) %
                                           static_cast<unsigned>(ntiles))
                        : 0;
    const int rows_used = g * ntok;
    const int nq = NQ > 1 && rows_used > 128 ? 2 : 1;   // Q tiles with any row to compute
    // A CTA whose rows fit one Q tile (at most 128) gives that tile the idle
    // tile's tensor memory as a second S buffer, at column kTileCols, so the
    // tile's next QK runs under its softmax instead of after its PV.
    constexpr bool kCanDual = PA_PREFILL_DUAL && C::kSBufs == 1 && NQ == 2;
    const bool dual = kCanDual && nq == 1 && static_cast<int>(gridDim.x) <= PA_PREFILL_DUAL_MAX_CTAS;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        mbar_init(q_full, 1);
        mbar_init(vtail, 1);
        mbar_init(mma_done, 1);
        for (int i = 0; i < NK; ++i) {
            mbar_init(k_full + i * 8, 1);
            mbar_init(k_empty + i * 8, 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(v_full + i * 8, 1);
            mbar_init(v_empty + i * 8, 1);
        }
        for (int t = 0; t < NQ; ++t) {
            const uint32_t tb = tile_bars + t * C::kTileBarBytes;
            for (int i = 0; i < 2; ++i) {
                mbar_init(tb + i * 8, 1);          // s_full
                mbar_init(tb + 16 + i * 8, 4 * C::kSplit);   // p_full: one arrive per softmax warp
                mbar_init(tb + 32 + i * 8, 1);     // s_free
            }
            mbar_init(tb + 48, 1);                 // o_full
            mbar_init(tb + 56, 4 * C::kSplit);     // p_half
            if (C::kSplit > 1)
                for (int i = 0; i < 3; ++i) mbar_init(base + C::kXBarOffset + (t * 3 + i) * 8, 8);
        }
        fence_mbar_init();
    }
    if (warp == 1) tc05::alloc(slot, C::kTmemCols);
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::kSlotOffset);

    if (warp == 0 || warp == C::kVWarp) {
        // ------------------------------ producers ------------------------------
        // warp 0 loads Q and the K tiles, the last warp the V tiles, each
        // through its own stages, so a K copy never waits behind a V stage
        const int32_t *bt_row = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
        const int nbox = (kv_end + kTile - 1) / kTile;
        constexpr int kBoxes = N / kTile;   // 16-token boxes per tile
        static_assert(2 * kBoxes <= 32, "one copy per lane");
        // Each producer lane copies one 16-token box of a tile, all its pieces;
        // with block_size 8 a box spans two blocks, and lane pairs copy its halves.
        const bool b8 = p.block_size < kTile;
        const int op_box = b8 ? lane >> 1 : lane, half = b8 ? lane & 1 : 0;
        const bool has = op_box < kBoxes;
        auto first_token = [&](int jt) { return (jt * kBoxes + op_box) * kTile + half * (kTile / 2); };
        // block of this lane's box (half) of tile jt (0 when the lane has no
        // copy or the half lies past the context).  The read goes out a tile
        // ahead and is checked only when the copy is issued, so its latency
        // overlaps the stage waits in between (with one stage, a read consumed
        // at once put ~3000 cycles on every tile's K load).
        auto box_block = [&](int jt) -> int {
            const int tok = first_token(jt);
            return has && tok < kv_end ? __ldg(bt_row + tok / p.block_size) : 0;
        };
        // the copy's 8-token group coordinate; -1 (a box of zeros) for a half
        // past the context or a block outside the cache (that one flagged)
        auto group_of = [&](int jt, int b) -> int {
            const int tok = first_token(jt);
            if (tok >= kv_end) return -1;
            if (static_cast<unsigned>(b) >= static_cast<unsigned>(p.num_blocks)) {
                atomicOr(p.status, kBadBlock);
                return -1;
            }
            return b * (p.block_size >> 3) + ((tok % p.block_size) >> 3);
        };
        // bytes of tile jt's boxes inside the context (K or V: the same)
        auto tile_bytes = [&](int jt) {
            int boxes = 0;
#pragma unroll
            for (int k = 0; k < kBoxes; ++k) boxes += jt * kBoxes + k < nbox;
            return static_cast<uint32_t>(boxes * C::kPieces * 2048);
        };
        bool ok = true;
        if (warp == 0) {
            // Q rows the box does not cover (kRows % group) are never loaded: zero
            // them so those rows stay finite (and never force an O rescale).
            const int qrows = g * p.tokens_per_cta;
            if (qrows < C::kRows) {
                for (int c = 0; c < C::kPieces; ++c)
                    for (int e = lane; e < (C::kRows - qrows) * 8; e += 32)
                        *reinterpret_cast<uint4 *>(smem + c * C::kQPiece + qrows * 128 + e * 16) =
                            make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                mbar_expect_tx(q_full, static_cast<uint32_t>(C::kPieces * 128 * qrows));
#pragma unroll
                for (int c = 0; c < C::kPieces; ++c)
                    tma_load_4d(q_smem + c * C::kQPiece, &tmQ, q_full, 0, c, kvh * g, row0 + tok0);
            }
            int jt = rot, phys_next = box_block(rot), issued = 0;
            for (int j = 0; j < ntiles; ++j) {   // j: order of use, jt: tile of the context
                const int st = j % NK, phys = phys_next, jc = jt;
                jt = jt + 1 == ntiles ? 0 : jt + 1;
                if (j + 1 < ntiles) phys_next = box_block(jt);   // next tile's entry
                // K of tile j once every QK of tile j - NK is done
                if (j >= NK) {
                    const bool w = mbar_wait_cycles(k_empty + st * 8, ((j / NK) - 1) & 1u);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                }
                // one copy per lane: a single thread issuing them back to back is
                // bound by the issue latency of each copy, not by the TMA engine
                if (lane == 0) mbar_expect_tx(k_full + st * 8, tile_bytes(jc));
                __syncwarp();
                // the cache maps: (element, row in group, piece, head, group)
                if (has && jc * kBoxes + op_box < nbox)
                    tma_load_5d(kstage0 + st * C::kTileBytes + op_box * C::kBoxBytes +
                                    half * (C::kPieces * 1024),
                                &tmK, k_full + st * 8, 0, 0, 0, kvh, group_of(jc, phys));
                issued = j + 1;
            }
            if (!ok && lane == 0) atomicOr(p.status, kWaitTimeout);
            // copies still landing must land before the CTA exits (at most NK
            // tiles' K are in flight: each waited for the QK of the one NK before)
            (void)mbar_wait_cycles(q_full, 0);
            for (int j = issued > NK ? issued - NK : 0; j < issued; ++j)
                (void)mbar_wait_cycles(k_full + (j % NK) * 8, (j / NK) & 1u);
        } else {
            int jt = rot, phys_next = box_block(rot), issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % NV, phys = phys_next, jc = jt;
                jt = jt + 1 == ntiles ? 0 : jt + 1;
                if (j + 1 < ntiles) phys_next = box_block(jt);
                const uint32_t vdst = vstage0 + st * C::kTileBytes;
                const bool last = jc == ntiles - 1;   // the context's tail tile
                const uint32_t vbar = last ? vtail : v_full + st * 8;
                // V of tile j once every PV of tile j - NV is done
                if (j >= NV) {
                    const bool w = mbar_wait_cycles(v_empty + st * 8, ((j / NV) - 1) & 1u);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                }
                if (lane == 0) mbar_expect_tx(vbar, tile_bytes(jc));
                __syncwarp();
                if (has && jc * kBoxes + op_box < nbox)
                    tma_load_5d(vdst + op_box * C::kBoxBytes + half * (C::kPieces * 1024), &tmV, vbar,
                                0, 0, 0, kvh, group_of(jc, phys));
                issued = j + 1;
                if (last) {
                    // V rows at or past kv_end hold cache data past the context (or
                    // nothing): zero them before the MMA reads V, since 0 * NaN != 0.
                    const bool w = mbar_wait_cycles(vtail, 0);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                    const int first_row = kv_end - jc * N;
                    const int nchunks = (N - first_row) * C::kPieces * 8;   // 16-byte chunks
                    for (int e = lane; e < nchunks; e += 32) {
                        const int r = first_row + e / (C::kPieces * 8);
                        const int c = (e / 8) % C::kPieces;
                        *reinterpret_cast<uint4 *>(smem + (vdst - base) + (r >> 3) * (C::kPieces * 1024) +
                                                   c * 1024 + (r & 7) * 128 + (e & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cta(v_full + st * 8);
                }
            }
            if (!ok && lane == 0) atomicOr(p.status, kWaitTimeout);
            // copies still landing must land before the CTA exits
            const int j_tail = ntiles - 1 - rot;   // use order of the tail tile
            for (int j = issued > NV ? issued - NV : 0; j < issued; ++j)
                if (j != j_tail) (void)mbar_wait_cycles(v_full + (j % NV) * 8, (j / NV) & 1u);
            if (issued > j_tail) (void)mbar_wait_cycles(vtail, 0);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        // The whole warp runs the issue sequence, its control flow warp-uniform,
        // and one elected lane issues each MMA and commit (a lone thread in a
        // divergent branch issued an MMA every ~47 cycles, slower than the pipe
        // once the softmax warps share its scheduler).  The sequence is fixed:
        // QK of the first SB tiles for every Q tile, then per K/V tile j and Q
        // tile t the PV of j and the QK of j + SB (the QK that overwrites an S
        // buffer right behind the PV that reads its P: one thread's MMAs run on
        // the tensor pipe in issue order, so the QK's writes come after the PV's
        // operand reads).  Each step waits (suspending, bounded) on exactly the
        // barrier it needs: a loop polling every tile's barriers saw a completed
        // phase ~1000 cycles late, the pipe idle meanwhile.  Every barrier waited
        // on depends only on MMAs issued earlier in the sequence, so the fixed
        // order cannot deadlock.
        constexpr uint32_t kAll = 0xffffffffu;
        constexpr uint32_t idesc_qk = tc05::f16_idesc(TcType<T>::code, 0, 0, N, 128);
        constexpr uint32_t idesc_pv = tc05::f16_idesc(TcType<T>::code, 0, 1, D, 128);
        bool ok = __all_sync(kAll, mbar_wait_cycles(q_full, 0));
        auto wait = [&](uint32_t bar, uint32_t parity) {
            ok = ok && __all_sync(kAll, mbar_wait_cycles(bar, parity));
            return ok;
        };
        // the issue sequence for SBX S buffers per Q tile (S buffer b at column b * SC)
        auto run = [&](auto sbt) {
            constexpr int SBX = decltype(sbt)::value;
            constexpr int SC = SBX == C::kSBufs ? N : C::kTileCols;
            // S_j = Q_t K_j^T into S buffer j % SBX; the last Q tile's QK frees the K stage
            auto issue_qk = [&](int t, int j) {
                const uint32_t tb = tile_bars + t * C::kTileBarBytes;
                const uint32_t tcol = tmem + t * C::kTileCols;
                const uint32_t kst = kstage0 + (j % NK) * C::kTileBytes;
                const uint32_t qst = q_smem + t * C::kQTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc05::mma_ss_elect(
                        tcol + (j % SBX) * SC,
                        tc05::sw128_desc(qst + (kk >> 2) * C::kQPiece + (kk & 3) * 32, 16, 1024),
                        tc05::sw128_desc(kst + (kk >> 2) * 1024 + (kk & 3) * 32, 16, C::kPieces * 1024),
                        idesc_qk, kk > 0 ? 1u : 0u);
                tc05::commit_elect(tb + (j % SBX) * 8);   // s_full
                if (t == nq - 1) tc05::commit_elect(k_empty + (j % NK) * 8);
            };
            // O_t += P_j V_j over the K-steps [kt0, kt1) (16 tokens each); the end of
            // the last Q tile's PV frees the V stage
            auto issue_pv = [&](int t, int j, int kt0, int kt1) {
                const uint32_t tb = tile_bars + t * C::kTileBarBytes;
                const uint32_t tcol = tmem + t * C::kTileCols;
                const uint32_t vst = vstage0 + (j % NV) * C::kTileBytes;
#pragma unroll
                for (int kt = kt0; kt < kt1; ++kt)
                    // tokens [16 kt, 16 kt + 16) lie in part (16 kt) / kHalfCols,
                    // whose P occupies the first half of its own S columns
                    tc05::mma_ts_elect(tcol + C::kOCol,
                                       tcol + (j % SBX) * SC +
                                           ((16 * kt) / C::kHalfCols) * (C::kHalfCols / 2) + kt * 8,
                                       tc05::sw128_desc(vst + kt * C::kBoxBytes, 1024, C::kPieces * 1024),
                                       idesc_pv, (j > 0 || kt > 0) ? 1u : 0u);
                if (kt1 < N / 16) return;
                // s_free: with one S buffer the commit of the QK issued next (S_{j+1})
                // tracks this PV as well, so none is needed
                if (SBX > 1) tc05::commit_elect(tb + 32 + (j % SBX) * 8);
                if (t == nq - 1) tc05::commit_elect(v_empty + (j % NV) * 8);
                if (j == ntiles - 1) tc05::commit_elect(tb + 48);   // o_full
            };
            for (int j = 0; ok && j < SBX && j < ntiles; ++j) {
                if (!wait(k_full + (j % NK) * 8, (j / NK) & 1u)) break;
                tc05::fence_after_sync();
                for (int t = 0; t < nq; ++t) issue_qk(t, j);
            }
            for (int j = 0; ok && j < ntiles; ++j) {
                if (!wait(v_full + (j % NV) * 8, (j / NV) & 1u)) break;
                const int jn = j + SBX;   // the QK issued behind this tile's PV
                for (int t = 0; t < nq; ++t) {
                    const uint32_t tb = tile_bars + t * C::kTileBarBytes;
                    int kt0 = 0;
                    // the PV of the first N / 2 tokens once their P is in (one S buffer
                    // only: p_half is one barrier per tile, which a second buffer's
                    // softmax could complete twice before this wait)
                    if (C::kHalfP && SBX == 1) {
                        if (!wait(tb + 56, j & 1u)) break;   // p_half
                        tc05::fence_after_sync();
                        issue_pv(t, j, 0, N / 32);
                        kt0 = N / 32;
                    }
                    if (!wait(tb + 16 + (j % SBX) * 8, (j / SBX) & 1u)) break;   // p_full
                    tc05::fence_after_sync();
                    issue_pv(t, j, kt0, N / 16);
                    if (jn < ntiles) {
                        if (t == 0 && !wait(k_full + (jn % NK) * 8, (jn / NK) & 1u)) break;
                        tc05::fence_after_sync();
                        issue_qk(t, jn);
                    }
                }
            }
        };
        if constexpr (kCanDual) {
            if (dual)
                run(IntTag<2>{});
            else
                run(IntTag<C::kSBufs>{});
        } else {
            run(IntTag<C::kSBufs>{});
        }
        if (!ok && lane == 0) atomicOr(p.status, kWaitTimeout);
        // every MMA issued has completed before tensor memory is freed
        tc05::commit_elect(mma_done);
        (void)mbar_wait_cycles(mma_done, 0);
        __syncwarp();
    } else {
        // ------------------------------ softmax ------------------------------
        constexpr int HC = C::kHalfCols;
        const int idx = warp - 2;
        constexpr int SP = C::kSplit;
        // column pairs (packed arithmetic) where the registers allow them: the
        // 18-warp CTA of head_dim 64 with split rows is capped at 96 per thread
        constexpr bool PK = D >= 128 || SP == 1;
        // whole rows of head_dim >= 128 keep S in registers between the passes
        constexpr bool RR = PA_PREFILL_REGROW && SP == 1 && N <= 128;
        constexpr int RC = RR ? N / 32 : 1;
        const int t = idx / (4 * SP);     // the Q tile of this warp
        const int hf = (idx >> 2) % SP;   // the part of the S columns it handles
        if (t < nq) {
            const int quarter = warp & 3;   // tensor-memory lanes 32*quarter .. +31
            const int rl = quarter * 32 + lane;   // row within the Q tile
            const int r = t * 128 + rl;
            const bool valid = r < rows_used;
            const int tq = valid ? r / g : ntok - 1, hq = valid ? r % g : 0;
            const int pos = pos_first + tq;   // last cache token this row sees
            const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
            const uint32_t tcol = tmem + lane_base + t * C::kTileCols;
            const uint32_t tb = tile_bars + t * C::kTileBarBytes;
            const uint32_t xbar = base + C::kXBarOffset + t * 3 * 8;   // max exchange x2, sums
            float *xch = reinterpret_cast<float *>(smem + C::kXOffset) + t * 3 * 256;
            const float sl2 = p.scale_log2;
            float m = -INFINITY, l = 0.f;   // l: this part's share of the row sum
            bool ok = true;
            auto tiles = [&](auto sbt) {
                constexpr int SBX = decltype(sbt)::value;
                constexpr int SC = SBX == C::kSBufs ? N : C::kTileCols;
                for (int j = 0; j < ntiles; ++j) {
                    const int b = j % SBX;
                    const bool w = mbar_wait_cycles(tb + b * 8, (j / SBX) & 1u);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                    tc05::fence_after_sync();
                    const uint32_t sb = tcol + b * SC + hf * HC;   // this part's S columns
                    const int jt = j + rot < ntiles ? j + rot : j + rot - ntiles;
                    const int lim = pos - jt * N - hf * HC;   // own columns c <= lim are visible
                    // pass 1: this part's row max (with two parts, swapped with the other's)
                    const bool full = __all_sync(0xffffffffu, lim >= HC - 1);
                    uint32_t sr[RC][32];
                    float pm;
                    if constexpr (RR)
                        pm = full ? row_load_max<N, false>(sr, sb, lim) : row_load_max<N, true>(sr, sb, lim);
                    else
                        pm = full ? tile_row_max<HC, false, PK>(sb, lim)
                                  : tile_row_max<HC, true, PK>(sb, lim);
                    float mt = pm;
                    if constexpr (SP > 1) {
                        xch[(j & 1) * 256 + hf * 128 + rl] = pm;
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cta(xbar + (j & 1) * 8);
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait_cycles(xbar + (j & 1) * 8, (j >> 1) & 1u))) {
                            ok = false;
                            break;
                        }
                        mt = fmaxf(pm, xch[(j & 1) * 256 + (1 - hf) * 128 + rl]);
                    }
                    mt *= sl2;   // log2 domain (scale > 0)
                    if (j == 0) {
                        m = mt;   // -inf when every column of the first tile is past the row
                    } else if (__any_sync(0xffffffffu, mt > m + 8.f)) {
                        // O must hold P_{j-1} V_{j-1} before it is rescaled (all parts
                        // see the same maxima, so all take this branch for a row).  With
                        // one S buffer, PV_{j-1} went out before QK_j from the same thread,
                        // so the S_j commit waited for above has already seen it finish.
                        if (SBX > 1) {
                            const bool w2 =
                                mbar_wait_cycles(tb + 32 + ((j - 1) % SBX) * 8, ((j - 1) / SBX) & 1u);
                            if (!__all_sync(0xffffffffu, w2)) {
                                ok = false;
                                break;
                            }
                            tc05::fence_after_sync();
                        }
                        const float mn = fmaxf(m, mt);
                        const float alpha = m == mn ? 1.f : ex2(m - mn);   // 0 when m was -inf
                        m = mn;
                        l *= alpha;
                        // this part's O columns, 16 at a time while the S row is held
                        constexpr int OC = RR ? 16 : 32;
#pragma unroll
                        for (int c0 = 0; c0 < D / SP; c0 += OC) {
                            uint32_t rr[OC];
                            const uint32_t oc = tcol + C::kOCol + hf * (D / SP) + c0;
                            if constexpr (RR) tc05::ld16(oc, rr); else tc05::ld32(oc, rr);
#pragma unroll
                            for (int i = 0; i < OC; ++i)
                                rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
                            if constexpr (RR) tc05::st16(oc, rr); else tc05::st32(oc, rr);
                        }
                    }
                    // pass 2: P of this part over the first half of its own S columns
                    const float mu = m == -INFINITY ? 0.f : m;   // no column seen yet: P = 0
                    const uint32_t hb = C::kHalfP && SBX == 1 ? tb + 56 : 0u;   // p_half
                    if constexpr (RR)
                        l += full ? row_p_regs<T, N, false>(sr, sb, lim, sl2, mu, hb, lane == 0)
                                  : row_p_regs<T, N, true>(sr, sb, lim, sl2, mu, hb, lane == 0);
                    else
                        l += full ? tile_row_p<T, HC, false, PK>(sb, lim, sl2, mu, hb, lane == 0)
                                  : tile_row_p<T, HC, true, PK>(sb, lim, sl2, mu, hb, lane == 0);
                    tc05::wait_st();
                    tc05::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cta(tb + 16 + b * 8);   // p_full
                }
            };
            if constexpr (kCanDual) {
                if (dual)
                    tiles(IntTag<2>{});
                else
                    tiles(IntTag<C::kSBufs>{});
            } else {
                tiles(IntTag<C::kSBufs>{});
            }
            if (SP > 1 && ok) {   // the row sum is the two parts' shares
                xch[2 * 256 + hf * 128 + rl] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive_cta(xbar + 16);
                ok = __all_sync(0xffffffffu, mbar_wait_cycles(xbar + 16, 0));
                if (ok) l += xch[2 * 256 + (1 - hf) * 128 + rl];
            }
            if (ok) {
                const bool w = mbar_wait_cycles(tb + 48, 0);   // o_full
                ok = __all_sync(0xffffffffu, w);
            }
            if (ok) {
                tc05::fence_after_sync();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                T *orow = static_cast<T *>(p.out) +
                          (static_cast<size_t>(row0 + tok0 + tq) * p.num_q_heads + kvh * g + hq) *
                              D + hf * (D / SP);
#pragma unroll
                for (int c0 = 0; c0 < D / SP; c0 += 32) {   // this part's output columns
                    uint32_t rr[32];
                    tc05::ld32(tcol + C::kOCol + hf * (D / SP) + c0, rr);
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) {
                            uint4 v;
                            v.x = Mma<T>::pack(__uint_as_float(rr[i]) * inv,
                                               __uint_as_float(rr[i + 1]) * inv);
                            v.y = Mma<T>::pack(__uint_as_float(rr[i + 2]) * inv,
                                               __uint_as_float(rr[i + 3]) * inv);
                            v.z = Mma<T>::pack(__uint_as_float(rr[i + 4]) * inv,
                                               __uint_as_float(rr[i + 5]) * inv);
                            v.w = Mma<T>::pack(__uint_as_float(rr[i + 6]) * inv,
                                               __uint_as_float(rr[i + 7]) * inv);
                            *reinterpret_cast<uint4 *>(orow + c0 + i) = v;
                        }
                    }
                }
            } else if (lane == 0) {
                atomicOr(p.status, kWaitTimeout);
            }
        }
    }
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    if (warp == 1) tc05::dealloc(tmem, C::kTmemCols);
}

template <typename T, int D>
inline cudaError_t launch_prefill_tc_d(const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                       const CUtensorMap &tmV, const PrefillParams &p, dim3 grid,
                                       cudaStream_t st) {
    using C = PrefillTcCfg<D>;
    static std::atomic<int> done[kMaxDevices];
    auto k = pa_prefill_tc_kernel<T, D>;
    cudaError_t e = ensure_smem(k, C::kLaunchBytes, done);
    if (e != cudaSuccess) return e;
    k<<<grid, C::kThreads, C::kLaunchBytes, st>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace pa
