// pa_kernels.cuh -- device code of the paged-attention decode library for
// GB300 (sm_103a).
//
// The method (page: project_6 commit cd0d9e1, "qwen3_6_scripts"):
//   * forward_decode heuristic: a decode query attends over its sequence's
//     whole KV range in one pass (V1) when the sequence is short, and over
//     fixed-size partitions processed in parallel (V2) when it is long;
//   * V2 description, phase 1: each partition yields a partial output
//     normalised by its own exp-sum, that exp-sum, and its maximum logit;
//     phase 2 merges the partitions with weights exp(partition max - global
//     max) * partition exp-sum;
//   * the same page notes that the tiling is Flash-Attention-style online
//     softmax and that the merge is the usual combination of partial
//     (max, sum) statistics of independent segments.  Here that merge is
//     used twice: between the warps of a CTA inside a partition, and between
//     partitions in the reduce kernel.
//
// GB300 design (how, not what):
//   * One work unit = (sequence, KV head, token range).  All query heads that
//     share the KV head (the GQA group, <= 8) are handled by the unit, so each
//     K/V byte is read from HBM once.
//   * Each warp of a CTA owns a ring of NS shared-memory stages and streams
//     16-token tiles of its share of the unit through them with TMA
//     (cp.async.bulk.tensor, 5-D tensor map over the cache, 128-byte swizzle)
//     completing on an mbarrier.  Block-table entries are prefetched 32 tiles
//     ahead into a lane-distributed register window.  A table entry outside
//     the cache becomes an out-of-bounds TMA coordinate, which reads zeros.
//   * The per-tile contraction is tiny (16 tokens x <=8 heads x head_dim), so
//     it runs on warp-level tensor-core MMAs (m16n8k16, fp32 accumulate) in a
//     transposed form: S^T = K Q^T (M = tokens, N = heads) and
//     O^T += V^T P^T (M = head_dim, N = heads).  The softmax probabilities go
//     from the S^T accumulator to the P^T operand with one movmatrix
//     transpose per 8x8 block, never touching shared memory.
//   * Softmax runs in the log2 domain (logit * scale * log2 e) with ex2.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_types.h"

namespace pa {

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of an mbarrier; false after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u && global_ns() - t0 > limit_ns) return false;
    }
}

// 5-D tiled TMA load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "r"(bar)
        : "memory");
}

// Programmatic dependent launch: the decode step's kernels are launched so the
// next one may start while the previous one drains.  A kernel waits, before
// its first global access, until the previous grid in the stream has
// completed with its memory visible (a no-op when launched without the
// attribute), and lets the next grid launch once its own work is done.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 eviction-priority policies.  Decode reads every K/V byte once, so its
// tile loads are marked evict-first and do not push out of L2 the partial
// results (written evict-last) that the reduce reads right after.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 5-D tiled TMA load with an L2 cache policy.
__device__ __forceinline__ void tma_load_5d_hint(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar, int c0, int c1, int c2, int c3,
                                                 int c4, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void st_global_hint(float *ptr, float v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T> struct Mma;

template <> struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    static __device__ __forceinline__ __nv_bfloat16 cvt(float x) { return __float2bfloat16_rn(x); }
};

template <> struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    static __device__ __forceinline__ __half cvt(float x) { return __float2half_rn(x); }
};

// Byte offset of element (row, col) of one 16-row tile as the TMA loads lay
// it out.  Piecewise layout (default): one 2 KB block per 64-element
// (128-byte) piece of the head dimension, holding that piece of the 16 rows
// as consecutive 128-byte rows, with the 128-byte swizzle (16-byte chunk
// index XOR row mod 8): the eight rows an ldmatrix reads hit eight different
// bank groups.  Row-major layout (PA_TILE_PIECES=0): the 16 rows of D
// elements one after the other, one TMA per tile; rows of 256 or 512 bytes
// make the swizzle repeat every 4 or 2 rows (2- or 4-way bank conflicts).
// Tiles start on 1024-byte boundaries.
#ifndef PA_TILE_PIECES
#define PA_TILE_PIECES 1
#endif
constexpr int kPieceBytes = kTile * 128;
constexpr bool kPiecewise = PA_TILE_PIECES != 0;

template <int D>
__device__ __forceinline__ uint32_t swz(int row, int col) {
    const int chunk = (col & 63) >> 3;
    if constexpr (kPiecewise) {
        return static_cast<uint32_t>((col >> 6) * kPieceBytes + row * 128 +
                                     ((chunk ^ (row & 7)) << 4) + ((col & 7) << 1));
    } else {
        const int r128 = row * (D / 64) + (col >> 6);
        return static_cast<uint32_t>(r128 * 128 + ((chunk ^ (r128 & 7)) << 4) + ((col & 7) << 1));
    }
}

// Byte offset of row `row` of piece `c` (the V rows past a sequence end are
// zeroed through it): contiguous 128-byte rows in both layouts.
template <int D>
__device__ __forceinline__ uint32_t row_piece_offset(int row, int c) {
    return kPiecewise ? static_cast<uint32_t>(c * kPieceBytes + row * 128)
                      : static_cast<uint32_t>((row * (D / 64) + c) * 128);
}

// Load one 16-row tile of KV head kvh, all completing on `bar`: rows
// row..row+15 of block b0 (block_size >= 16: one box of 16 rows per 64-element
// piece), or, with `split` (block_size 8), rows 0..7 of block b0 and rows 0..7
// of block b1 as two 8-row boxes per piece.  The second box lands 1024 bytes
// into the piece, on a whole 128-byte-swizzle period, so both halves have the
// layout of one 16-row box.
template <int D>
__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                              int kvh, int row, int b0, int b1, bool split) {
    if constexpr (kPiecewise) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            tma_load_5d(dst + c * kPieceBytes, map, bar, 0, c, kvh, row, b0);
            if (split) tma_load_5d(dst + c * kPieceBytes + 1024, map, bar, 0, c, kvh, 0, b1);
        }
    } else {
        tma_load_5d(dst, map, bar, 0, 0, kvh, row, b0);   // block_size 8 is refused on the host
    }
}

// The same with an L2 cache policy on every copy.
template <int D>
__device__ __forceinline__ void tma_load_tile_hint(uint32_t dst, const CUtensorMap *map,
                                                   uint32_t bar, int kvh, int row, int b0, int b1,
                                                   bool split, uint64_t policy) {
    if constexpr (kPiecewise) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            tma_load_5d_hint(dst + c * kPieceBytes, map, bar, 0, c, kvh, row, b0, policy);
            if (split)
                tma_load_5d_hint(dst + c * kPieceBytes + 1024, map, bar, 0, c, kvh, 0, b1, policy);
        }
    } else {
        tma_load_5d_hint(dst, map, bar, 0, 0, kvh, row, b0, policy);
    }
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ int dsmem_ld_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ int clamp_len(const int32_t *seq_lens, int s, int cap, int *status) {
    int L = __ldg(seq_lens + s);
    if (L < 0 || L > cap) {
        atomicOr(status, kLenClamped);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

__device__ __forceinline__ void dsmem_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void dsmem_st_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory plan of the attention kernel
// ---------------------------------------------------------------------------
template <int D, int NW, int NS, int HP>
struct Smem {
    static constexpr int kTileBytes = kTile * D * 2;            // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;          // K tile + V tile
    static constexpr int kStagesBytes = NW * NS * kStageBytes;
    static constexpr int kMergeBytes = NW * HP * (D + 2) * 4;
    // Cluster merge of the single-pass grid: CTA r of the cluster finishes the
    // r-th slice of the unit's output elements, so it receives from every CTA
    // (itself included) that CTA's merged values of the slice, o_in
    // [rank][slice] (slices of whole quads: at most HP * D + 32 floats for any
    // cluster size), and its
    // per-head maximum and sum, m_in / l_in [rank][HP], and abort flag.
    // Written only after every CTA of the cluster has finished with its stages
    // and its own merge area, so it overlaps both.
    static constexpr int kMaxCluster = 8;
    static constexpr int kInO = 0;
    static constexpr int kInM = kInO + (HP * D + 4 * kMaxCluster) * 4;
    static constexpr int kInL = kInM + kMaxCluster * HP * 4;
    static constexpr int kInAbort = kInL + kMaxCluster * HP * 4;
    static constexpr int kClusterEnd = kInAbort + kMaxCluster * 4;
    static constexpr int kUsed = kMergeBytes > kClusterEnd ? kMergeBytes : kClusterEnd;
    static constexpr int kBarOffset =
        ((kStagesBytes > kUsed ? kStagesBytes : kUsed) + 15) / 16 * 16;
    static constexpr int kBytes = kBarOffset + NW * NS * 8 + 16;
    static constexpr int kLaunchBytes = kBytes + 1024;          // slack for 1024-byte alignment
};

// ---------------------------------------------------------------------------
// One work unit: tokens [t0, t1) of (seq, head group v), v = (KV head kvh,
// head group hg) with kvh = v / hg_count: the query heads hg*HP .. hg*HP+HP-1
// of kvh's GQA group (all of them when the group has at most HP heads), so a
// K/V byte is read once per head group.  HP = 8 or 16 heads: one or two n8
// tiles of the warp MMAs.
// `span()` gives t1 once the unit's first loads are in flight: the block-table
// window and the query fragments do not wait for the sequence length, so the
// length read and the table reads overlap.  A negative t1 means the unit does
// not exist (a partition past the sequence end): nothing is written.
// With a cluster of `csize` CTAs (single-pass grid only), CTA `crank` takes
// every csize-th group of NW tiles and the other CTAs push their merged
// states into the leader's shared memory, which writes the output.  Returns
// false if a pipeline wait gave up (the CTA must stop).
// ---------------------------------------------------------------------------
template <typename T, int D, int NW, int NS, int HP, typename Span>
__device__ __forceinline__ bool attend_unit(const Params &p, const CUtensorMap *tmK,
                                            const CUtensorMap *tmV, uint8_t *smem, uint32_t bar0,
                                            uint32_t &uses, int seq, int vkh, int t0, Span span,
                                            int out_kind, int part, int slot, int *s_abort,
                                            int crank = 0, int csize = 1) {
    using SM = Smem<D, NW, NS, HP>;
    constexpr int KT = D / 16;   // k-steps of S^T, m-tiles of O^T
    constexpr int NT8 = HP / 8;  // n8 tiles (heads) of S^T and O^T
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kvh = vkh / p.hg_count;
    const int h0 = (vkh - kvh * p.hg_count) * HP;        // first head of the group
    const int gh = min(HP, p.group - h0);                // heads of this unit
    const int qhead0 = kvh * p.group + h0;               // its first query head
    const int woff = crank * NW + warp;    // this warp's first tile
    const int wstride = csize * NW;        // tiles between two of this warp's tiles
    const int32_t *bt_row = p.block_tables + static_cast<size_t>(seq) * p.max_blocks;
    const bool split = p.block_size < kTile;   // block_size 8: two blocks per tile

    // Block-table window: lane l holds the entry of local tile base+l (with
    // block_size 8, of the tile's first block; the second is the next entry).
    // Reads are bounded by the table row, not by the length, which is not
    // known yet; an entry is checked against the cache when its tile is issued.
    auto entry = [&](long long j) -> int { return j < p.max_blocks ? __ldg(bt_row + j) : 0; };
    auto fetch = [&](int i, int second) -> int {
        const long long tok = t0 + (static_cast<long long>(woff) + static_cast<long long>(i) *
                                                                        wstride) * kTile;
        return entry(tok / p.block_size + second);
    };
    int win_cur = fetch(lane, 0);
    int win_next = fetch(32 + lane, 0);
    int win2_cur = split ? fetch(lane, 1) : 0;
    int win2_next = split ? fetch(32 + lane, 1) : 0;
    int win_base = 0;

    // Query fragments (the B operand of S^T = K Q^T): lane holds head
    // lane/4 + 8 nt of the unit, dims 2*(lane%4)+{0,1} and +8 of every 16-dim
    // step; padded heads are 0.
    uint32_t qf[NT8][KT][2];
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
        const int h = (lane >> 2) + 8 * nt;
        const T *qrow = static_cast<const T *>(p.q) +
                        (static_cast<size_t>(seq) * p.num_q_heads + qhead0 + (h < gh ? h : 0)) * D;
        const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow);
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            qf[nt][kk][0] = h < gh ? __ldg(q32 + (kk * 16 + 2 * (lane & 3)) / 2) : 0u;
            qf[nt][kk][1] = h < gh ? __ldg(q32 + (kk * 16 + 8 + 2 * (lane & 3)) / 2) : 0u;
        }
    }

    const int t1 = span();
    if (t1 < 0) return true;   // CTA-uniform: every thread resolves the same span
    const int ntiles = (t1 - t0 + kTile - 1) / kTile;
    const int my_tiles = woff < ntiles ? (ntiles - woff + wstride - 1) / wstride : 0;

    auto advance = [&](int i) {   // warp-uniform, called with i = 0, 1, 2, ...
        if (i - win_base >= 32) {
            win_cur = win_next;
            win2_cur = win2_next;
            win_base += 32;
            win_next = fetch(win_base + 32 + lane, 0);
            if (split) win2_next = fetch(win_base + 32 + lane, 1);
        }
    };

    const uint32_t stage0 = smem_u32(smem) + warp * NS * SM::kStageBytes;
    auto issue = [&](int i) {
        advance(i);
        const int b = __shfl_sync(0xffffffffu, win_cur, i - win_base);
        int b2 = split ? __shfl_sync(0xffffffffu, win2_cur, i - win_base) : 0;
        if (lane == 0) {
            const int tt = t0 + (woff + i * wstride) * kTile;
            // an entry outside the cache becomes an out-of-range TMA box (zeros)
            if (static_cast<unsigned>(b) >= static_cast<unsigned>(p.num_blocks))
                atomicOr(p.status, kBadBlock);
            if (split) {
                // the second block only when the tile reaches into it; else an
                // out-of-range box (zeros, never read: its rows are masked)
                if (tt + 8 >= t1)
                    b2 = -1;
                else if (static_cast<unsigned>(b2) >= static_cast<unsigned>(p.num_blocks))
                    atomicOr(p.status, kBadBlock);
            }
            const uint32_t st = (uses + i) % NS;
            const uint32_t bar = bar0 + (warp * NS + st) * 8;
            const uint32_t dk = stage0 + st * SM::kStageBytes;
            const int row = split ? 0 : tt % p.block_size;
            mbar_expect_tx(bar, SM::kStageBytes);
            const uint64_t once = l2_evict_first_policy();   // read once: evict first
            tma_load_tile_hint<D>(dk, tmK, bar, kvh, row, b, b2, split, once);
            tma_load_tile_hint<D>(dk + SM::kTileBytes, tmV, bar, kvh, row, b, b2, split, once);
        }
    };

    float o[KT][NT8][4];
#pragma unroll
    for (int mt = 0; mt < KT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    float m[NT8][2], l[NT8][2];
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) m[nt][0] = m[nt][1] = -INFINITY, l[nt][0] = l[nt][1] = 0.f;

    const int mi = lane >> 3, ri = lane & 7;
    const int rowK = (mi & 1) * 8 + ri, hiK = mi >> 1;   // S^T A operand (K, row-major)
    const int rowV = (mi >> 1) * 8 + ri, hiV = mi & 1;   // O^T A operand (V^T via .trans)
    const int r0 = lane >> 2;

    for (int i = 0; i < NS && i < my_tiles; ++i) issue(i);

    bool ok = true;
    for (int i = 0; i < my_tiles; ++i) {
        const uint32_t st = (uses + i) % NS;
        const uint32_t bar = bar0 + (warp * NS + st) * 8;
        if (!mbar_wait_bounded(bar, ((uses + i) / NS) & 1u)) {
            // Give the copies already issued a bounded chance to land, then stop.
            for (int j = i + 1; j < my_tiles && j < i + NS; ++j)
                mbar_wait_bounded(bar0 + (warp * NS + (uses + j) % NS) * 8, ((uses + j) / NS) & 1u);
            if (lane == 0) atomicOr(p.status, kWaitTimeout);
            ok = false;
            break;
        }
        const uint32_t kb = stage0 + st * SM::kStageBytes;
        const uint32_t vb = kb + SM::kTileBytes;
        const int tt = t0 + (woff + i * wstride) * kTile;
        const int nvalid = min(kTile, t1 - tt);
        if (nvalid < kTile) {
            // Rows past the sequence end hold whatever the block holds; zero
            // their V so that 0 * garbage cannot reach the accumulator.
            uint8_t *vtile = smem + (vb - smem_u32(smem));
            // (16 - nvalid) rows x (D/64) pieces of 128 bytes, 8 uint4 each
            const int n16 = (kTile - nvalid) * (D / 64) * 8;
            for (int e = lane; e < n16; e += 32) {
                const int rp = e >> 3, row = nvalid + rp / (D / 64), c = rp % (D / 64);
                *reinterpret_cast<uint4 *>(vtile + row_piece_offset<D>(row, c) + (e & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        // S^T[16 tokens][HP heads] = K[16][D] . Q^T[D][HP]
        float sacc[NT8][4];
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            uint32_t a[4];
            ldsm_x4(a, kb + swz<D>(rowK, kk * 16 + hiK * 8));
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt) Mma<T>::run(sacc[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
        }
        uint32_t pb0[NT8], pb1[NT8];
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt) {
            // lane: tokens r0 and r0+8, heads 2*(lane%4)+{0,1} of n-tile nt
            const float y0 = r0 < nvalid ? sacc[nt][0] * p.scale_log2 : -INFINITY;
            const float y1 = r0 < nvalid ? sacc[nt][1] * p.scale_log2 : -INFINITY;
            const float y2 = r0 + 8 < nvalid ? sacc[nt][2] * p.scale_log2 : -INFINITY;
            const float y3 = r0 + 8 < nvalid ? sacc[nt][3] * p.scale_log2 : -INFINITY;
            float mx0 = fmaxf(y0, y2), mx1 = fmaxf(y1, y3);
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
            }
            const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
            const float a0 = ex2(m[nt][0] - mn0), a1 = ex2(m[nt][1] - mn1);
            const float p0 = ex2(y0 - mn0), p1 = ex2(y1 - mn1);
            const float p2 = ex2(y2 - mn0), p3 = ex2(y3 - mn1);
            l[nt][0] = l[nt][0] * a0 + (p0 + p2);
            l[nt][1] = l[nt][1] * a1 + (p1 + p3);
            m[nt][0] = mn0;
            m[nt][1] = mn1;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
                o[mt][nt][0] *= a0;
                o[mt][nt][1] *= a1;
                o[mt][nt][2] *= a0;
                o[mt][nt][3] *= a1;
            }
            // P^T operand: transpose the (token, head) pairs into (head, token) pairs.
            pb0[nt] = movmatrix_t(Mma<T>::pack(p0, p1));
            pb1[nt] = movmatrix_t(Mma<T>::pack(p2, p3));
        }
        // O^T[D][HP heads] += V^T[D][16] . P^T[16][HP]
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
            uint32_t a[4];
            ldsm_x4_t(a, vb + swz<D>(rowV, mt * 16 + hiV * 8));
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt) Mma<T>::run(o[mt][nt], a, pb0[nt], pb1[nt]);
        }
        __syncwarp();
        if (i + NS < my_tiles) issue(i + NS);
    }
    uses += my_tiles;
    if (!ok) *s_abort = 1;   // benign race: every writer stores 1

    // Per-lane exp-sums cover the lane's tokens: sum over the 8 lanes of a head.
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
            l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], x);
            l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], x);
        }

    __syncthreads();   // every warp is done reading its stages
    float *sm_o = reinterpret_cast<float *>(smem);              // [NW][HP][D]
    float *sm_m = sm_o + NW * HP * D;                            // [NW][HP]
    float *sm_l = sm_m + NW * HP;                                // [NW][HP]
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
        const int hb = 8 * nt + 2 * (lane & 3);
        if (lane < 4) {
            sm_m[warp * HP + hb] = m[nt][0];
            sm_m[warp * HP + hb + 1] = m[nt][1];
            sm_l[warp * HP + hb] = l[nt][0];
            sm_l[warp * HP + hb + 1] = l[nt][1];
        }
        float *w0 = sm_o + (warp * HP + hb) * D;
        float *w1 = w0 + D;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
            const int dim = mt * 16 + r0;
            w0[dim] = o[mt][nt][0];
            w1[dim] = o[mt][nt][1];
            w0[dim + 8] = o[mt][nt][2];
            w1[dim + 8] = o[mt][nt][3];
        }
    }
    __syncthreads();
    const bool write = (*s_abort == 0);
    const int Hq = p.num_q_heads;
    constexpr int NT = NW * 32;
    const bool clustered = csize > 1;
    // Per head: the merged maximum M and sum L of the warps' states, and the
    // weight of each warp's normalised output, exp(m_w - M) / L * (its own
    // sum, folded into o_w), so that an output element is a plain weighted
    // sum of the warps' o_w: one pass over the heads, not one per element.
    __shared__ float s_coef[NW][HP];
    __shared__ float s_hm[HP], s_hl[HP];
    if (threadIdx.x < gh) {
        const int h = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * HP + h]);
        float c[NW], L = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            c[w] = M != -INFINITY ? ex2(sm_m[w * HP + h] - M) : 0.f;
            L += c[w] * sm_l[w * HP + h];
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) s_coef[w][h] = c[w] * inv;
        s_hm[h] = M;
        s_hl[h] = L;
    }
    __syncthreads();
    auto merged = [&](int h, int dim) -> float {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) acc += s_coef[w][h] * sm_o[(w * HP + h) * D + dim];
        return acc;
    };
    if (!clustered) {
        for (int e = threadIdx.x; e < gh * D && write; e += NT) {
            const int h = e / D, dim = e - (e / D) * D;
            const float res = merged(h, dim);
            const int head = qhead0 + h;
            if (out_kind == kOutFinal) {
                static_cast<T *>(p.out)[(static_cast<size_t>(seq) * Hq + head) * D + dim] =
                    Mma<T>::cvt(res);
            } else {
                size_t srow;
                if (out_kind == kOutPartialDense)
                    srow = (static_cast<size_t>(seq) * Hq + head) * p.max_parts + part;
                else
                    srow = static_cast<size_t>(slot) * Hq + head;
                // the reduce reads the partials next: keep them in L2
                const uint64_t keep_l2 = l2_evict_last_policy();
                st_global_hint(p.tmp_out + srow * D + dim, res, keep_l2);
                if (dim == 0) {
                    st_global_hint(p.exp_sums + srow, s_hl[h], keep_l2);
                    st_global_hint(p.max_logits + srow,
                                   s_hm[h] == -INFINITY ? -INFINITY : s_hm[h] * kLn2, keep_l2);
                }
            }
        }
    } else {
        // this CTA's merged output for the thread's elements, kept in registers
        // Values go four at a time (a thread holds quads of consecutive output
        // elements, sent with 16-byte stores): a quarter of the transfers.
        constexpr int KQ = (HP * D / 4 + NT - 1) / NT;   // quads per thread, at most
        float4 keep[KQ];
#pragma unroll
        for (int k = 0; k < KQ; ++k) {
            const int e = 4 * (threadIdx.x + k * NT);
            keep[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < gh * D) {
                const int h = e / D, dim = e - (e / D) * D;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float c = s_coef[w][h];
                    const float4 v = *reinterpret_cast<const float4 *>(sm_o + (w * HP + h) * D + dim);
                    keep[k].x += c * v.x;
                    keep[k].y += c * v.y;
                    keep[k].z += c * v.z;
                    keep[k].w += c * v.w;
                }
            }
        }
        cluster_sync();   // every CTA is done with its stages and its merge area
        // send each of this CTA's values to the CTA that finishes its slice
        const int E = gh * D;
        const int slice = ((E + csize - 1) / csize + 3) / 4 * 4;   // whole quads
        const uint32_t base = smem_u32(smem);
        if (write) {
#pragma unroll
            for (int k = 0; k < KQ; ++k) {
                const int e = 4 * (threadIdx.x + k * NT);
                if (e < E) {
                    const int owner = e / slice;
                    dsmem_st_v4(dsmem_addr(base + SM::kInO + (crank * slice + e - owner * slice) * 4,
                                           owner),
                                keep[k]);
                }
            }
            for (int t = threadIdx.x; t < csize * gh; t += NT) {
                const int dst = t / gh, h = t - dst * gh;
                dsmem_st_f32(dsmem_addr(base + SM::kInM + (crank * HP + h) * 4, dst), s_hm[h]);
                dsmem_st_f32(dsmem_addr(base + SM::kInL + (crank * HP + h) * 4, dst), s_hl[h]);
            }
        }
        if (threadIdx.x < csize)
            dsmem_st_s32(dsmem_addr(base + SM::kInAbort + crank * 4, threadIdx.x), write ? 0 : 1);
        cluster_sync();   // every CTA's values of this CTA's slice have arrived
        const float *in_o = reinterpret_cast<const float *>(smem + SM::kInO);
        const float *in_m = reinterpret_cast<const float *>(smem + SM::kInM);
        const float *in_l = reinterpret_cast<const float *>(smem + SM::kInL);
        const int *in_abort = reinterpret_cast<const int *>(smem + SM::kInAbort);
        bool any_abort = false;
        for (int r = 0; r < csize; ++r) any_abort |= in_abort[r] != 0;
        const int e0 = crank * slice, e1 = min(e0 + slice, E);
        if (!any_abort && e0 < e1) {
            // per head of the slice: the weight of each CTA's normalised output
            __shared__ float s_cw[SM::kMaxCluster][HP];
            const int h_lo = e0 / D, h_hi = (e1 - 1) / D;
            if (threadIdx.x <= h_hi - h_lo) {
                const int h = h_lo + threadIdx.x;
                float M = -INFINITY;
                for (int r = 0; r < csize; ++r) M = fmaxf(M, in_m[r * HP + h]);
                float L = 0.f;
                for (int r = 0; r < csize; ++r) {
                    const float w = M != -INFINITY ? ex2(in_m[r * HP + h] - M) * in_l[r * HP + h]
                                                   : 0.f;
                    s_cw[r][h] = w;
                    L += w;
                }
                const float inv = L > 0.f ? 1.f / L : 0.f;
                for (int r = 0; r < csize; ++r) s_cw[r][h] *= inv;
            }
            __syncthreads();
            T *orow = static_cast<T *>(p.out) + (static_cast<size_t>(seq) * Hq + qhead0) * D;
            for (int e = e0 + threadIdx.x; e < e1; e += NT) {
                const int h = e / D;
                float acc = 0.f;
                for (int r = 0; r < csize; ++r) acc += s_cw[r][h] * in_o[r * slice + e - e0];
                orow[e] = Mma<T>::cvt(acc);
            }
        }
    }
    // The merge wrote this memory through the generic proxy; order those
    // writes before any later TMA into it, then let every thread finish.
    fence_proxy_async_smem();
    __syncthreads();
    return ok;
}

// ---------------------------------------------------------------------------
// Attention kernel: single-pass grid, partitioned grid, or persistent work list.
// Grid y / the units' second field index (KV head, head group) pairs.
// ---------------------------------------------------------------------------
template <typename T, int D, int NW, int NS, int MODE, int HP>
__global__ void __launch_bounds__(NW * 32)
    pa_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Params p) {
    using SM = Smem<D, NW, NS, HP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ int s_abort;
    __shared__ int s_next;
    const uint32_t bar0 = smem_u32(smem + SM::kBarOffset);
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        s_abort = 0;
    }
    if (threadIdx.x < NW * NS) mbar_init(bar0 + threadIdx.x * 8, 1);
    fence_mbar_init();
    __syncthreads();
    grid_dep_wait();   // inputs (and the work list) are complete from here on

    uint32_t uses = 0;
    const int cap = p.max_blocks * p.block_size;
    if constexpr (MODE == kModeSingle) {
        // grid (cluster size, Hkv x head groups, S); the CTAs of one cluster share a unit
        const int crank = blockIdx.x, vkh = blockIdx.y, seq = blockIdx.z;
        attend_unit<T, D, NW, NS, HP>(
            p, &tmK, &tmV, smem, bar0, uses, seq, vkh, 0,
            [&]() { return clamp_len(p.seq_lens, seq, cap, p.status); }, kOutFinal, 0, 0,
            &s_abort, crank, p.cluster);
    } else if constexpr (MODE == kModePartitioned) {
        const int part = blockIdx.x, vkh = blockIdx.y, seq = blockIdx.z;
        const int P = p.partition_size;
        const int t0 = part * P;
        attend_unit<T, D, NW, NS, HP>(
            p, &tmK, &tmV, smem, bar0, uses, seq, vkh, t0,
            [&]() {
                const int L = clamp_len(p.seq_lens, seq, cap, p.status);
                int n = (L + P - 1) / P;
                if (n > p.max_parts) {
                    if (part == 0 && vkh == 0 && threadIdx.x == 0)
                        atomicOr(p.status, kTooManyParts);
                    n = p.max_parts;
                }
                return part < n ? min(t0 + P, L) : -1;
            },
            kOutPartialDense, part, 0, &s_abort);
    } else {
        const int total = *p.unit_count;
        if (threadIdx.x == 0) s_next = atomicAdd(p.unit_counter, 1);
        __syncthreads();
        int u = s_next;
        while (u < total) {
            int nxt = 0;
            if (threadIdx.x == 0) nxt = atomicAdd(p.unit_counter, 1);   // prefetch the next unit
            const int4 d = p.units[u];
            const int seq = d.x, vkh = d.y, part = d.z, kind = d.w;
            bool ok;
            if (kind == kOutFinal) {
                ok = attend_unit<T, D, NW, NS, HP>(
                    p, &tmK, &tmV, smem, bar0, uses, seq, vkh, 0,
                    [&]() { return clamp_len(p.seq_lens, seq, cap, p.status); }, kOutFinal, 0, 0,
                    &s_abort);
            } else {
                const int P = p.partition_size;
                const int t0 = part * P;
                ok = attend_unit<T, D, NW, NS, HP>(
                    p, &tmK, &tmV, smem, bar0, uses, seq, vkh, t0,
                    [&]() { return min(t0 + P, clamp_len(p.seq_lens, seq, cap, p.status)); },
                    kOutPartialCompact, part, __ldg(p.part_base + seq) + part, &s_abort);
            }
            if (threadIdx.x == 0) s_next = nxt;
            __syncthreads();
            if (!ok || s_abort) break;   // s_abort is CTA-uniform here
            u = s_next;
        }
    }
    grid_dep_trigger();   // the reduce (or the next step) may launch
}

// ---------------------------------------------------------------------------
// Phase 2: log-sum-exp merge of the partials of one (sequence, query head).
// The merge weights are exp(m_p - M) * l_p with M the maximum over the
// partitions.  Each warp streams its partitions once, keeping a running
// maximum and rescaling its running sums when the maximum grows (the same
// value up to rounding), then the warps' states are merged with the same
// weights.  Loads of kReduceUnroll partitions are issued before any is used.
// ---------------------------------------------------------------------------
// Threads per (sequence, head): the dense reduce (few sequences with many
// partitions) uses 512; the compact one (many sequences with fewer
// partitions) uses 128 so that more sequences are in flight at once.
// Threads per reduce CTA.  The dense form (one CTA per (sequence, head))
// runs 256: at 512 a 32 x 16-row batch took 1.7 waves of CTAs and the
// reduce ran 14.3 us where 256 runs 12.3 (8 x 100K: 12.3 -> 10.3 us).
template <bool COMPACT> struct ReduceThreads { static constexpr int value = COMPACT ? 128 : 256; };
// Partitions each warp loads before accumulating (head_dim 256 keeps fewer
// so that two CTAs fit per SM).
template <int D> struct ReduceUnroll { static constexpr int value = D <= 128 ? 8 : 4; };

// One (sequence, query head): the merged output of its n partitions.  The
// first round of loads is issued for the first nb (an upper bound on n
// known without reading seq_lens) partitions before n is needed, so the
// length read and the partial reads overlap; slots at or past n are dropped
// by selection (never by multiplying, so unwritten slots cannot leak in).
template <typename T, int D, int kReduceThreads>
__device__ __forceinline__ void reduce_one(const ReduceParams &r, int s, int h, size_t stat0,
                                           size_t pstride, int nb, int n_known) {
    constexpr int NWR = kReduceThreads / 32;
    constexpr int VEC = D / 32;   // floats per lane: 2, 4 or 8
    constexpr int U = ReduceUnroll<D>::value;
    __shared__ float s_m[NWR];
    __shared__ float s_l[NWR];
    __shared__ float s_acc[NWR][D];
    const int Hq = r.num_q_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    T *out = static_cast<T *>(r.out) + (static_cast<size_t>(s) * Hq + h) * D;

    float m_run = -INFINITY, l_run = 0.f;   // log2-domain running max, weight sum
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    // n_known < 0: n comes from seq_lens[s], read after the first round's
    // loads are issued
    int n = -1;
    const int len_raw = n_known < 0 ? __ldg(r.seq_lens + s) : 0;
    auto resolve_n = [&]() {
        if (n_known >= 0) return n_known;
        int L = len_raw;
        if (L < 0 || L > r.len_cap) {
            if (threadIdx.x == 0) atomicOr(r.status, kLenClamped);
            L = L < 0 ? 0 : r.len_cap;
        }
        const int np = (L + r.partition_size - 1) / r.partition_size;
        return np < r.max_parts ? np : r.max_parts;
    };
    for (int q0 = warp; q0 < (n < 0 ? nb : n); q0 += NWR * U) {
        float mq[U], lq[U], x[U][VEC];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = q0 + u * NWR;
            const int qc = q < nb ? q : nb - 1;   // always a slot of the buffer
            const size_t si = stat0 + qc * pstride;
            mq[u] = __ldg(r.max_logits + si);
            lq[u] = __ldg(r.exp_sums + si);
            const float *src = r.tmp_out + si * D + lane * VEC;
#pragma unroll
            for (int v = 0; v < VEC; v += (VEC >= 4 ? 4 : 2)) {
                if constexpr (VEC >= 4) {
                    const float4 t = __ldg(reinterpret_cast<const float4 *>(src + v));
                    x[u][v] = t.x;
                    x[u][v + 1] = t.y;
                    x[u][v + 2] = t.z;
                    x[u][v + 3] = t.w;
                } else {
                    const float2 t = __ldg(reinterpret_cast<const float2 *>(src + v));
                    x[u][v] = t.x;
                    x[u][v + 1] = t.y;
                }
            }
        }
        if (n < 0) n = resolve_n();
        bool live[U];
        float mb = m_run;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            live[u] = q0 + u * NWR < n;
            mq[u] = live[u] ? mq[u] * kLog2e : -INFINITY;
            mb = fmaxf(mb, mq[u]);
        }
        if (mb == -INFINITY) continue;   // no live partition in this round (past n)
        const float sc = ex2(m_run - mb);   // 0 while nothing is accumulated yet
        l_run *= sc;
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[v] *= sc;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (live[u]) {
                const float w = ex2(mq[u] - mb) * lq[u];
                l_run += w;
#pragma unroll
                for (int v = 0; v < VEC; ++v) acc[v] += w * x[u][v];
            }
        }
        m_run = mb;
    }
    if (n < 0) n = resolve_n();   // this warp had no first-round partition
    if (lane == 0) {
        s_m[warp] = m_run;
        s_l[warp] = l_run;
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) s_acc[warp][lane * VEC + v] = acc[v];
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWR; ++w) M = fmaxf(M, s_m[w]);
    float tot = 0.f;
    if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NWR; ++w) tot += ex2(s_m[w] - M) * s_l[w];
    }
    for (int i = threadIdx.x; i < D; i += kReduceThreads) {
        float a = 0.f;
        if (tot > 0.f) {
#pragma unroll
            for (int w = 0; w < NWR; ++w) a += ex2(s_m[w] - M) * s_acc[w][i];
        }
        out[i] = Mma<T>::cvt(tot > 0.f ? a / tot : 0.f);   // n == 0 gives zeros
    }
    __syncthreads();   // the shared arrays are reused by the CTA's next item
}

// Dense layout: grid (Hq, S), one (sequence, head) per CTA.  Compact layout
// (the mixed step): grid (Hq, G); CTA row y takes the entries y, y + G, ... of
// the planner's list of partitioned sequences (sequence, first slot, count),
// so no CTA is spent on sequences that were finished in one pass.
template <typename T, int D, bool COMPACT>
__global__ void __launch_bounds__(ReduceThreads<COMPACT>::value, 2)
    pa_reduce_kernel(const ReduceParams r) {
    constexpr int NT = ReduceThreads<COMPACT>::value;
    const int h = blockIdx.x;
    const int Hq = r.num_q_heads;
    grid_dep_wait();   // the attention kernel's partials are complete
    grid_dep_trigger();
    if constexpr (COMPACT) {
        const int count = *r.pseq_count;
        for (int y = blockIdx.y; y < count; y += gridDim.y) {
            const int4 e = r.pseq_list[y];   // (sequence, first slot, partitions, -)
            if (e.z <= 0) {
                // every partition of the sequence was dropped by the planner
                // (flagged there): zeros, and no slot is read
                T *o = static_cast<T *>(r.out) + (static_cast<size_t>(e.x) * Hq + h) * D;
                for (int i = threadIdx.x; i < D; i += NT) o[i] = Mma<T>::cvt(0.f);
                continue;
            }
            reduce_one<T, D, NT>(r, e.x, h, static_cast<size_t>(e.y) * Hq + h, Hq, e.z, e.z);
        }
    } else {
        const int s = blockIdx.y;
        reduce_one<T, D, NT>(r, s, h, (static_cast<size_t>(s) * Hq + h) * r.max_parts, 1,
                             r.max_parts, -1);
    }
}

}  // namespace pa
