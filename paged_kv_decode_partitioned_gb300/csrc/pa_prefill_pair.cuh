// pa_prefill_pair.cuh -- paged prefix prefill on CTA pairs sharing 2-SM
// tcgen05 MMAs (cta_group::2), for GB300 (sm_103a).
//
// Same operation as pa_prefill_tc.cuh (page: project_6 commit cd0d9e1,
// "qwen3_6_scripts", the prefix-prefill part of the paged_attn.py rewrite):
// each chunk row attends to its sequence's cached context up to its own
// position, through the block table, with the online softmax of the pages'
// tile loop.  What differs is how the work sits on the SMs.
//
// A cluster of two CTAs (a pair, on two SMs) takes 256 query rows of one
// (sequence, KV head): 128 per CTA, row = chunk token x query head of the
// GQA group.  Each MMA is issued once, by one thread of the even CTA, for
// both: S = Q K^T is an M = 256, N = 128 MMA whose A rows (Q) and D rows (S)
// stay in each CTA's own shared / tensor memory, and O += P V an M = 256,
// N = head_dim MMA with P read from each CTA's tensor memory.  B is split by
// columns: each CTA holds half of every K tile (64 of its 128 tokens) and half
// of every V tile (head_dim / 2 of its columns).  So each SM stages half the
// K/V bytes per tile of the single-CTA kernel, which buys the head_dim-256
// layout (its O alone takes 256 tensor-memory columns) a second K/V stage,
// and every loaded K/V byte still feeds 256 rows.  Each CTA keeps two S
// buffers in tensor memory, so the QK of the next tile runs under the
// softmax of the current one.
//
// Warp roles (96 + 128 kSplit NQ threads per CTA: 224 at head_dim 256):
//   warp 0     TMA producer of this CTA's Q rows (once) and K halves, the last
//              warp of its V halves, each through NS stages (one copy per
//              lane).  The copies of both CTAs complete on the even CTA's
//              barriers (the cta_group::2 form of the copy), which the even CTA
//              arms with both halves' bytes, so the MMA warp sees a whole tile
//              land without a message from the odd CTA;
//   warp 1     tensor-memory owner; in the even CTA it runs the pair's fixed
//              MMA sequence, one elected lane issuing each MMA and committing
//              it to both CTAs' barriers;
//   warps 2..  softmax, as in the single-CTA kernel: kSplit warpgroups per
//              Q tile (one by default: a thread per whole row, its S held in
//              registers), P written over S in this CTA's tensor memory and
//              reported to the even CTA; O rescaled in place when a row's max
//              grows by more than 2^8; O / l -> out.
// Arrivals from the odd CTA on the even CTA's barriers are CTA-scope
// releases (a cluster-scope release costs ~3x the round trip between the
// SMs, measured: 945 against 364 cycles) except for the two that publish
// plain stores the MMAs then read (the zeroed Q rows and V tail rows), which
// happen once per CTA.
// Every mbarrier wait is bounded; a role that gives up raises
// PA_DEV_WAIT_TIMEOUT and leaves its loop.  Both CTAs meet at a cluster
// barrier before tensor memory is freed and before either exits, so no MMA,
// copy or remote arrive is in flight against a CTA that has left.
#pragma once

#include "pa_prefill_tc.cuh"

namespace pa {

// Softmax warpgroups per Q tile on pairs (as PA_PREFILL_SPLIT_* for single
// CTAs): one thread per whole row, the row's S held in registers, measured
// 1940 -> 2050 TFLOP/s at head_dim 256 against two warpgroups on column halves.
#ifndef PA_PREFILL_PAIR_SPLIT_D128
#define PA_PREFILL_PAIR_SPLIT_D128 1
#endif
#ifndef PA_PREFILL_PAIR_SPLIT_D256
#define PA_PREFILL_PAIR_SPLIT_D256 1
#endif

template <int D>
struct PrefillPairCfg {
    static_assert(D == 128 || D == 256, "pair layout: head_dim 128 or 256");
    // head_dim 128: two Q tiles per CTA, one S buffer each (the tiles take turns
    // on the tensor pipe, as in the single-CTA kernel); head_dim 256 (its O
    // alone takes 256 tensor-memory columns): one Q tile with two S buffers
    static constexpr int kQTiles = D == 128 ? 2 : 1;
    static constexpr int kSBufs = kQTiles == 2 ? 1 : 2;
    static constexpr int kRows = 128 * kQTiles;       // query rows per CTA
    static constexpr int kN = 128;                    // cache tokens per K/V tile
    static constexpr int kHalfN = kN / 2;             // K tokens each CTA holds
    static constexpr int kPieces = D / 64;            // 64-element pieces of a Q / K row
    static constexpr int kVPieces = D / 128;          // 64-column pieces of V each CTA holds
    static constexpr int kQPiece = kRows * 128;
    static constexpr int kQTileBytes = 128 * 128;     // one Q tile's rows in a piece
    static constexpr int kQBytes = kPieces * kQPiece;
    // K and V land one 16-token box per copy as 8-token groups, the CTA's
    // pieces of each group after one another: [group][piece][8 rows][128 B]
    // (128-byte swizzled); K holds every piece of the CTA's 64 tokens (read
    // K-major), V the CTA's kVPieces pieces of all 128 tokens (MN-major)
    static constexpr int kKBoxBytes = kPieces * 2048;
    static constexpr int kVBoxBytes = kVPieces * 2048;
    static constexpr int kKBytes = (kHalfN / 16) * kKBoxBytes;
    static constexpr int kVBytes = (kN / 16) * kVBoxBytes;
    static constexpr int kStageBytes = kKBytes + kVBytes;
    static constexpr int kStages = D == 128 ? 4 : 2;
    static constexpr int kBarOffset = kQBytes + kStages * kStageBytes;
    // q_full, vtail, mma_done, vtail2, k_full[NS], v_full[NS], k_empty[NS],
    // v_empty[NS]; per Q tile s_full[2], s_free[2], p_full[2], o_full (the
    // first kSBufs of each pair in use).  q_full, k_full, v_full, vtail2 and
    // p_full are the MMA thread's (used in the even CTA), the rest each CTA's own
    static constexpr int kTileBars = 7;
    static constexpr int kNumBars = 4 + 4 * kStages + kTileBars * kQTiles;
    static constexpr int kSlotOffset = kBarOffset + kNumBars * 8;
    // kSplit softmax warpgroups per Q tile, each 1 / kSplit of the S columns of
    // every row; with two, they swap row maxima (two buffers by tile parity)
    // and, at the end, row sums: xbar[2] and xend per Q tile
    static constexpr int kSplit = D == 128 ? PA_PREFILL_PAIR_SPLIT_D128 : PA_PREFILL_PAIR_SPLIT_D256;
    static_assert(kSplit == 1 || kSplit == 2, "one or two softmax warpgroups per Q tile");
    static constexpr int kHalfCols = kN / kSplit;
    static constexpr int kXBarOffset = kSlotOffset + 16;
    static constexpr int kXOffset = kXBarOffset + kQTiles * 3 * 8 + 8;
    static constexpr int kXBytes = kSplit > 1 ? kQTiles * 3 * 2 * 128 * 4 : 0;   // [tile][max0, max1, sum][half][row]
    static constexpr int kLaunchBytes = kXOffset + kXBytes + 1024;
    static constexpr int kSoftmaxWarp0 = 2;
    // warp 0 Q and K producer, warp 1 MMA, the softmax warps, then the V producer
    static constexpr int kVWarp = kSoftmaxWarp0 + 4 * kSplit * kQTiles;
    static constexpr int kThreads = 32 * (kVWarp + 1);
    // tensor memory per Q tile: S buffers [0, kSBufs N), O [kSBufs N, kSBufs N + D)
    static constexpr int kOCol = kSBufs * kN;
    static constexpr int kTileCols = kSBufs * kN + D;
    static constexpr int kTmemCols = 512;
    static_assert(kTileCols * kQTiles <= kTmemCols, "tensor memory plan too large");
    static_assert(kLaunchBytes <= 227 * 1024, "shared memory plan too large");
    static_assert(4 * kPieces <= 32, "one copy per lane");
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Arrive on the barrier at shared::cluster address `bar` (either CTA's),
// releasing this thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}

// Arrive on the barrier at shared::cluster address `bar` with the default
// (CTA-scope) release: the signal for tensor-memory hand-offs ordered by the
// tcgen05 fences around it.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 5-D tiled TMA load into this CTA's shared memory whose completion lands on
// `bar`, an mbarrier in this CTA or in its peer of the pair.
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(PrefillPairCfg<D>::kThreads, 1)
    pa_prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    using C = PrefillPairCfg<D>;
    constexpr int N = C::kN, NS = C::kStages, HC = C::kHalfCols, NQ = C::kQTiles, SB = C::kSBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t base = smem_u32(smem);
    const uint32_t q_smem = base;
    const uint32_t stage0 = base + C::kQBytes;
    const uint32_t bars = base + C::kBarOffset;
    const uint32_t q_full = bars, vtail = bars + 8, mma_done = bars + 16, vtail2 = bars + 24;
    const uint32_t k_full = bars + 32, v_full = k_full + NS * 8;
    const uint32_t k_empty = v_full + NS * 8, v_empty = k_empty + NS * 8;
    // per Q tile t at tile_bars + 56 t: s_full[2] +0, s_free[2] +16, p_full[2] +32, o_full +48
    const uint32_t tile_bars = v_empty + NS * 8;
    const uint32_t slot = base + C::kSlotOffset;
    const uint32_t rank = cluster_ctarank();   // 0: the pair's MMA-issuing CTA
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int npairs = static_cast<int>(gridDim.x) >> 1;
    const int qp = npairs - 1 - static_cast<int>(blockIdx.x >> 1);   // the pair's Q tiles
    const int qt = 2 * qp + static_cast<int>(rank);                   // this CTA's
    const int kvh = blockIdx.y, s = blockIdx.z;
    const int g = p.group, tpc = p.tokens_per_cta;

    // ---- rows and context: the early exits depend on the pair only ----
    const int cap = p.max_blocks * p.block_size;
    const int L = clamp_len(p.seq_lens, s, cap, p.status);
    const int row0 = __ldg(p.q_start + s), row1 = __ldg(p.q_start + s + 1);
    const bool first = blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0;
    if (row0 < 0 || row1 < row0 || row1 > p.num_rows) {
        if (first) atomicOr(p.status, kBadRows);
        return;
    }
    const int n = row1 - row0;
    if (n > L) {
        if (first) atomicOr(p.status, kBadRows);
        return;
    }
    if (first && n > static_cast<int>(gridDim.x) * tpc) atomicOr(p.status, kLenClamped);
    if (2 * qp * tpc >= n) return;   // neither CTA of the pair has a row
    const int tok0 = qt * tpc;
    const int ntok = max(0, min(tpc, n - tok0));   // 0: the odd CTA past the chunk's end
    const int pair_end = min(n, (2 * qp + 2) * tpc);
    const int kv_end = L - n + pair_end;   // cache tokens any row of the pair sees
    const int ntiles = (kv_end + N - 1) / N;
    const int rot = static_cast<int>(gridDim.x / 2) >= PA_PREFILL_ROT_MIN_CTAS
                        ? static_cast<int>((static_cast<unsigned>(qp) * PA_PREFILL_ROT_STEP_PAIR) %
                                           static_cast<unsigned>(ntiles))
                        : 0;
    const int pos_first = L - n + tok0;
    const int rows_used = g * ntok;
    const int j_tail = ntiles - 1 - rot;   // use order of the context's tail tile
    // Q tiles with any row in either CTA (the even CTA has at least the odd one's rows)
    const int rows_even = g * min(tpc, n - 2 * qp * tpc);
    const int nq = NQ > 1 && rows_even > 128 ? 2 : 1;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        mbar_init(q_full, 2);   // the even CTA's arm + the odd CTA's "Q rows in place"
        mbar_init(vtail, 1);
        mbar_init(mma_done, 1);
        mbar_init(vtail2, 2);   // each CTA's zeroed V tail rows
        for (int i = 0; i < NS; ++i) {
            mbar_init(k_full + i * 8, 1);
            mbar_init(v_full + i * 8, 1);
            mbar_init(k_empty + i * 8, 1);
            mbar_init(v_empty + i * 8, 1);
        }
        for (int t = 0; t < NQ; ++t) {
            const uint32_t tb = tile_bars + t * 56;
            for (int i = 0; i < 2; ++i) {
                mbar_init(tb + i * 8, 1);          // s_full
                mbar_init(tb + 16 + i * 8, 1);     // s_free
                mbar_init(tb + 32 + i * 8, 8 * C::kSplit);   // p_full: one arrive per softmax warp of both CTAs
            }
            mbar_init(tb + 48, 1);                 // o_full
            if (C::kSplit > 1)
                for (int i = 0; i < 3; ++i) mbar_init(base + C::kXBarOffset + (t * 3 + i) * 8, 8);
        }
        fence_mbar_init();
    }
    __syncthreads();
    cluster_sync();   // both CTAs run and their barriers are initialised
    if (warp == 1) tc05::alloc2(slot, C::kTmemCols);
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::kSlotOffset);

    if (warp == 0 || warp == C::kVWarp) {
        // ------------------------------ producers ------------------------------
        // warp 0 loads this CTA's Q rows and K halves, the last warp its V halves,
        // so a K copy never waits behind a V stage (one producer for both cost
        // ~9 % at head_dim 128 on single CTAs)
        const int32_t *bt_row = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
        const int nbox = (kv_end + kTile - 1) / kTile;
        constexpr int kKOps = 4;   // this CTA's 4 boxes of K, every piece in one copy
        constexpr int kVOps = 8;   // all 8 boxes of V, this CTA's pieces in one copy
        const bool lead = rank == 0;
        // block_size 8: a 16-token box spans two blocks, a copy each (lane
        // pairs take the two halves of one box)
        const bool b8 = p.block_size < kTile;
        const int op = b8 ? lane >> 1 : lane, half = b8 ? lane & 1 : 0;
        const int k_box = 4 * static_cast<int>(rank) + op % kKOps;
        const int v_box = op % kVOps;
        const int v_piece = static_cast<int>(rank) * C::kVPieces;   // first piece of the box
        auto first_token = [&](int jt, int box) { return (jt * (N / kTile) + box) * kTile + half * (kTile / 2); };
        // block of this lane's K (V) box (half) of tile jt (0 when the lane has
        // no copy or the half lies past the context), read a tile ahead and
        // checked only when the copy is issued
        auto block_of = [&](int jt, int box, bool has) -> int {
            const int tok = first_token(jt, box);
            return has && tok < kv_end ? __ldg(bt_row + tok / p.block_size) : 0;
        };
        // the copy's 8-token group coordinate; -1 (a box of zeros) for a half
        // past the context or a block outside the cache (that one flagged)
        auto group_of = [&](int jt, int box, int b) -> int {
            const int tok = first_token(jt, box);
            if (tok >= kv_end) return -1;
            if (static_cast<unsigned>(b) >= static_cast<unsigned>(p.num_blocks)) {
                atomicOr(p.status, kBadBlock);
                return -1;
            }
            return b * (p.block_size >> 3) + ((tok % p.block_size) >> 3);
        };
        // the even CTA's barrier at the same offset (this CTA's own in the even CTA)
        auto lead_bar = [&](uint32_t bar) -> uint32_t { return lead ? bar : dsmem_addr(bar, 0); };
        const bool k_has = op < kKOps, v_has = op < kVOps;
        if (warp == 0) {
            // Q: the box covers g * tpc rows; rows past it (and every row of a CTA
            // without chunk tokens) are zeroed so they stay finite
            const int qrows = ntok > 0 ? g * tpc : 0;
            if (qrows < C::kRows) {
                for (int c = 0; c < C::kPieces; ++c)
                    for (int e = lane; e < (C::kRows - qrows) * 8; e += 32)
                        *reinterpret_cast<uint4 *>(smem + c * C::kQPiece + qrows * 128 + e * 16) =
                            make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                if (lead) {   // arm q_full with both CTAs' Q bytes
                    const int ntok1 = max(0, min(tpc, n - (2 * qp + 1) * tpc));
                    const int qrows1 = ntok1 > 0 ? g * tpc : 0;
                    mbar_expect_tx(q_full, static_cast<uint32_t>(C::kPieces * 128 * (qrows + qrows1)));
                }
                if (qrows > 0) {
#pragma unroll
                    for (int c = 0; c < C::kPieces; ++c)
                        tma_load_4d_pair(q_smem + c * C::kQPiece, &tmQ, lead_bar(q_full), 0, c, kvh * g,
                                         row0 + tok0);
                }
                if (!lead) mbar_arrive_cluster(lead_bar(q_full));   // zeroed rows published
            }
        }
        auto tile_at = [&](int j) -> int { return j + rot < ntiles ? j + rot : j + rot - ntiles; };
        // 16-token boxes of context tile jt inside the context
        auto boxes_of = [&](int jt) -> int {
            int b = 0;
#pragma unroll
            for (int k = 0; k < N / kTile; ++k) b += jt * (N / kTile) + k < nbox;
            return b;
        };
        // each stream's block lookups go out one of its tiles ahead
        int kb_next = block_of(tile_at(0), k_box, k_has), vb_next = block_of(tile_at(0), v_box, v_has);
        int k_issued = 0, issued = 0;   // tiles whose K (V) copies went out
        bool ok = true;
        // K of use-order tile j (its stage free once the QK of j - NS is done)
        auto issue_k = [&](int j) -> bool {
            const int st = j % NS, jt = tile_at(j), kb = kb_next;
            if (j + 1 < ntiles) kb_next = block_of(tile_at(j + 1), k_box, k_has);
            if (j >= NS) {
                const bool w = mbar_wait_cycles(k_empty + st * 8, ((j / NS) - 1) & 1u);
                if (!__all_sync(0xffffffffu, w)) return false;
            }
            if (lead && lane == 0)   // both CTAs' K halves
                mbar_expect_tx(k_full + st * 8, static_cast<uint32_t>(boxes_of(jt) * C::kPieces * 2048));
            __syncwarp();
            if (k_has && jt * (N / kTile) + k_box < nbox)
                // the cache maps: (element, row in group, piece, head, group)
                tma_load_5d_pair(stage0 + st * C::kStageBytes +
                                     (k_box - 4 * static_cast<int>(rank)) * C::kKBoxBytes +
                                     half * (C::kPieces * 1024),
                                 &tmK, lead_bar(k_full + st * 8), 0, 0, 0, kvh, group_of(jt, k_box, kb));
            k_issued = j + 1;
            return true;
        };
        // V of use-order tile j (its stage free once the PV of j - NS is done)
        auto issue_v = [&](int j) -> bool {
            const int st = j % NS, jt = tile_at(j), vb = vb_next;
            if (j + 1 < ntiles) vb_next = block_of(tile_at(j + 1), v_box, v_has);
            const uint32_t vdst = stage0 + st * C::kStageBytes + C::kKBytes;
            const bool last = jt == ntiles - 1;
            const int boxes = boxes_of(jt);
            if (j >= NS) {
                const bool w = mbar_wait_cycles(v_empty + st * 8, ((j / NS) - 1) & 1u);
                if (!__all_sync(0xffffffffu, w)) return false;
            }
            // the tail tile's V lands on this CTA's own vtail, to be zeroed past
            // the context before the MMA may read it
            const uint32_t vbar = last ? vtail : lead_bar(v_full + st * 8);
            if (lane == 0) {
                if (last)
                    mbar_expect_tx(vtail, static_cast<uint32_t>(boxes * C::kVPieces * 2048));
                else if (lead)   // both CTAs' V halves
                    mbar_expect_tx(v_full + st * 8, static_cast<uint32_t>(boxes * 2 * C::kVPieces * 2048));
            }
            __syncwarp();
            if (v_has && jt * (N / kTile) + v_box < nbox)
                tma_load_5d_pair(vdst + v_box * C::kVBoxBytes + half * (C::kVPieces * 1024), &tmV, vbar,
                                 0, 0, v_piece, kvh, group_of(jt, v_box, vb));
            issued = j + 1;
            if (last) {
                const bool w = mbar_wait_cycles(vtail, 0);
                if (!__all_sync(0xffffffffu, w)) return false;
                const int first_row = kv_end - jt * N;
                const int nchunks = (N - first_row) * C::kVPieces * 8;   // 16-byte chunks
                for (int e = lane; e < nchunks; e += 32) {
                    const int r = first_row + e / (C::kVPieces * 8);
                    const int c = (e / 8) % C::kVPieces;
                    *reinterpret_cast<uint4 *>(smem + (vdst - base) + (r >> 3) * (C::kVPieces * 1024) +
                                               c * 1024 + (r & 7) * 128 + (e & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_cluster(lead_bar(vtail2));   // zeroed rows published
                    if (lead) mbar_arrive_cta(v_full + st * 8);   // the stage's phase moves on
                }
            }
            return true;
        };
        if (warp == 0) {
            for (int j = 0; ok && j < ntiles; ++j) ok = issue_k(j);
        } else {
            for (int j = 0; ok && j < ntiles; ++j) ok = issue_v(j);
        }
        if (!ok && lane == 0) atomicOr(p.status, kWaitTimeout);
        // copies still landing must land before the CTA exits: the even CTA's
        // barriers count both CTAs' bytes, so the even CTA waits for the pair
        if (warp == 0 && lead) {
            (void)mbar_wait_cycles(q_full, 0);
            for (int j = k_issued > NS ? k_issued - NS : 0; j < k_issued; ++j)
                (void)mbar_wait_cycles(k_full + (j % NS) * 8, (j / NS) & 1u);
        }
        if (warp != 0) {
            if (lead)
                for (int j = issued > NS ? issued - NS : 0; j < issued; ++j)
                    if (j != j_tail) (void)mbar_wait_cycles(v_full + (j % NS) * 8, (j / NS) & 1u);
            if (issued > j_tail) (void)mbar_wait_cycles(vtail, 0);
        }
    } else if (warp == 1) {
        // ------------------------- MMA issuer (even CTA) -------------------------
        // The whole warp runs a fixed issue sequence (warp-uniform control flow)
        // and one elected lane issues each MMA and commit: QK of the first SB
        // tiles for every Q tile, then per K/V tile j and Q tile t the PV of j
        // and the QK of j + SB.  Each step waits (suspending, bounded) on the one
        // barrier it needs, and every barrier waited on depends only on MMAs
        // issued earlier in the sequence, so the order cannot deadlock.
        if (rank == 0) {
            constexpr uint32_t kAll = 0xffffffffu;
            constexpr uint32_t idesc_qk = tc05::f16_idesc(TcType<T>::code, 0, 0, N, 256);
            constexpr uint32_t idesc_pv = tc05::f16_idesc(TcType<T>::code, 0, 1, D, 256);
            constexpr uint16_t kBoth = 0x3;
            bool ok = __all_sync(kAll, mbar_wait_cycles(q_full, 0));
            auto wait = [&](uint32_t bar, uint32_t parity) {
                ok = ok && __all_sync(kAll, mbar_wait_cycles(bar, parity));
                return ok;
            };
            // S_j = Q_t K_j^T into S buffer j % SB; the last Q tile's QK frees the K stage
            auto issue_qk = [&](int t, int j) {
                const uint32_t tb = tile_bars + t * 56;
                const uint32_t tcol = tmem + t * C::kTileCols;
                const uint32_t kst = stage0 + (j % NS) * C::kStageBytes;
                const uint32_t qst = q_smem + t * C::kQTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc05::mma2_ss_elect(
                        tcol + (j % SB) * N,
                        tc05::sw128_desc(qst + (kk >> 2) * C::kQPiece + (kk & 3) * 32, 16, 1024),
                        tc05::sw128_desc(kst + (kk >> 2) * 1024 + (kk & 3) * 32, 16, C::kPieces * 1024),
                        idesc_qk, kk > 0 ? 1u : 0u);
                tc05::commit2_elect(tb + (j % SB) * 8, kBoth);   // s_full
                if (t == nq - 1) tc05::commit2_elect(k_empty + (j % NS) * 8, kBoth);
            };
            // O_t += P_j V_j; the last Q tile's PV frees the V stage
            auto issue_pv = [&](int t, int j) {
                const uint32_t tb = tile_bars + t * 56;
                const uint32_t tcol = tmem + t * C::kTileCols;
                const uint32_t vst = stage0 + (j % NS) * C::kStageBytes + C::kKBytes;
#pragma unroll
                for (int kt = 0; kt < N / 16; ++kt)
                    // tokens [16 kt, 16 kt + 16) lie in half (16 kt) / HC, whose P
                    // occupies the first half of that half's S columns
                    tc05::mma2_ts_elect(tcol + C::kOCol,
                                        tcol + (j % SB) * N + ((16 * kt) / HC) * (HC / 2) + kt * 8,
                                        tc05::sw128_desc(vst + kt * C::kVBoxBytes, 1024, C::kVPieces * 1024),
                                        idesc_pv, (j > 0 || kt > 0) ? 1u : 0u);
                // s_free: with one S buffer the commit of the QK issued next
                // (S_{j+1}) tracks this PV as well, so none is needed
                if (SB > 1) tc05::commit2_elect(tb + 16 + (j % SB) * 8, kBoth);
                if (t == nq - 1) tc05::commit2_elect(v_empty + (j % NS) * 8, kBoth);
                if (j == ntiles - 1) tc05::commit2_elect(tb + 48, kBoth);   // o_full
            };
            for (int j = 0; ok && j < SB && j < ntiles; ++j) {
                if (!wait(k_full + (j % NS) * 8, (j / NS) & 1u)) break;
                tc05::fence_after_sync();
                for (int t = 0; t < nq; ++t) issue_qk(t, j);
            }
            for (int j = 0; ok && j < ntiles; ++j) {
                // V of tile j: both halves landed, and in the tail tile both CTAs'
                // rows past the context zeroed
                if (!wait(v_full + (j % NS) * 8, (j / NS) & 1u)) break;
                if (j == j_tail && !wait(vtail2, 0)) break;
                const int jn = j + SB;   // the QK issued behind this tile's PV
                for (int t = 0; t < nq; ++t) {
                    if (!wait(tile_bars + t * 56 + 32 + (j % SB) * 8, (j / SB) & 1u)) break;   // p_full
                    tc05::fence_after_sync();
                    issue_pv(t, j);
                    if (jn < ntiles) {
                        if (t == 0 && !wait(k_full + (jn % NS) * 8, (jn / NS) & 1u)) break;
                        tc05::fence_after_sync();
                        issue_qk(t, jn);
                    }
                }
            }
            if (!ok && lane == 0) atomicOr(p.status, kWaitTimeout);
            tc05::commit2_elect(mma_done, 0x1);
            (void)mbar_wait_cycles(mma_done, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------ softmax ------------------------------
        constexpr int SP = C::kSplit;
        // one thread per whole row keeps the row's S in registers between passes
        constexpr bool RR = SP == 1;
        const int idx = warp - C::kSoftmaxWarp0;
        const int t = idx / (4 * SP);         // the Q tile of this warp
        const int hf = (idx >> 2) % SP;       // the part of the S columns it handles
        if (t < nq) {
            const int quarter = warp & 3;         // tensor-memory lanes 32*quarter .. +31
            const int rl = quarter * 32 + lane;   // row within the Q tile
            const int r = t * 128 + rl;           // row within the CTA
            const bool valid = r < rows_used;
            const int tq = valid ? r / g : (ntok > 0 ? ntok - 1 : 0), hq = valid ? r % g : 0;
            // last cache token the row sees (a CTA without rows takes the pair's last)
            const int pos = ntok > 0 ? pos_first + tq : kv_end - 1;
            const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
            const uint32_t tcol = tmem + lane_base + t * C::kTileCols;
            const uint32_t tb = tile_bars + t * 56;
            const uint32_t xbar = base + C::kXBarOffset + t * 3 * 8;
            float *xch = reinterpret_cast<float *>(smem + C::kXOffset) + t * 3 * 256;
            const float sl2 = p.scale_log2;
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < ntiles; ++j) {
                const int b = j % SB;
                const bool w = mbar_wait_cycles(tb + b * 8, (j / SB) & 1u);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
                tc05::fence_after_sync();
                const uint32_t sb = tcol + b * N + hf * HC;
                const int jt = j + rot < ntiles ? j + rot : j + rot - ntiles;
                const int lim = pos - jt * N - hf * HC;
                const bool full = __all_sync(0xffffffffu, lim >= HC - 1);
                uint32_t sr[RR ? N / 32 : 1][32];
                float pm;
                if constexpr (RR)
                    pm = full ? row_load_max<N, false>(sr, sb, lim) : row_load_max<N, true>(sr, sb, lim);
                else
                    pm = full ? tile_row_max<HC, false, true>(sb, lim)
                              : tile_row_max<HC, true, true>(sb, lim);
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
                mt *= sl2;
                if (j == 0) {
                    m = mt;
                } else if (__any_sync(0xffffffffu, mt > m + 8.f)) {
                    // O must hold P_{j-1} V_{j-1} before it is rescaled.  With one S
                    // buffer, PV_{j-1} went out before QK_j from the same thread, so
                    // the S_j commit waited for above has already seen it finish.
                    if (SB > 1) {
                        const bool w2 = mbar_wait_cycles(tb + 16 + ((j - 1) % SB) * 8, ((j - 1) / SB) & 1u);
                        if (!__all_sync(0xffffffffu, w2)) {
                            ok = false;
                            break;
                        }
                        tc05::fence_after_sync();
                    }
                    const float mn = fmaxf(m, mt);
                    const float alpha = m == mn ? 1.f : ex2(m - mn);
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
                const float mu = m == -INFINITY ? 0.f : m;
                if constexpr (RR)
                    l += full ? row_p_regs<T, N, false>(sr, sb, lim, sl2, mu, 0u, false)
                              : row_p_regs<T, N, true>(sr, sb, lim, sl2, mu, 0u, false);
                else
                    l += full ? tile_row_p<T, HC, false, true>(sb, lim, sl2, mu, 0u, false)
                              : tile_row_p<T, HC, true, true>(sb, lim, sl2, mu, 0u, false);
                tc05::wait_st();
                tc05::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0)
                        mbar_arrive_cta(tb + 32 + b * 8);
                    else
                        mbar_arrive_remote(dsmem_addr(tb + 32 + b * 8, 0));
                }
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
                          (static_cast<size_t>(row0 + tok0 + tq) * p.num_q_heads + kvh * g + hq) * D +
                          hf * (D / SP);
#pragma unroll
                for (int c0 = 0; c0 < D / SP; c0 += 32) {
                    uint32_t rr[32];
                    tc05::ld32(tcol + C::kOCol + hf * (D / SP) + c0, rr);
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) {
                            uint4 v;
                            v.x = Mma<T>::pack(__uint_as_float(rr[i]) * inv, __uint_as_float(rr[i + 1]) * inv);
                            v.y = Mma<T>::pack(__uint_as_float(rr[i + 2]) * inv, __uint_as_float(rr[i + 3]) * inv);
                            v.z = Mma<T>::pack(__uint_as_float(rr[i + 4]) * inv, __uint_as_float(rr[i + 5]) * inv);
                            v.w = Mma<T>::pack(__uint_as_float(rr[i + 6]) * inv, __uint_as_float(rr[i + 7]) * inv);
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
    cluster_sync();   // every MMA, copy, tensor-memory access and remote arrive of the pair is done
    tc05::fence_after_sync();
    if (warp == 1) tc05::dealloc2(tmem, C::kTmemCols);
}

template <typename T, int D>
inline cudaError_t launch_prefill_pair_d(const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                         const CUtensorMap &tmV, const PrefillParams &p,
                                         dim3 grid, cudaStream_t st) {
    using C = PrefillPairCfg<D>;
    static std::atomic<int> done[kMaxDevices];
    auto k = pa_prefill_pair_kernel<T, D>;
    cudaError_t e = ensure_smem(k, C::kLaunchBytes, done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid.x + (grid.x & 1u), grid.y, grid.z);   // whole pairs
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kLaunchBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k, tmQ, tmK, tmV, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pa
