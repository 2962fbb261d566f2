// pa_prefill.cuh -- paged prefix-prefill attention for GB300 (sm_103a).
//
// The operation (page: project_6 commit cd0d9e1, "qwen3_6_scripts", the
// prefix-prefill part of the paged_attn.py rewrite): a chunk of new tokens of
// each sequence attends to the sequence's whole cached context and, causally,
// to the chunk itself.  The new tokens' K/V are already in the paged cache,
// so chunk row i of sequence s (n chunk tokens, L cached tokens in all) sits
// at position p = L - n + i and attends to cache tokens 0..p.
//
// GB300 design: the work is a dense contraction (chunk rows x context tokens
// x head_dim), so it runs on the tensor cores.  A CTA takes up to 128 query
// rows of one (sequence, KV head) -- row = (chunk token, query head of the
// GQA group), so every row of the CTA shares every K/V tile -- in 8 compute
// warps of 16 rows each, plus one producer warp.  The producer walks the
// block table (a lane-distributed window of 16-token box ids) and streams
// 32-token K and V tiles through a 4-stage shared-memory ring with TMA (the
// decode path's tensor map: one box per 64-element piece of 16 rows,
// 128-byte swizzle), completing "full" mbarriers; each compute warp runs an
// online-softmax loop on warp MMAs (m16n8k16, fp32 accumulate): S = Q K^T
// with Q held in registers, the causal mask per row, P taken straight from
// the S accumulator as the A operand of O += P V, then an arrive on the
// stage's "empty" mbarrier.  Every wait is bounded.
#pragma once

#include "pa_launch.cuh"

namespace pa {

template <int D>
struct PrefillCfg {
    static constexpr int kWarps = 8;                      // compute warps
    static constexpr int kRows = kWarps * 16;             // query rows per CTA
    static_assert(kRows == kPrefillRows, "the host sizes the grid with kPrefillRows");
    static constexpr int kKv = 32;                        // cache tokens per stage
    static constexpr int kBoxes = kKv / kTile;            // 16-token boxes per stage
    static constexpr int kStages = 4;
    static constexpr int kBoxBytes = kTile * D * 2;       // one 16-row box, all pieces
    static constexpr int kTileBytes = kBoxes * kBoxBytes; // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kBarOffset = kStages * kStageBytes;
    static constexpr int kThreads = (kWarps + 1) * 32;
    static constexpr int kLaunchBytes = kBarOffset + 2 * kStages * 8 + 1024;
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Keep the low / high bf16|f16 half of a packed pair when the flag is set.
__device__ __forceinline__ uint32_t pair_mask(bool lo, bool hi) {
    return (lo ? 0x0000ffffu : 0u) | (hi ? 0xffff0000u : 0u);
}

template <typename T, int D>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 1)
    pa_prefill_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    using C = PrefillCfg<D>;
    constexpr int KT = D / 16;   // k-steps of S = Q K^T
    constexpr int NO = D / 8;    // n-tiles of O
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t base = smem_u32(smem);
    const uint32_t full0 = base + C::kBarOffset;
    const uint32_t empty0 = full0 + C::kStages * 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the tiles nearest the end of a chunk see the most context: launch them first
    const int qt = gridDim.x - 1 - blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
    const int g = p.group;

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
    const int ntiles = (kv_end + C::kKv - 1) / C::kKv;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(full0 + i * 8, 1);
            mbar_init(empty0 + i * 8, C::kWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == C::kWarps) {
        // ------------------------------ producer ------------------------------
        const int32_t *bt_row = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
        const int nbox = (kv_end + kTile - 1) / kTile;
        auto fetch = [&](int bx) -> int {
            if (bx >= nbox) return 0;
            const int b = __ldg(bt_row + (bx * kTile) / p.block_size);
            if (static_cast<unsigned>(b) >= static_cast<unsigned>(p.num_blocks))
                atomicOr(p.status, kBadBlock);   // the TMA reads zeros there
            return b;
        };
        // lane l holds the block of box win_base + l (and of the next 32 boxes)
        int win_cur = fetch(lane), win_next = fetch(32 + lane), win_base = 0;
        int issued = 0;
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % C::kStages;
            if (j >= C::kStages) {
                const bool w = mbar_wait_bounded(empty0 + st * 8, ((j / C::kStages) - 1) & 1u);
                if (!__all_sync(0xffffffffu, w)) {
                    if (lane == 0) atomicOr(p.status, kWaitTimeout);
                    break;
                }
            }
            if (j * C::kBoxes - win_base >= 32) {
                win_cur = win_next;
                win_base += 32;
                win_next = fetch(win_base + 32 + lane);
            }
            int phys[C::kBoxes];
#pragma unroll
            for (int k = 0; k < C::kBoxes; ++k)
                phys[k] = __shfl_sync(0xffffffffu, win_cur, j * C::kBoxes + k - win_base);
            if (lane == 0) {
                int boxes = 0;
#pragma unroll
                for (int k = 0; k < C::kBoxes; ++k) boxes += (j * C::kBoxes + k < nbox);
                const uint32_t bar = full0 + st * 8;
                const uint32_t dk = base + st * C::kStageBytes;
                mbar_expect_tx(bar, static_cast<uint32_t>(boxes * 2 * C::kBoxBytes));
#pragma unroll
                for (int k = 0; k < C::kBoxes; ++k) {
                    const int bx = j * C::kBoxes + k;
                    if (bx < nbox) {
                        const int row = (bx * kTile) % p.block_size;
                        tma_load_tile<D>(dk + k * C::kBoxBytes, &tmK, bar, kvh, row, phys[k]);
                        tma_load_tile<D>(dk + C::kTileBytes + k * C::kBoxBytes, &tmV, bar, kvh,
                                         row, phys[k]);
                    }
                }
            }
            issued = j + 1;
        }
        // Do not leave while copies of this CTA are still landing (only a
        // timed-out consumer can make this wait do anything).
        for (int j = issued > C::kStages ? issued - C::kStages : 0; j < issued; ++j)
            (void)mbar_wait_bounded(full0 + (j % C::kStages) * 8, (j / C::kStages) & 1u);
        return;
    }

    // ------------------------------ consumers ------------------------------
    // This lane's rows: rr0 = warp*16 + lane/4 and rr1 = rr0 + 8, row = token*g + head.
    const int rows_used = g * ntok;
    const bool active = warp * 16 < rows_used;
    const int rr0 = warp * 16 + (lane >> 2), rr1 = rr0 + 8;
    const bool w0 = rr0 < rows_used, w1 = rr1 < rows_used;
    const int tq0 = w0 ? rr0 / g : ntok - 1, hq0 = w0 ? rr0 % g : 0;
    const int tq1 = w1 ? rr1 / g : ntok - 1, hq1 = w1 ? rr1 % g : 0;
    const int pos0 = pos_first + tq0, pos1 = pos_first + tq1;   // last visible token
    const int Hq = p.num_q_heads;
    const size_t off0 = (static_cast<size_t>(row0 + tok0 + tq0) * Hq + kvh * g + hq0) * D;
    const size_t off1 = (static_cast<size_t>(row0 + tok0 + tq1) * Hq + kvh * g + hq1) * D;
    const int cpair = 2 * (lane & 3);

    uint32_t qa[KT][4];   // Q as the A operand, k-step kk
    if (active) {
        const uint32_t *a = reinterpret_cast<const uint32_t *>(static_cast<const T *>(p.q) + off0);
        const uint32_t *b = reinterpret_cast<const uint32_t *>(static_cast<const T *>(p.q) + off1);
        const int c = lane & 3;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            qa[kk][0] = __ldg(a + kk * 8 + c);
            qa[kk][1] = __ldg(b + kk * 8 + c);
            qa[kk][2] = __ldg(a + kk * 8 + 4 + c);
            qa[kk][3] = __ldg(b + kk * 8 + 4 + c);
        }
    }
    float o[NO][4];
#pragma unroll
    for (int nt = 0; nt < NO; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int mi = lane >> 3, ri = lane & 7;
    const int krow = (mi >> 1) * 8 + ri, kcol = (mi & 1) * 8;   // K rows: B of Q K^T
    const int vrow = (mi & 1) * 8 + ri, vcol = (mi >> 1) * 8;   // V rows: B of P V (.trans)
    bool ok = true;

    for (int j = 0; j < ntiles; ++j) {
        const int st = j % C::kStages;
        const bool w = mbar_wait_bounded(full0 + st * 8, (j / C::kStages) & 1u);
        if (!__all_sync(0xffffffffu, w)) {
            if (lane == 0) atomicOr(p.status, kWaitTimeout);
            ok = false;
            break;
        }
        if (active) {
            const uint32_t kb = base + st * C::kStageBytes;
            const uint32_t vb = kb + C::kTileBytes;
            const int t0 = j * C::kKv;
            // S[16 rows][32 tokens] = Q K^T
            float sc[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t b[4];
                    ldsm_x4(b, kb + h2 * C::kBoxBytes + swz<D>(krow, kk * 16 + kcol));
                    Mma<T>::run(sc[2 * h2], qa[kk], b[0], b[1]);
                    Mma<T>::run(sc[2 * h2 + 1], qa[kk], b[2], b[3]);
                }
            }
            // log2-domain logits; tokens past a row's position are masked
            // (this also discards the unloaded / stale rows of the last stage)
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int t = t0 + nt * 8 + cpair;
                sc[nt][0] = t <= pos0 ? sc[nt][0] * p.scale_log2 : -INFINITY;
                sc[nt][1] = t + 1 <= pos0 ? sc[nt][1] * p.scale_log2 : -INFINITY;
                sc[nt][2] = t <= pos1 ? sc[nt][2] * p.scale_log2 : -INFINITY;
                sc[nt][3] = t + 1 <= pos1 ? sc[nt][3] * p.scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
                mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
            }
#pragma unroll
            for (int x = 1; x < 4; x <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
            }
            // every row sees token 0 in the first tile, so the new max is finite
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float a0 = ex2(m0 - mn0), a1 = ex2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            float s0 = 0.f, s1 = 0.f;
            uint32_t pa[2][4];   // P as the A operand of the two 16-token k-steps
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const float e0 = ex2(sc[nt][0] - mn0), e1 = ex2(sc[nt][1] - mn0);
                const float e2 = ex2(sc[nt][2] - mn1), e3 = ex2(sc[nt][3] - mn1);
                s0 += e0 + e1;
                s1 += e2 + e3;
                pa[nt >> 1][(nt & 1) * 2] = Mma<T>::pack(e0, e1);
                pa[nt >> 1][(nt & 1) * 2 + 1] = Mma<T>::pack(e2, e3);
            }
            l0 = l0 * a0 + s0;
            l1 = l1 * a1 + s1;
#pragma unroll
            for (int nt = 0; nt < NO; ++nt) {
                o[nt][0] *= a0;
                o[nt][1] *= a0;
                o[nt][2] *= a1;
                o[nt][3] *= a1;
            }
            // O[16 rows][D] += P[16][32] V[32][D].  In the last stage the V rows
            // at or past kv_end were not loaded (or hold cache data past the
            // context): their P is 0, but 0 * NaN is not, so zero them here.
            const bool tail = t0 + C::kKv > kv_end;
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int tv = t0 + k2 * 16 + cpair;   // tokens of this lane's B halves
                const uint32_t mlo = pair_mask(tv < kv_end, tv + 1 < kv_end);
                const uint32_t mhi = pair_mask(tv + 8 < kv_end, tv + 9 < kv_end);
#pragma unroll
                for (int np = 0; np < NO / 2; ++np) {
                    uint32_t b[4];
                    ldsm_x4_t(b, vb + k2 * C::kBoxBytes + swz<D>(vrow, np * 16 + vcol));
                    if (tail) {
                        b[0] &= mlo;
                        b[1] &= mhi;
                        b[2] &= mlo;
                        b[3] &= mhi;
                    }
                    Mma<T>::run(o[2 * np], pa[k2], b[0], b[1]);
                    Mma<T>::run(o[2 * np + 1], pa[k2], b[2], b[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + st * 8);
    }
    if (!ok || !active) return;
#pragma unroll
    for (int x = 1; x < 4; x <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, x);
        l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    }
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    T *out0 = static_cast<T *>(p.out) + off0;
    T *out1 = static_cast<T *>(p.out) + off1;
#pragma unroll
    for (int nt = 0; nt < NO; ++nt) {
        const int dim = nt * 8 + cpair;
        if (w0)
            *reinterpret_cast<uint32_t *>(out0 + dim) =
                Mma<T>::pack(o[nt][0] * inv0, o[nt][1] * inv0);
        if (w1)
            *reinterpret_cast<uint32_t *>(out1 + dim) =
                Mma<T>::pack(o[nt][2] * inv1, o[nt][3] * inv1);
    }
}

template <typename T, int D>
inline cudaError_t launch_prefill_d(const CUtensorMap &tmK, const CUtensorMap &tmV,
                                    const PrefillParams &p, dim3 grid, cudaStream_t st) {
    using C = PrefillCfg<D>;
    static std::atomic<int> done[kMaxDevices];
    auto k = pa_prefill_kernel<T, D>;
    cudaError_t e = ensure_smem(k, C::kLaunchBytes, done);
    if (e != cudaSuccess) return e;
    k<<<grid, C::kThreads, C::kLaunchBytes, st>>>(tmK, tmV, p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill(int D, const CUtensorMap &tmK, const CUtensorMap &tmV,
                           const PrefillParams &p, dim3 grid, cudaStream_t st) {
    if (D == 64) return launch_prefill_d<T, 64>(tmK, tmV, p, grid, st);
    if (D == 128) return launch_prefill_d<T, 128>(tmK, tmV, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace pa
