// pa_aux.cu -- the work-list planner of the mixed decode step and the
// block-table gather test kernel, with their launchers.
#include "pa_launch.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// Work-list planner: one CTA per chunk of 1 .. kPlanSeqs sequences.  Unit order:
// every single-pass unit (sequence order), then every partition unit
// (slot-major, head group minor).  part_base[s] is the compact partial slot of
// partition 0 of s.  Each CTA sums the counts of the sequences before its
// chunk (and of all of them) with one pass over the lengths, then a warp scan
// gives each sequence of the chunk its offsets, and the chunk's units are
// written by all of the CTA's threads (a long sequence has hundreds): the
// lengths are read at most 256 S times in all (S^2 / 32 past 8192 sequences),
// not S^2.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 256;
constexpr int kPlanSeqs = 32;   // sequences per CTA at most: one lane each of the scan warp
constexpr int kPlanCtas = 256;  // CTAs the planner aims for: one sequence each up to 256
                                // sequences, then ceil(S / 256) per CTA (at most 32)

__global__ void __launch_bounds__(kPlanThreads) pa_plan_kernel(const PlanParams pp) {
    __shared__ int s_red[2][kPlanThreads / 32];
    __shared__ int s_unit_off[kPlanSeqs + 1], s_dst[kPlanSeqs], s_kind[kPlanSeqs];
    const int chunk = pp.chunk;   // sequences of this CTA (1 .. kPlanSeqs)
    grid_dep_wait();      // seq_lens are complete
    grid_dep_trigger();   // the attention kernel may launch: it waits for this grid
    const int s0 = blockIdx.x * chunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int P = pp.partition_size, thr = pp.single_pass_max_len;
    // partitions a sequence gets: ceil(L / P), at most max_parts (the
    // planner's prefix sums use the same clamped count, so the units and
    // slots of the sequences stay contiguous when one is cut short)
    auto parts_of = [&](int L) { return L <= thr ? 0 : min((L + P - 1) / P, pp.max_parts); };
    auto len_of = [&](int i) {
        int L = __ldg(pp.seq_lens + i);
        return L < 0 ? 0 : (L > pp.len_cap ? pp.len_cap : L);
    };
    // counts over sequences before the chunk (and the totals over all of them)
    int singles_before = 0, slots_before = 0, singles_all = 0, slots_all = 0;
    for (int i = threadIdx.x; i < pp.num_seqs; i += kPlanThreads) {
        const int L = len_of(i);
        const int np = parts_of(L);
        const int single = (L <= thr) ? 1 : 0;
        singles_all += single;
        slots_all += np;
        if (i < s0) {
            singles_before += single;
            slots_before += np;
        }
    }
    auto block_sum2 = [&](int &a, int &b) {
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, x);
            b += __shfl_xor_sync(0xffffffffu, b, x);
        }
        __syncthreads();
        if (lane == 0) {
            s_red[0][warp] = a;
            s_red[1][warp] = b;
        }
        __syncthreads();
        a = b = 0;
#pragma unroll
        for (int w = 0; w < kPlanThreads / 32; ++w) {
            a += s_red[0][w];
            b += s_red[1][w];
        }
    };
    block_sum2(singles_before, slots_before);
    block_sum2(singles_all, slots_all);

    // offsets of the chunk's sequences: an exclusive warp scan (lane = sequence)
    // of their single-pass units, partition slots and work-list units
    const int Hkv = pp.num_kv_heads;
    if (warp == 0) {
        const int s = s0 + lane;
        const bool mine = lane < chunk && s < pp.num_seqs;   // a sequence of the chunk
        int L = 0;
        if (mine) {
            L = __ldg(pp.seq_lens + s);
            if (L < 0 || L > pp.len_cap) {
                atomicOr(pp.status, kLenClamped);
                L = L < 0 ? 0 : pp.len_cap;
            }
        }
        const int single = mine && L <= thr ? 1 : 0;
        const int np = mine ? parts_of(L) : 0;
        int inc_single = single, inc_slots = np;
#pragma unroll
        for (int x = 1; x < 32; x <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, inc_single, x);
            const int b = __shfl_up_sync(0xffffffffu, inc_slots, x);
            if (lane >= x) {
                inc_single += a;
                inc_slots += b;
            }
        }
        const int sb = singles_before + inc_single - single;   // single-pass units before s
        const int pb = slots_before + inc_slots - np;         // partition slots before s
        // the sequence's partitions after the workspace's bounds (the caller's
        // bounds on the longest sequence and on the batch's tokens): partitions
        // past either bound are dropped and flagged
        int npw = 0;
        if (mine && !single) {
            npw = (L + P - 1) / P;
            const int room = pb < pp.max_slots ? pp.max_slots - pb : 0;
            if (npw > pp.max_parts || npw > room) {
                atomicOr(pp.status, kTooManyParts);
                npw = min(npw, min(pp.max_parts, room));
            }
            pp.part_base[s] = pb;
            // entry at the sequence's rank among the partitioned sequences
            pp.pseq_list[s - sb] = make_int4(s, pb, npw, 0);
        } else if (mine) {
            pp.part_base[s] = -1;
        }
        const int nu = mine ? (single ? Hkv : npw * Hkv) : 0;   // its units
        int inc_u = nu;
#pragma unroll
        for (int x = 1; x < 32; x <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, inc_u, x);
            if (lane >= x) inc_u += a;
        }
        if (lane < chunk) {
            s_unit_off[lane] = inc_u - nu;
            s_dst[lane] = single ? sb * Hkv : singles_all * Hkv + min(pb, pp.max_slots) * Hkv;
            s_kind[lane] = single;
        }
        if (lane == chunk - 1) s_unit_off[chunk] = inc_u;
    }
    __syncthreads();
    // the chunk's units, spread over all threads: u -> (sequence j, index k)
    const int total_u = s_unit_off[chunk];
    for (int u = threadIdx.x; u < total_u; u += kPlanThreads) {
        int lo = 0, hi = chunk - 1;   // last j with s_unit_off[j] <= u
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_unit_off[mid] <= u) lo = mid; else hi = mid - 1;
        }
        const int j = lo, k = u - s_unit_off[j];
        pp.units[s_dst[j] + k] = s_kind[j] ? make_int4(s0 + j, k, 0, kOutFinal)
                                           : make_int4(s0 + j, k % Hkv, k / Hkv,
                                                       kOutPartialCompact);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *pp.unit_count = (singles_all + min(slots_all, pp.max_slots)) * Hkv;
        *pp.unit_counter = 0;
        *pp.pseq_count = pp.num_seqs - singles_all;
    }
}

// ---------------------------------------------------------------------------
// Test kernel: gather one 16-token tile of (seq, kvh) through the same tensor
// map, swizzle and block-table indexing the attention kernel uses.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(32)
    pa_gather_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const GatherParams gp) {
    constexpr int kTileBytes = kTile * D * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ alignas(8) uint64_t bar_storage;
    const int tile = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
    const int lane = threadIdx.x;
    const int L = clamp_len(gp.seq_lens, s, gp.max_blocks * gp.block_size, gp.status);
    const int Lc = L < gp.max_len ? L : gp.max_len;
    const int tt = tile * kTile;
    if (tt >= Lc) return;
    const uint32_t bar = smem_u32(&bar_storage);
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const int32_t *bt_row = gp.block_tables + static_cast<size_t>(s) * gp.max_blocks;
    const bool split = gp.block_size < kTile;   // block_size 8: two blocks per tile
    const int b = __ldg(bt_row + tt / gp.block_size);
    // second block of a block-size-8 tile, when the tile reaches into it
    const bool need2 = split && tt + 8 < Lc;
    const int b2 = need2 ? __ldg(bt_row + tt / gp.block_size + 1) : -1;
    if (lane == 0) {
        if (static_cast<unsigned>(b) >= static_cast<unsigned>(gp.num_blocks))
            atomicOr(gp.status, kBadBlock);
        if (need2 && static_cast<unsigned>(b2) >= static_cast<unsigned>(gp.num_blocks))
            atomicOr(gp.status, kBadBlock);
        const int row = split ? 0 : tt % gp.block_size;
        mbar_expect_tx(bar, 2 * kTileBytes);
        tma_load_tile<D>(smem_u32(smem), &tmK, bar, kvh, row, b, b2, split);
        tma_load_tile<D>(smem_u32(smem) + kTileBytes, &tmV, bar, kvh, row, b, b2, split);
    }
    if (!mbar_wait_bounded(bar, 0)) {
        if (lane == 0) atomicOr(gp.status, kWaitTimeout);
        return;
    }
    const int nvalid = min(kTile, Lc - tt);
    const int Hkv = gp.num_kv_heads;
    for (int e = lane; e < nvalid * (D / 8); e += 32) {
        const int row = e / (D / 8), c8 = (e % (D / 8)) * 8;
        const size_t dst = ((static_cast<size_t>(s) * gp.max_len + tt + row) * Hkv + kvh) * D + c8;
        const uint4 kx = *reinterpret_cast<const uint4 *>(smem + swz<D>(row, c8));
        const uint4 vx = *reinterpret_cast<const uint4 *>(smem + kTileBytes + swz<D>(row, c8));
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(gp.k_dense) + dst) = kx;
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(gp.v_dense) + dst) = vx;
    }
}


// Test kernel of the failure path: waits on an mbarrier that nothing will
// complete (no copy is issued), gives up after limit_ns and raises the
// time-out flag exactly as the attention kernel does.
__global__ void __launch_bounds__(32) pa_wait_timeout_kernel(int *status,
                                                             unsigned long long limit_ns) {
    __shared__ alignas(8) uint64_t bar_storage;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (!mbar_wait_bounded(bar, 0, limit_ns) && threadIdx.x == 0) atomicOr(status, kWaitTimeout);
}

cudaError_t launch_wait_timeout_test(int *status, unsigned long long limit_ns, cudaStream_t st) {
    pa_wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_plan(const PlanParams &pp, cudaStream_t st) {
    if (pp.num_seqs <= 0) return cudaSuccess;
    PlanParams q = pp;
    q.chunk = (pp.num_seqs + kPlanCtas - 1) / kPlanCtas;
    if (q.chunk > kPlanSeqs) q.chunk = kPlanSeqs;
    const cudaError_t e =
        launch_dependent(pa_plan_kernel, dim3((pp.num_seqs + q.chunk - 1) / q.chunk),
                         dim3(kPlanThreads), 0, st, nullptr, q);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D>
static cudaError_t launch_gather_d(const CUtensorMap &tmK, const CUtensorMap &tmV,
                                   const GatherParams &gp, dim3 grid, cudaStream_t st) {
    const int bytes = 2 * kTile * D * 2 + 1024;
    cudaError_t e = cudaFuncSetAttribute(pa_gather_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    pa_gather_kernel<D><<<grid, 32, bytes, st>>>(tmK, tmV, gp);
    return cudaGetLastError();
}

cudaError_t launch_gather(int D, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          const GatherParams &gp, dim3 grid, cudaStream_t st) {
    if (D == 64) return launch_gather_d<64>(tmK, tmV, gp, grid, st);
    if (D == 128) return launch_gather_d<128>(tmK, tmV, gp, grid, st);
    if (D == 256) return launch_gather_d<256>(tmK, tmV, gp, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace pa
