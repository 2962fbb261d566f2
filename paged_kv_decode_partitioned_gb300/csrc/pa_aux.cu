// pa_aux.cu -- the work-list planner of the mixed decode step and the
// block-table gather test kernel, with their launchers.
#include "pa_launch.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// Work-list planner: one CTA per sequence.  Unit order: every single-pass
// unit (sequence order), then every partition unit (slot-major, KV head
// minor).  part_base[s] is the compact partial slot of partition 0 of s.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 256;

__global__ void __launch_bounds__(kPlanThreads) pa_plan_kernel(const PlanParams pp) {
    __shared__ int s_red[2][kPlanThreads / 32];
    grid_dep_wait();      // seq_lens are complete
    grid_dep_trigger();   // the attention kernel may launch: it waits for this grid
    const int s = blockIdx.x;
    const int P = pp.partition_size, thr = pp.single_pass_max_len;
    // partitions a sequence gets: ceil(L / P), at most max_parts (the
    // planner's prefix sums use the same clamped count, so the units and
    // slots of the sequences stay contiguous when one is cut short)
    auto parts_of = [&](int L) { return L <= thr ? 0 : min((L + P - 1) / P, pp.max_parts); };
    auto len_of = [&](int i) {
        int L = __ldg(pp.seq_lens + i);
        return L < 0 ? 0 : (L > pp.len_cap ? pp.len_cap : L);
    };
    // counts over sequences before s (and the totals over all of them)
    int singles_before = 0, slots_before = 0, singles_all = 0, slots_all = 0;
    for (int i = threadIdx.x; i < pp.num_seqs; i += kPlanThreads) {
        const int L = len_of(i);
        const int np = parts_of(L);
        const int single = (L <= thr) ? 1 : 0;
        singles_all += single;
        slots_all += np;
        if (i < s) {
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
        if ((threadIdx.x & 31) == 0) {
            s_red[0][threadIdx.x >> 5] = a;
            s_red[1][threadIdx.x >> 5] = b;
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

    const int Hkv = pp.num_kv_heads;
    int L = __ldg(pp.seq_lens + s);
    if (L < 0 || L > pp.len_cap) {
        if (threadIdx.x == 0) atomicOr(pp.status, kLenClamped);
        L = L < 0 ? 0 : pp.len_cap;
    }
    if (L <= thr) {
        for (int k = threadIdx.x; k < Hkv; k += kPlanThreads)
            pp.units[singles_before * Hkv + k] = make_int4(s, k, 0, kOutFinal);
        if (threadIdx.x == 0) pp.part_base[s] = -1;
    } else {
        int np = (L + P - 1) / P;
        // The workspace was sized for at most max_parts partitions per
        // sequence and max_slots in all (the caller's bounds on the longest
        // sequence and on the batch's tokens): partitions past either bound
        // are dropped and flagged.
        const int room = slots_before < pp.max_slots ? pp.max_slots - slots_before : 0;
        if (np > pp.max_parts || np > room) {
            if (threadIdx.x == 0) atomicOr(pp.status, kTooManyParts);
            np = min(np, min(pp.max_parts, room));
        }
        const int base_unit = singles_all * Hkv + min(slots_before, pp.max_slots) * Hkv;
        for (int k = threadIdx.x; k < np * Hkv; k += kPlanThreads)
            pp.units[base_unit + k] = make_int4(s, k % Hkv, k / Hkv, kOutPartialCompact);
        if (threadIdx.x == 0) {
            pp.part_base[s] = slots_before;
            // entry at the sequence's rank among the partitioned sequences
            pp.pseq_list[s - singles_before] = make_int4(s, slots_before, np, 0);
        }
    }
    if (s == 0 && threadIdx.x == 0) {
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
    const cudaError_t e = launch_dependent(pa_plan_kernel, dim3(pp.num_seqs), dim3(kPlanThreads),
                                           0, st, nullptr, pp);
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
