// pa_moe.cu -- MoE router and token regrouping kernels for GB300 (sm_103a).
//
// The operations (page: project_6 commit cd0d9e1, "qwen3_6_scripts", the MoE
// prefill rewrite: 256 experts x top_k = 8, flatten the T x K token-expert
// pairs, sort them by expert so each expert's tokens are contiguous, gather
// the hidden rows in that order, scatter the expert outputs back with
// index_add_; page: commit 490ff98, "Dockerfile": the topk_softmax router
// kernel, which the pages rebuilt for a 64-wide warp):
//   * topk_softmax: one 32-lane warp per token; each lane holds E/32
//     consecutive logits (a 16-byte load per lane for bf16 at E = 256).  The
//     top-k are chosen on the logits themselves (softmax is monotonic), k
//     rounds of a warp arg-max on order-preserving keys, so the chosen ids are
//     exact whatever the rounding of the probabilities: for 16-bit logits the
//     key and the expert id pack into one u32 (one redux.sync per round on
//     per-lane sorted values), for fp32 two reductions per round (largest key,
//     then lowest id holding it).  The softmax max is the first winner (16-bit)
//     or a warp reduction (fp32); the normaliser is a warp sum.
//   * sort: a stable counting sort in three launches -- per-chunk expert
//     histograms, one CTA turning them into each chunk's first position per
//     expert, and a scatter in which each warp walks its share of the chunk in
//     order, ranking equal experts inside a 32-pair step with __match_any_sync.
//   * gather: token-major -- one warp reads a token's hidden row once and
//     writes it to the sorted positions of the token's K pairs (streaming
//     stores), so every hidden byte crosses DRAM once and every regrouped
//     byte is written once.
//   * scatter-back: index_add_ written as a gather-reduce -- one warp per
//     (token, 1 KB block of the row) sums the token's K weighted rows in fp32
//     in slot order and rounds once, so the result is deterministic and needs
//     no atomics.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <utility>

#include "pa_launch.h"

namespace pa {

namespace {

// Programmatic dependent launch: the kernels of the MoE chain are launched so
// that the next one may start while the previous one drains.  Each kernel
// waits, before its first global access, for the previous grid in the stream
// to complete with its memory visible (a no-op when launched without the
// attribute), and lets the next grid launch once its own work is issued.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// VPL consecutive logits of one lane as fp32 (exact for every input type).
template <typename TL, int VPL>
__device__ __forceinline__ void load_logits(const TL *row, int lane, float (&x)[VPL]) {
    const TL *src = row + lane * VPL;
    constexpr int kBytes = VPL * static_cast<int>(sizeof(TL));
    if constexpr (kBytes % 16 == 0) {
        constexpr int kPer = 16 / static_cast<int>(sizeof(TL));
#pragma unroll
        for (int c = 0; c < VPL / kPer; ++c) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + c);
            const TL *e = reinterpret_cast<const TL *>(&v);
#pragma unroll
            for (int i = 0; i < kPer; ++i) x[c * kPer + i] = to_f32(e[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < VPL; ++i) x[i] = to_f32(src[i]);
    }
}

// Order-preserving map of a float to an unsigned key (larger float, larger
// key; -0 and +0 share one key as they compare equal; every float maps to a
// key >= 1, so 0 can mean "none").
__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t u = __float_as_uint(x == 0.f ? 0.f : x);
    const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return k == 0u ? 1u : k;
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// 16-bit logits (bf16, f16): the same order-preserving map on the raw bits
// (-0 and +0 share a key), and its inverse.
__device__ __forceinline__ uint32_t order_key16(uint32_t h) {
    h = h == 0x8000u ? 0u : h;
    return (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
}
__device__ __forceinline__ uint32_t key16_bits(uint32_t k) {
    return (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
}
__device__ __forceinline__ float bits16_f32(uint32_t h, __nv_bfloat16) { return __uint_as_float(h << 16); }
__device__ __forceinline__ float bits16_f32(uint32_t h, __half) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// VPL consecutive 16-bit logits of one lane as raw bits.
template <int VPL>
__device__ __forceinline__ void load_bits16(const uint16_t *row, int lane, uint32_t (&h)[VPL]) {
    const uint16_t *src = row + lane * VPL;
    if constexpr (VPL % 8 == 0) {
#pragma unroll
        for (int c = 0; c < VPL / 8; ++c) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[c * 8 + 2 * i] = w[i] & 0xffffu;
                h[c * 8 + 2 * i + 1] = w[i] >> 16;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < VPL; ++i) h[i] = __ldg(src + i);
    }
}

// Descending bitonic sort of n (a power of two) keys in registers.
template <int n>
__device__ __forceinline__ void sort_desc(uint32_t (&v)[n]) {
#pragma unroll
    for (int k = 2; k <= n; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    const uint32_t a = v[i], b = v[l];
                    const bool desc = (i & k) == 0;
                    v[i] = desc ? max(a, b) : min(a, b);
                    v[l] = desc ? min(a, b) : max(a, b);
                }
            }
}

}  // namespace

// Router for 16-bit logits.  A logit's order key takes 16 bits, so key and
// expert id pack into one u32, (key << 16) | (0xffff - id): the largest packed
// value is the largest logit and, among equal logits, the lowest id.  Each lane
// sorts its packed values once; a round is then one warp max of the lanes'
// heads, and the lane whose head won moves to its next value.  The row max of
// the softmax is the first round's winner, and with renormalisation the sum
// over all experts cancels, so only the top-k exponentials are taken.
template <typename TL, int VPL>
__device__ __forceinline__ void topk_softmax_16(const TopkParams &p, int t, int lane) {
    constexpr int E = VPL * 32;
    uint32_t h[VPL], v[VPL];
    load_bits16<VPL>(static_cast<const uint16_t *>(p.logits) + static_cast<size_t>(t) * E, lane, h);
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        v[i] = (order_key16(h[i]) << 16) | (0xffffu - static_cast<uint32_t>(lane * VPL + i));
    if constexpr (VPL > 1) sort_desc<VPL>(v);
    uint32_t mine = 0u, first = 0u;   // lane r keeps the winner of round r
    for (int r = 0; r < p.topk; ++r) {
        const uint32_t top = __reduce_max_sync(0xffffffffu, v[0]);
        if (r == 0) first = top;
        if (lane == r) mine = top;
        const bool own = v[0] == top;   // packed values are unique
#pragma unroll
        for (int i = 0; i + 1 < VPL; ++i) v[i] = own ? v[i + 1] : v[i];
        v[VPL - 1] = own ? 0u : v[VPL - 1];
    }
    const float m = bits16_f32(key16_bits(first >> 16), TL());
    float w = lane < p.topk ? __expf(bits16_f32(key16_bits(mine >> 16), TL()) - m) : 0.f;
    float s = 0.f;   // the normaliser: the top-k's exponentials, or every expert's
    if (p.renormalize) {
        s = w;
    } else {
#pragma unroll
        for (int i = 0; i < VPL; ++i) s += __expf(bits16_f32(h[i], TL()) - m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane < p.topk) {
        p.weights[static_cast<size_t>(t) * p.topk + lane] = w / s;
        p.ids[static_cast<size_t>(t) * p.topk + lane] = static_cast<int>(0xffffu - (mine & 0xffffu));
    }
}

template <typename TL, int VPL>
__global__ void __launch_bounds__(256) pa_topk_softmax_kernel(const TopkParams p) {
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= p.num_tokens) return;
    if constexpr (sizeof(TL) == 2) {
        topk_softmax_16<TL, VPL>(p, t, lane);
        pdl_trigger();
        return;
    }
    constexpr int E = VPL * 32;
    float x[VPL];
    load_logits<TL, VPL>(static_cast<const TL *>(p.logits) + static_cast<size_t>(t) * E, lane, x);
    float m = x[0];
#pragma unroll
    for (int i = 1; i < VPL; ++i) m = fmaxf(m, x[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) z += __expf(x[i] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);

    // Each round: the lane's best remaining logit as an order-preserving
    // unsigned key (0 = nothing left), the warp's largest key by one redux, then
    // the lowest expert id holding that key by a second one.
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) key[i] = order_key(x[i]);
    int my_id = 0;          // lane r keeps the id and logit of choice r
    float my_x = 0.f;
    for (int r = 0; r < p.topk; ++r) {
        uint32_t bk = 0;
        int bi = 0;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (key[i] > bk) {   // strict: the lowest index wins a tie inside the lane
                bk = key[i];
                bi = i;
            }
        const uint32_t top = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t e = __reduce_min_sync(
            0xffffffffu, bk == top ? static_cast<uint32_t>(lane * VPL + bi) : 0xffffffffu);
        if (static_cast<int>(e) / VPL == lane) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (i == static_cast<int>(e) % VPL) key[i] = 0;
        }
        if (lane == r) {
            my_id = static_cast<int>(e);
            my_x = key_value(top);
        }
    }
    float w = lane < p.topk ? __expf(my_x - m) / z : 0.f;
    if (p.renormalize) {
        float s = w;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        w = w / s;
    }
    if (lane < p.topk) {
        p.weights[static_cast<size_t>(t) * p.topk + lane] = w;
        p.ids[static_cast<size_t>(t) * p.topk + lane] = my_id;
    }
    pdl_trigger();   // the next kernel in the stream may launch
}

// ---------------------------------------------------------------------------
// Stable counting sort of the flat pairs by expert id
// ---------------------------------------------------------------------------
constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortChunk = 2048;   // pairs per CTA (256 per warp)

// hist[c][e] = pairs of chunk c with expert e
__global__ void __launch_bounds__(kSortThreads) pa_moe_hist_kernel(const SortParams p) {
    pdl_wait();
    extern __shared__ int h[];
    for (int e = threadIdx.x; e < p.num_experts; e += kSortThreads) h[e] = 0;
    __syncthreads();
    const int c0 = blockIdx.x * kSortChunk;
    const int c1 = min(c0 + kSortChunk, p.num_pairs);
    bool bad = false;
    for (int i = c0 + threadIdx.x; i < c1; i += kSortThreads) {
        const int e = __ldg(p.expert_ids + i);
        if (static_cast<unsigned>(e) < static_cast<unsigned>(p.num_experts))
            atomicAdd(&h[e], 1);
        else
            bad = true;
    }
    if (bad) atomicOr(p.status, kBadExpert);
    __syncthreads();
    for (int e = threadIdx.x; e < p.num_experts; e += kSortThreads)
        p.hist[static_cast<size_t>(blockIdx.x) * p.num_experts + e] = h[e];
    pdl_trigger();   // the next kernel in the stream may launch
}

// One CTA: hist[c][e] becomes the first sorted position of chunk c's pairs of
// expert e; offsets[e] the first position of expert e, offsets[E] the total.
__global__ void __launch_bounds__(1024) pa_moe_scan_kernel(const SortParams p) {
    pdl_wait();
    __shared__ int part[1024];    // [group][expert] chunk sums
    __shared__ int first[1024];   // [expert] first sorted position
    __shared__ int warp_sum[32];
    // thread = (chunk group g, expert e): the chunks are split over the
    // 1024 / E groups, so every thread walks only its share of the columns
    const int E = p.num_experts, C = p.num_chunks;
    const int G = 1024 / E;
    const int g = threadIdx.x / E, e = threadIdx.x - g * E;
    const bool act = g < G;
    const int per = (C + G - 1) / G;
    const int c_begin = act ? min(g * per, C) : 0, c_end = act ? min(c_begin + per, C) : 0;
    constexpr int kBatch = 16;   // loads issued together, ahead of any use
    int sum = 0;
    for (int c0 = c_begin; c0 < c_end; c0 += kBatch) {
        int v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            v[i] = c0 + i < c_end ? p.hist[static_cast<size_t>(c0 + i) * E + e] : 0;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) sum += v[i];
    }
    part[threadIdx.x] = sum;
    __syncthreads();
    int pre = 0, tot = 0;   // this group's offset within expert e, and e's total
    if (act) {
        for (int q = 0; q < G; ++q) {
            const int x = part[q * E + e];
            pre += q < g ? x : 0;
            tot += x;
        }
    }
    // exclusive scan of the totals over the experts (threads 0 .. E-1)
    const int val = g == 0 ? tot : 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = val;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += x;
        }
        warp_sum[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    if (g == 0) {
        const int start = incl - val + (warp > 0 ? warp_sum[warp - 1] : 0);
        first[e] = start;
        p.offsets[e] = start;
        if (e == E - 1) p.offsets[E] = start + tot;
    }
    __syncthreads();
    if (act) {   // hist[c][e] becomes the first position of chunk c's pairs of e
        int run = first[e] + pre;
        for (int c0 = c_begin; c0 < c_end; c0 += kBatch) {
            int v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                v[i] = c0 + i < c_end ? p.hist[static_cast<size_t>(c0 + i) * E + e] : 0;
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (c0 + i < c_end) p.hist[static_cast<size_t>(c0 + i) * E + e] = run;
                run += v[i];
            }
        }
    }
    pdl_trigger();   // the next kernel in the stream may launch
}

// Each warp places its 256 pairs in order: within a 32-pair step, pairs with
// the same expert are ranked by lane (match_any + popc of the lower lanes).
__global__ void __launch_bounds__(kSortThreads) pa_moe_place_kernel(const SortParams p) {
    pdl_wait();
    extern __shared__ int cnt[];   // [kSortWarps][E]: this warp's next position per expert
    const int E = p.num_experts;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kSortWarps * E; i += kSortThreads) cnt[i] = 0;
    __syncthreads();
    constexpr int kSub = kSortChunk / kSortWarps;
    const int w0 = blockIdx.x * kSortChunk + warp * kSub;
    const int w1 = min(w0 + kSub, p.num_pairs);
    int *mine = cnt + warp * E;
    for (int i = w0 + lane; i < w1; i += 32) {
        const int e = __ldg(p.expert_ids + i);
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&mine[e], 1);
    }
    __syncthreads();
    // per-warp counts -> per-warp first positions
    for (int e = threadIdx.x; e < E; e += kSortThreads) {
        int run = p.hist[static_cast<size_t>(blockIdx.x) * E + e];
        for (int w = 0; w < kSortWarps; ++w) {
            const int n = cnt[w * E + e];
            cnt[w * E + e] = run;
            run += n;
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        int e = i < w1 ? __ldg(p.expert_ids + i) : -1;
        const bool ok = static_cast<unsigned>(e) < static_cast<unsigned>(E);
        if (!ok) e = -1;
        const unsigned same = __match_any_sync(0xffffffffu, e);
        if (ok) {
            const int pos = mine[e] + __popc(same & lt);
            p.sorted_pairs[pos] = i;
            p.pair_pos[i] = pos;
        } else if (i < w1) {
            p.pair_pos[i] = -1;
        }
        __syncwarp();
        if (ok && (same & lt) == 0) mine[e] += __popc(same);
        __syncwarp();
    }
    pdl_trigger();   // the next kernel in the stream may launch
}

// ---------------------------------------------------------------------------
// Gather and scatter-back
// ---------------------------------------------------------------------------
// sorted_hidden[pair_pos[p]] = hidden[p / K], token-major: one warp reads its
// token's row once (16-byte loads, up to 8 per lane in flight) and writes it
// to the K sorted positions of the token's pairs with streaming stores, so
// every hidden byte crosses DRAM once.
__global__ void __launch_bounds__(256) pa_moe_gather_kernel(const MoeGatherParams p) {
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= p.num_tokens) return;
    const int K = p.topk;
    int my_pos = -1;   // lane k: sorted position of pair (t, k)
    if (lane < K) {
        my_pos = __ldg(p.pair_pos + static_cast<size_t>(t) * K + lane);
        if (my_pos != -1 && static_cast<unsigned>(my_pos) >= static_cast<unsigned>(p.num_rows)) {
            atomicOr(p.status, kBadExpert);   // a position outside the output: not written
            my_pos = -1;
        }
    }
    const int n16 = p.row_bytes / 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.hidden) +
                                                       static_cast<size_t>(t) * p.row_bytes);
    uint4 *out = static_cast<uint4 *>(p.out);
    for (int c0 = 0; c0 < n16; c0 += 256) {   // 8 chunks of 16 bytes per lane per round
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + i * 32 + lane;
            if (c < n16) v[i] = __ldcs(src + c);
        }
        for (int k = 0; k < K; ++k) {
            const int r = __shfl_sync(0xffffffffu, my_pos, k);
            if (r < 0) continue;   // a pair that was not placed (flagged by the sort)
            uint4 *dst = out + static_cast<size_t>(r) * n16;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = c0 + i * 32 + lane;
                if (c < n16) __stcs(dst + c, v[i]);
            }
        }
    }
    pdl_trigger();   // the next kernel in the stream may launch
}

// 16-byte columns (8 elements) of a scatter-back work unit: 1 KB of a row
constexpr int kScatterBlock = 64;

template <typename T>
struct Vec8;
template <>
struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ void unpack(const uint4 &v, float (&f)[8]) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = __bfloat1622float2(h[i]);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
    static __device__ __forceinline__ uint4 pack(const float (&f)[8]) {
        uint4 v;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        return v;
    }
};
template <>
struct Vec8<__half> {
    static __device__ __forceinline__ void unpack(const uint4 &v, float (&f)[8]) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = __half22float2(h[i]);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
    static __device__ __forceinline__ uint4 pack(const float (&f)[8]) {
        uint4 v;
        __half2 *h = reinterpret_cast<__half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        return v;
    }
};

// out[t] = sum_k w[t][k] * y[pair_pos[t*K + k]], fp32 in slot order, one rounding.
template <typename T>
__global__ void __launch_bounds__(256) pa_moe_scatter_kernel(const MoeScatterParams p) {
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // one warp per (token, 1 KB block of columns): a warp per whole token gave
    // 1.7 waves of warps at 16384 tokens, whose partial last wave left the
    // DRAM under-used for a sixth of the launch
    const int n16 = p.hidden_size / 8;
    const int nblk = (n16 + kScatterBlock - 1) / kScatterBlock;
    const long long u = static_cast<long long>(blockIdx.x) * 8 + warp;
    if (u >= static_cast<long long>(p.num_tokens) * nblk) return;
    const int t = static_cast<int>(u / nblk);
    const int cb = static_cast<int>(u % nblk) * kScatterBlock;
    const int K = p.topk;
    int my_pos = 0;
    float my_w = 0.f;
    if (lane < K) {
        my_pos = __ldg(p.pair_pos + static_cast<size_t>(t) * K + lane);
        my_w = __ldg(p.weights + static_cast<size_t>(t) * K + lane);
        if (static_cast<unsigned>(my_pos) >= static_cast<unsigned>(p.num_pairs)) {
            atomicOr(p.status, kBadExpert);   // a pair that was never placed adds nothing
            my_pos = -1;
        }
    }
    const uint4 *y = static_cast<const uint4 *>(p.y);
    uint4 *out = static_cast<uint4 *>(p.out) + static_cast<size_t>(t) * n16;
    // the column loop is uniform over the warp: every lane takes part in the
    // shuffles that broadcast the K (row, weight) pairs
    const int cend = min(cb + kScatterBlock, n16);
    for (int c0 = cb; c0 < cend; c0 += 64) {
        const int c = c0 + lane;
        const bool one = c < cend, two = c + 32 < cend;
        float a0[8], a1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a0[i] = a1[i] = 0.f;
        for (int k = 0; k < K; ++k) {
            const int r = __shfl_sync(0xffffffffu, my_pos, k);
            const float w = __shfl_sync(0xffffffffu, my_w, k);
            if (r < 0) continue;
            const uint4 *row = y + static_cast<size_t>(r) * n16;
            float f[8];
            if (one) {
                Vec8<T>::unpack(__ldg(row + c), f);
#pragma unroll
                for (int i = 0; i < 8; ++i) a0[i] = fmaf(w, f[i], a0[i]);
            }
            if (two) {
                Vec8<T>::unpack(__ldg(row + c + 32), f);
#pragma unroll
                for (int i = 0; i < 8; ++i) a1[i] = fmaf(w, f[i], a1[i]);
            }
        }
        if (one) out[c] = Vec8<T>::pack(a0);
        if (two) out[c + 32] = Vec8<T>::pack(a1);
    }
    pdl_trigger();   // the next kernel in the stream may launch
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
// A launch with programmatic stream serialisation: the kernel may start while
// the previous one in the stream drains; its pdl_wait() orders its accesses.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_topk_softmax(int logits_type, int num_experts, const TopkParams &p,
                                cudaStream_t st) {
    const dim3 grid((p.num_tokens + 7) / 8);
    cudaError_t e = cudaSuccess;
#define PA_TOPK(TL, VPL) e = launch_pdl(pa_topk_softmax_kernel<TL, VPL>, grid, dim3(256), 0, st, p)
#define PA_TOPK_E(TL)                                  \
    switch (num_experts) {                             \
        case 32: PA_TOPK(TL, 1); break;                \
        case 64: PA_TOPK(TL, 2); break;                \
        case 128: PA_TOPK(TL, 4); break;               \
        case 256: PA_TOPK(TL, 8); break;               \
        case 512: PA_TOPK(TL, 16); break;              \
        default: return cudaErrorInvalidValue;         \
    }
    if (logits_type == 0) {
        PA_TOPK_E(__half)
    } else if (logits_type == 1) {
        PA_TOPK_E(__nv_bfloat16)
    } else if (logits_type == 2) {
        PA_TOPK_E(float)
    } else {
        return cudaErrorInvalidValue;
    }
#undef PA_TOPK_E
#undef PA_TOPK
    return e;
}

int moe_sort_chunks(int num_pairs) { return (num_pairs + kSortChunk - 1) / kSortChunk; }

cudaError_t launch_moe_sort(const SortParams &p, cudaStream_t st) {
    const int E = p.num_experts;
    cudaError_t e;
    if (p.num_chunks > 0) {
        e = launch_pdl(pa_moe_hist_kernel, dim3(p.num_chunks), dim3(kSortThreads),
                       E * sizeof(int), st, p);
        if (e != cudaSuccess) return e;
    }
    if ((e = launch_pdl(pa_moe_scan_kernel, dim3(1), dim3(1024), 0, st, p)) != cudaSuccess) return e;
    if (p.num_chunks == 0) return cudaSuccess;
    const int smem = kSortWarps * E * static_cast<int>(sizeof(int));
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(pa_moe_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(pa_moe_place_kernel, dim3(p.num_chunks), dim3(kSortThreads), smem, st, p);
}

cudaError_t launch_moe_gather(const MoeGatherParams &p, cudaStream_t st) {
    return launch_pdl(pa_moe_gather_kernel, dim3((p.num_tokens + 7) / 8), dim3(256), 0, st, p);
}

cudaError_t launch_moe_scatter(bool bf16, const MoeScatterParams &p, cudaStream_t st) {
    const long long nblk = (p.hidden_size / 8 + kScatterBlock - 1) / kScatterBlock;
    const long long units = static_cast<long long>(p.num_tokens) * nblk;
    if (units == 0) return cudaSuccess;
    if ((units + 7) / 8 > INT_MAX) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>((units + 7) / 8));
    return bf16 ? launch_pdl(pa_moe_scatter_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, p)
                : launch_pdl(pa_moe_scatter_kernel<__half>, grid, dim3(256), 0, st, p);
}

}  // namespace pa
