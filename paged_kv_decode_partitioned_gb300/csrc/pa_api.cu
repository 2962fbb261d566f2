// pa_api.cu -- the C ABI of libpadecode.so (declared in include/pa_decode.h):
// argument checks, TMA tensor maps over the caches, work decomposition and
// kernel launches.  Every check happens here, before anything is launched.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <mutex>

#include "pa_decode.h"
#include "pa_launch.h"
#include "pa_moe.h"

#ifndef PA_TILE_PIECES
#define PA_TILE_PIECES 1
#endif

namespace {

using namespace pa;

// Device status word (PA_DEV_* flags), one per device that loads the library.
__device__ int g_pa_status_word;

constexpr int kMaxDev = 64;
constexpr int kVersion = 10000;   // 1.0.0

struct DevInfo {
    int *status = nullptr;
    int num_sms = 0;
    bool ready = false;
};

std::mutex g_dev_mu;
DevInfo g_dev[kMaxDev];

int device_info(DevInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return PA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &d = g_dev[dev];
    if (!d.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_status_word) != cudaSuccess) return PA_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PA_ERR_CUDA;
        d.status = static_cast<int *>(p);
        d.num_sms = sms;
        d.ready = true;
    }
    *out = &d;
    return PA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 5-D view of a cache [num_blocks][bs][Hkv][D] for TMA: (element within a
// 64-element piece, piece index, KV head, row in block, block); one box = one
// 64-element piece of 16 rows of one KV head (2 KB; 8 rows for block_size 8),
// 128-byte swizzled.  Out-of-range boxes read zeros.
int make_cache_map(CUtensorMap *m, const void *cache, pa_dtype_t dtype, int D, int Hkv, int bs,
                   int num_blocks) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PA_ERR_NO_DEVICE;
    const cuuint64_t e = 2;
    cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(Hkv),
                          static_cast<cuuint64_t>(bs), static_cast<cuuint64_t>(num_blocks)};
    cuuint64_t strides[4] = {64 * e, D * e, static_cast<cuuint64_t>(Hkv) * D * e,
                             static_cast<cuuint64_t>(bs) * Hkv * D * e};
#if PA_TILE_PIECES
    // 16 rows of one block, or 8 (block_size 8: a tile is two 8-row boxes)
    const cuuint32_t rows = static_cast<cuuint32_t>(bs < kTile ? bs : kTile);
    cuuint32_t box[5] = {64, 1, 1, rows, 1};
#else
    cuuint32_t box[5] = {64, static_cast<cuuint32_t>(D / 64), 1, static_cast<cuuint32_t>(kTile), 1};
#endif
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    5, const_cast<void *>(cache), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// 5-D view of a cache as 8-token groups: (element within a 64-element piece,
// row in the group, piece, KV head, group), group g holding the cache's rows
// 8 g .. 8 g + 7 counted across blocks (block b, row r: g = b * bs / 8 + r / 8;
// bs a multiple of 8).  One box = `pieces` consecutive pieces of `groups`
// consecutive groups of one KV head, landing as [group][piece][8 rows][128 B]
// (128-byte swizzled): the operand layout of the prefill kernels, a uniform
// stride of `pieces` KB between 8-token groups.  Two groups (16 tokens of one
// block) per copy when bs is a multiple of 16, one with block_size 8.
// Out-of-range boxes read zeros.
int make_cache_map_groups(CUtensorMap *m, const void *cache, pa_dtype_t dtype, int D, int Hkv,
                          int bs, int num_blocks, int pieces) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PA_ERR_NO_DEVICE;
    const cuuint64_t e = 2;
    const cuuint64_t row = static_cast<cuuint64_t>(Hkv) * D * e;   // bytes between cache rows
    cuuint64_t dims[5] = {64, 8, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(Hkv),
                          static_cast<cuuint64_t>(num_blocks) * (bs / 8)};
    cuuint64_t strides[4] = {row, 64 * e, D * e, 8 * row};
    cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(pieces), 1, bs % kTile == 0 ? 2u : 1u};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    5, const_cast<void *>(cache), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// 4-D view of a prefill query [num_rows][Hq][D] for TMA: (element within a
// 64-element piece, piece, query head, row); one box = one piece of the
// `group` heads of a KV head for `tokens` consecutive rows, landing as
// (row, head)-ordered 128-byte rows, 128-byte swizzled.  Rows past num_rows
// read zeros.
int make_query_map(CUtensorMap *m, const void *query, pa_dtype_t dtype, int D, int Hq,
                   int num_rows, int group, int tokens) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PA_ERR_NO_DEVICE;
    const cuuint64_t e = 2;
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(Hq),
                          static_cast<cuuint64_t>(num_rows)};
    cuuint64_t strides[3] = {64 * e, D * e, static_cast<cuuint64_t>(Hq) * D * e};
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tokens)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    4, const_cast<void *>(query), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Shape {
    int S, Hq, Hkv, D, bs, num_blocks, max_blocks;
};

// Checks shared by the attention entry points.  Returns PA_OK, or 1 when
// there is nothing to do (num_seqs == 0), or a negative status.
int check_attention(const Shape &s, pa_dtype_t dtype, const void *query, const void *kc,
                    const void *vc, const int32_t *bt, const int32_t *sl) {
    if (s.S < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.D <= 0 || s.bs <= 0 || s.num_blocks < 0 ||
        s.max_blocks < 0)
        return PA_ERR_INVALID_ARGUMENT;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARGUMENT;
    if (s.Hq % s.Hkv != 0) return PA_ERR_INVALID_ARGUMENT;
    if (s.D != 64 && s.D != 128 && s.D != 256) return PA_ERR_UNSUPPORTED;
    if (s.bs % kTile != 0 && !(s.bs == 8 && PA_TILE_PIECES)) return PA_ERR_UNSUPPORTED;
    if (s.Hq / s.Hkv > kMaxGroup) return PA_ERR_UNSUPPORTED;
    if (s.S > 65535 || s.Hkv > 65535 || s.Hq > 65535) return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(s.max_blocks) * s.bs > INT_MAX) return PA_ERR_UNSUPPORTED;
    if (s.S == 0) return 1;
    if (!query || !kc || !vc || !bt || !sl) return PA_ERR_INVALID_ARGUMENT;
    if (s.num_blocks == 0 || s.max_blocks == 0) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(query, 16) || !aligned(kc, 16) || !aligned(vc, 16) || !aligned(bt, 4) ||
        !aligned(sl, 4))
        return PA_ERR_MISALIGNED;
    return PA_OK;
}

// CTAs per (sequence, KV head) of the single-pass grid: enough that the
// launch has about PA_SINGLE_CLUSTER_FACTOR times as many CTAs as can be
// resident, at most PA_SINGLE_CLUSTER_MAX (8, the portable cluster size).
#ifndef PA_SINGLE_CLUSTER_FACTOR
#define PA_SINGLE_CLUSTER_FACTOR 2
#endif
#ifndef PA_SINGLE_CLUSTER_MAX
#define PA_SINGLE_CLUSTER_MAX 8
#endif
int single_pass_cluster(int units, int resident_ctas) {
    if (units <= 0 || resident_ctas <= 0) return 1;
    const int64_t want = static_cast<int64_t>(PA_SINGLE_CLUSTER_FACTOR) * resident_ctas;
    const int64_t c = (want + units - 1) / units;
    return c < 1 ? 1 : (c > PA_SINGLE_CLUSTER_MAX ? PA_SINGLE_CLUSTER_MAX : static_cast<int>(c));
}

// Query heads one decode unit holds: 8 (one MMA n-tile), or 16 (two) when the
// GQA group is larger than 8 and head_dim is 64 or 128.  A group larger than
// that is split into ceil(group / heads) head groups, each its own unit
// (reading the same K/V, mostly from L2).
int unit_heads(int D, int group) { return group > kHeadsPad && D <= 128 ? kHeadsWide : kHeadsPad; }
int head_groups(int D, int group) {
    const int hp = unit_heads(D, group);
    return (group + hp - 1) / hp;
}

Params base_params(const Shape &s, const void *query, const int32_t *bt, const int32_t *sl,
                   float scale, int *status) {
    Params p{};
    p.q = query;
    p.block_tables = bt;
    p.seq_lens = sl;
    p.status = status;
    p.num_seqs = s.S;
    p.num_q_heads = s.Hq;
    p.num_kv_heads = s.Hkv;
    p.group = s.Hq / s.Hkv;
    p.block_size = s.bs;
    p.max_blocks = s.max_blocks;
    p.num_blocks = s.num_blocks;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.cluster = 1;
    p.hg_count = head_groups(s.D, p.group);
    return p;
}

cudaError_t attn(pa_dtype_t dt, int D, int mode, const CUtensorMap &tk, const CUtensorMap &tv,
                 const Params &p, dim3 grid, cudaStream_t st) {
    const int hp = unit_heads(D, p.group);
    return dt == PA_BF16 ? launch_attn<__nv_bfloat16>(D, mode, hp, tk, tv, p, grid, st)
                         : launch_attn<__half>(D, mode, hp, tk, tv, p, grid, st);
}

int ctas_per_sm(pa_dtype_t dt, int D, int mode, int group) {
    const int hp = unit_heads(D, group);
    return dt == PA_BF16 ? attn_ctas_per_sm<__nv_bfloat16>(D, mode, hp)
                         : attn_ctas_per_sm<__half>(D, mode, hp);
}

cudaError_t reduce(pa_dtype_t dt, int D, bool compact, const ReduceParams &r, dim3 grid,
                   cudaStream_t st) {
    return dt == PA_BF16 ? launch_reduce<__nv_bfloat16>(D, compact, r, grid, st)
                         : launch_reduce<__half>(D, compact, r, grid, st);
}

// Workspace layout of pa_decode_auto.  Work-list form: counters, the work
// list, per-sequence slot bases, the list of partitioned sequences, then the
// compact partials [slot][Hq] (stats) and [slot][Hq][D] (tmp_out).  Dense
// form (few sequences): the dense partials of pa_decode_partitioned.
struct AutoLayout {
    size_t counter, units, part_base, pseq_list, exp_sums, max_logits, tmp_out, total;
    int max_parts, max_slots, max_units;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Dense partials of pa_decode_partitioned in one buffer: tmp_out, exp_sums,
// max_logits, each region 256-byte aligned.
bool dense_layout(int S, int Hq, int D, int NP, AutoLayout *L) {
    if (S < 0 || Hq <= 0 || D <= 0 || NP <= 0) return false;
    const int64_t rows = static_cast<int64_t>(S) * Hq * NP;
    if (rows * D > (static_cast<int64_t>(1) << 40)) return false;
    L->max_parts = NP;
    L->max_slots = 0;
    L->max_units = 0;
    L->counter = L->units = L->part_base = L->pseq_list = 0;
    size_t off = 0;
    L->tmp_out = off;
    off = align256(off + static_cast<size_t>(rows) * D * sizeof(float));
    L->exp_sums = off;
    off = align256(off + static_cast<size_t>(rows) * sizeof(float));
    L->max_logits = off;
    off = align256(off + static_cast<size_t>(rows) * sizeof(float));
    L->total = off;
    return true;
}

// Work-list layout.  Partition slots: at most ceil(max_seq_len / P) per
// partitioned sequence, and, when the caller bounds the batch's total tokens
// T, at most floor((T + S_p (P - 1)) / P) in all, S_p <= min(S, T / (thr + 1))
// being the most sequences that can be longer than the threshold.
bool auto_layout(int S, int Hq, int Hkv, int D, int max_seq_len, long long max_total, int thr,
                 int P, AutoLayout *L) {
    if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_seq_len < 0 || P <= 0 || thr < 0)
        return false;
    const int64_t parts = max_seq_len > thr ? (static_cast<int64_t>(max_seq_len) + P - 1) / P : 0;
    int64_t slots = static_cast<int64_t>(S) * parts;
    if (max_total > 0 && parts > 0) {
        const int64_t sp = std::min<int64_t>(S, max_total / (static_cast<int64_t>(thr) + 1));
        slots = std::min<int64_t>(slots, (max_total + sp * (P - 1)) / P);
    }
    // units: (sequence or partition) x KV head x head group
    const int64_t units = (static_cast<int64_t>(S) + slots) * Hkv * head_groups(D, Hq / Hkv);
    if (slots * Hq > INT_MAX || units > INT_MAX) return false;
    L->max_parts = static_cast<int>(parts);
    L->max_slots = static_cast<int>(slots);
    L->max_units = static_cast<int>(units);
    size_t off = 0;
    L->counter = off;   // work-list cursor, unit count, partitioned-sequence count
    off = align256(off + 3 * sizeof(int));
    L->units = off;
    off = align256(off + static_cast<size_t>(units) * sizeof(int4));
    L->part_base = off;
    off = align256(off + static_cast<size_t>(S) * sizeof(int32_t));
    L->pseq_list = off;
    off = align256(off + static_cast<size_t>(S) * sizeof(int4));
    L->exp_sums = off;
    off = align256(off + static_cast<size_t>(slots) * Hq * sizeof(float));
    L->max_logits = off;
    off = align256(off + static_cast<size_t>(slots) * Hq * sizeof(float));
    L->tmp_out = off;
    off = align256(off + static_cast<size_t>(slots) * Hq * D * sizeof(float));
    L->total = off;
    return true;
}

// The single-pass threshold of the launch heuristic: the pages' 8192 when the
// batch has at least as many (sequence, KV head) units as SMs, else the
// partition size (too few units to fill the GPU: split everything longer than
// one partition).
int default_thr(int S, int Hkv, int P, int num_sms) {
    const int64_t units = static_cast<int64_t>(S) * Hkv;
    return units >= static_cast<int64_t>(num_sms) ? 8192 : P;
}

// Resident attention CTAs per SM of the partitioned grid (head_dim 64 and 128:
// 3, head_dim 256: 3; queried once from the occupancy calculator).
int partitioned_slots_per_sm(int D) {
    static std::atomic<int> cache[3];
    const int k = D == 64 ? 0 : (D == 128 ? 1 : 2);
    int v = cache[k].load(std::memory_order_relaxed);
    if (v == 0) {
        v = attn_ctas_per_sm<__nv_bfloat16>(D, kModePartitioned, kHeadsPad);
        if (v <= 0) v = 3;
        cache[k].store(v, std::memory_order_relaxed);
    }
    return v;
}

// The partition size of the launch heuristic: of 256, 512 and 1024 tokens
// (each rounded up to a multiple of the block size), the one that minimises
// waves x (P + 256): the partition units (sequence x KV head x partition) run
// in ceil(units / resident CTAs) waves, each as long as a partition plus a
// fixed cost worth ~256 tokens (a unit's set-up, its partials, its share of
// the reduce); ties go to the longer partition, which writes fewer partials.
// Fitted to the GB300 sweep over 1..256 sequences of 1K..64K tokens, where it
// picks the fastest size, or one within 1 % of it, at every point.
int default_partition(int S, int Hkv, int bs, int max_seq_len, int num_sms, int slots_per_sm) {
    const int64_t wave = static_cast<int64_t>(num_sms) * slots_per_sm;
    int best = 0;
    int64_t best_cost = 0;
    for (int cand : {1024, 512, 256}) {
        const int P = bs > 0 && cand % bs != 0 ? (cand + bs - 1) / bs * bs : cand;
        const int64_t units = static_cast<int64_t>(S) * Hkv * ((max_seq_len + P - 1) / P);
        const int64_t cost = (units + wave - 1) / wave * (P + 256);
        if (best == 0 || cost < best_cost) {
            best = P;
            best_cost = cost;
        }
    }
    return best;
}

// The launch form pa_decode_auto takes for a batch (host values only):
//   single   -- every sequence fits the single-pass limit: the single-pass grid;
//   dense    -- few (sequence, KV head) units and every sequence longer than one
//               partition is split: the partitioned grid of pa_decode_partitioned
//               with its partials in the workspace, then the dense reduce (two
//               launches, no planner);
//   worklist -- the planner's device work list (single-pass and partition units
//               in one attention launch), then the reduce over the partitioned
//               sequences.
struct AutoPlan {
    int thr, P, form;
    bool uniform;   // the host bounds say every sequence has about max_seq_len tokens
};

// A batch whose token bound T is at least 9/10 of S * max_seq_len has nearly
// equal lengths: one pass per (sequence, KV head) is then balanced by itself.
bool near_uniform(int S, int max_seq_len, long long max_total) {
    return max_total > 0 && S > 0 && max_seq_len > 0 &&
           10 * max_total >= 9 * static_cast<long long>(S) * max_seq_len;
}

int resolve_auto(int S, int Hkv, int D, int bs, int max_seq_len, long long max_total, int thr_in,
                 int P_in, int num_sms, AutoPlan *a) {
    if (S < 0 || Hkv <= 0 || bs <= 0 || max_seq_len < 0 || num_sms <= 0)
        return PA_ERR_INVALID_ARGUMENT;
    int P = P_in;
    if (P <= 0)
        P = default_partition(S, Hkv, bs, max_seq_len, num_sms,
                              D == 64 || D == 128 || D == 256 ? partitioned_slots_per_sm(D) : 3);
    if (P % bs != 0) return PA_ERR_UNSUPPORTED;
    const bool uniform = near_uniform(S, max_seq_len, max_total);
    int thr = thr_in;
    if (thr < 0) {
        thr = default_thr(S, Hkv, P, num_sms);
        // enough units and (nearly) equal lengths: the single pass is balanced
        // and writes no partials, at any length (measured on GB300 at 64 and
        // 256 sequences of 16K-64K tokens: 2-4 % faster than partitioning)
        if (uniform && static_cast<int64_t>(S) * Hkv >= num_sms && max_seq_len > thr)
            thr = max_seq_len;
    }
    int form = PA_AUTO_WORKLIST;
    if (max_seq_len <= thr)
        form = PA_AUTO_SINGLE_PASS;
    else if (thr <= P && static_cast<int64_t>(S) * Hkv < num_sms)
        form = PA_AUTO_DENSE;
    if (form == PA_AUTO_DENSE && thr_in < 0) {
        // A batch so small that the single-pass grid (each unit split over a
        // cluster of C CTAs, C as launch_single_pass picks it) fits one wave
        // with no CTA taking more tokens than a partition: one launch instead
        // of two (1 x 1024 tokens on GB300: 10.2 against 12.3 us).
        const int64_t units = static_cast<int64_t>(S) * Hkv;
        const int64_t resident = static_cast<int64_t>(num_sms) *
                                 (D == 64 || D == 128 || D == 256 ? partitioned_slots_per_sm(D) : 3);
        const int64_t C = units > 0 ? single_pass_cluster(static_cast<int>(units),
                                                          static_cast<int>(resident))
                                    : 1;
        if (units * C <= resident && (max_seq_len + C - 1) / C <= P) {
            thr = max_seq_len;
            form = PA_AUTO_SINGLE_PASS;
        }
    }
    a->thr = thr;
    a->P = P;
    a->form = form;
    a->uniform = uniform;
    return PA_OK;
}

bool plan_layout(int S, int Hq, int Hkv, int D, int max_seq_len, long long max_total,
                 const AutoPlan &a, AutoLayout *L) {
    if (a.form == PA_AUTO_DENSE)
        return dense_layout(S, Hq, D, static_cast<int>((static_cast<int64_t>(max_seq_len) + a.P - 1) /
                                                         a.P),
                            L);
    return auto_layout(S, Hq, Hkv, D, max_seq_len, max_total, a.thr, a.P, L);
}

int num_sms_now() {
    DevInfo *d = nullptr;
    if (device_info(&d) != PA_OK) return 0;
    return d->num_sms;
}


// The single-pass grid: each (sequence, KV head) split over a cluster of CTAs
// when the batch has too few units to keep every SM streaming (few or
// unequal sequences).  `uniform`: the caller's bounds say the lengths are
// nearly equal; with at least half a wave of units the units are then not
// split (a cluster's merge and the extra CTAs' set-up cost more than the
// balance they buy: 64 x 1024 tokens 28.7 against 38.9 us, 64 x 8192 158.8
// against 171.0 us on GB300).
int launch_single_pass(const Shape &s, void *out, const void *query, const int32_t *bt,
                       const int32_t *sl, float scale, pa_dtype_t dtype, const CUtensorMap &tk,
                       const CUtensorMap &tv, const DevInfo *di, cudaStream_t st,
                       bool uniform = false) {
    Params p = base_params(s, query, bt, sl, scale, di->status);
    p.out = out;
    const int per_sm = ctas_per_sm(dtype, s.D, kModeSingle, p.group);
    if (per_sm <= 0) return PA_ERR_CUDA;
    const int vheads = s.Hkv * p.hg_count;
    const int64_t units = static_cast<int64_t>(s.S) * vheads;
    const int64_t resident = static_cast<int64_t>(per_sm) * di->num_sms;
    p.cluster = uniform && 2 * units >= resident
                    ? 1
                    : single_pass_cluster(static_cast<int>(units), static_cast<int>(resident));
    const dim3 grid(p.cluster, vheads, s.S);
    return attn(dtype, s.D, kModeSingle, tk, tv, p, grid, st) == cudaSuccess ? PA_OK
                                                                             : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

int pa_version(void) { return kVersion; }

const char *pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARGUMENT: return "PA_ERR_INVALID_ARGUMENT";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_MISALIGNED: return "PA_ERR_MISALIGNED";
        case PA_ERR_WORKSPACE_TOO_SMALL: return "PA_ERR_WORKSPACE_TOO_SMALL";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
        case PA_ERR_NO_DEVICE: return "PA_ERR_NO_DEVICE";
        default: return "PA_ERR_UNKNOWN";
    }
}

int pa_decode(void *out, const void *query, const void *key_cache, const void *value_cache,
              const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
              int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
              int max_blocks_per_seq, float scale, pa_dtype_t dtype, void *stream) {
    const Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks_per_seq};
    int rc = check_attention(s, dtype, query, key_cache, value_cache, block_tables, seq_lens);
    if (rc != PA_OK) return rc > 0 ? PA_OK : rc;
    if (!out) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(out, 16)) return PA_ERR_MISALIGNED;
    DevInfo *di = nullptr;
    if ((rc = device_info(&di)) != PA_OK) return rc;
    CUtensorMap tk, tv;
    if ((rc = make_cache_map(&tk, key_cache, dtype, head_dim, num_kv_heads, block_size,
                             num_blocks)) != PA_OK)
        return rc;
    if ((rc = make_cache_map(&tv, value_cache, dtype, head_dim, num_kv_heads, block_size,
                             num_blocks)) != PA_OK)
        return rc;
    return launch_single_pass(s, out, query, block_tables, seq_lens, scale, dtype, tk, tv, di,
                              static_cast<cudaStream_t>(stream));
}

int pa_decode_partitioned(float *tmp_out, float *exp_sums, float *max_logits, const void *query,
                          const void *key_cache, const void *value_cache,
                          const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, int max_blocks_per_seq, float scale,
                          int partition_size, int max_num_partitions, pa_dtype_t dtype,
                          void *stream) {
    const Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks_per_seq};
    int rc = check_attention(s, dtype, query, key_cache, value_cache, block_tables, seq_lens);
    if (rc < 0) return rc;
    if (partition_size <= 0 || max_num_partitions <= 0) return PA_ERR_INVALID_ARGUMENT;
    if (partition_size % block_size != 0) return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(num_seqs) * num_q_heads * max_num_partitions * head_dim >
        (static_cast<int64_t>(1) << 40))
        return PA_ERR_INVALID_ARGUMENT;
    if (rc > 0) return PA_OK;
    if (!tmp_out || !exp_sums || !max_logits) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(tmp_out, 16) || !aligned(exp_sums, 4) || !aligned(max_logits, 4))
        return PA_ERR_MISALIGNED;
    DevInfo *di = nullptr;
    if ((rc = device_info(&di)) != PA_OK) return rc;
    CUtensorMap tk, tv;
    if ((rc = make_cache_map(&tk, key_cache, dtype, head_dim, num_kv_heads, block_size,
                             num_blocks)) != PA_OK)
        return rc;
    if ((rc = make_cache_map(&tv, value_cache, dtype, head_dim, num_kv_heads, block_size,
                             num_blocks)) != PA_OK)
        return rc;
    Params p = base_params(s, query, block_tables, seq_lens, scale, di->status);
    p.tmp_out = tmp_out;
    p.exp_sums = exp_sums;
    p.max_logits = max_logits;
    p.partition_size = partition_size;
    p.max_parts = max_num_partitions;
    const dim3 grid(max_num_partitions, num_kv_heads * p.hg_count, num_seqs);
    return attn(dtype, head_dim, kModePartitioned, tk, tv, p, grid,
                static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int pa_partition_reduce(void *out, const float *tmp_out, const float *exp_sums,
                        const float *max_logits, const int32_t *seq_lens, int num_seqs,
                        int num_q_heads, int head_dim, int partition_size,
                        int max_num_partitions, pa_dtype_t dtype, void *stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || partition_size <= 0 || max_num_partitions <= 0)
        return PA_ERR_INVALID_ARGUMENT;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARGUMENT;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_q_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !tmp_out || !exp_sums || !max_logits || !seq_lens) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(out, 16) || !aligned(tmp_out, 16) || !aligned(exp_sums, 4) ||
        !aligned(max_logits, 4) || !aligned(seq_lens, 4))
        return PA_ERR_MISALIGNED;
    DevInfo *di = nullptr;
    int rc = device_info(&di);
    if (rc != PA_OK) return rc;
    ReduceParams r{};
    r.out = out;
    r.tmp_out = tmp_out;
    r.exp_sums = exp_sums;
    r.max_logits = max_logits;
    r.seq_lens = seq_lens;
    r.status = di->status;
    r.num_q_heads = num_q_heads;
    r.partition_size = partition_size;
    r.max_parts = max_num_partitions;
    r.single_pass_max_len = -1;
    r.len_cap = INT_MAX;
    return reduce(dtype, head_dim, false, r, dim3(num_q_heads, num_seqs),
                  static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int pa_default_single_pass_max_len(int num_seqs, int num_kv_heads, int partition_size,
                                   int num_sms) {
    if (num_sms <= 0) num_sms = num_sms_now();
    if (num_sms <= 0) num_sms = 1;
    return default_thr(num_seqs, num_kv_heads, partition_size, num_sms);
}

int pa_default_partition_size(int num_seqs, int num_kv_heads, int block_size, int head_dim,
                              int max_seq_len, int num_sms) {
    if (num_seqs < 0 || num_kv_heads <= 0 || block_size <= 0 || max_seq_len < 0) return 0;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return 0;
    if (num_sms <= 0) num_sms = num_sms_now();
    if (num_sms <= 0) num_sms = 1;
    return default_partition(num_seqs, num_kv_heads, block_size, max_seq_len, num_sms,
                             partitioned_slots_per_sm(head_dim));
}

int pa_auto_resolve(int num_seqs, int num_kv_heads, int head_dim, int block_size,
                    int max_seq_len, long long max_total_tokens, int single_pass_max_len,
                    int partition_size, int num_sms, int *out_single_pass_max_len,
                    int *out_partition_size, int *out_form) {
    if (num_sms <= 0) num_sms = num_sms_now();
    if (num_sms <= 0) num_sms = 1;
    AutoPlan a;
    const int rc = resolve_auto(num_seqs, num_kv_heads, head_dim, block_size, max_seq_len,
                                max_total_tokens, single_pass_max_len, partition_size, num_sms,
                                &a);
    if (rc != PA_OK) return rc;
    if (out_single_pass_max_len) *out_single_pass_max_len = a.thr;
    if (out_partition_size) *out_partition_size = a.P;
    if (out_form) *out_form = a.form;
    return PA_OK;
}

size_t pa_partition_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                    int max_num_partitions) {
    AutoLayout L;
    if (!dense_layout(num_seqs, num_q_heads, head_dim, max_num_partitions, &L)) return 0;
    return L.total;
}

size_t pa_auto_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int max_seq_len, long long max_total_tokens,
                               int single_pass_max_len, int partition_size) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
    int num_sms = 0;
    if (single_pass_max_len < 0 || partition_size <= 0) num_sms = num_sms_now();
    if (num_sms <= 0) num_sms = 1;
    AutoPlan a;
    if (resolve_auto(num_seqs, num_kv_heads, head_dim, block_size, max_seq_len,
                     max_total_tokens, single_pass_max_len, partition_size, num_sms,
                     &a) != PA_OK)
        return 0;
    AutoLayout L;
    if (a.form == PA_AUTO_SINGLE_PASS) return 256;   // no scratch is used
    if (!plan_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                     max_total_tokens, a, &L))
        return 0;
    return L.total;
}

int pa_decode_auto_phases(void *out, const void *query, const void *key_cache,
                          const void *value_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          int max_blocks_per_seq, float scale, int max_seq_len,
                          long long max_total_tokens, int single_pass_max_len,
                          int partition_size, void *workspace, size_t workspace_bytes,
                          pa_dtype_t dtype, void *stream, int phases) {
    const Shape s{num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks_per_seq};
    int rc = check_attention(s, dtype, query, key_cache, value_cache, block_tables, seq_lens);
    if (rc < 0) return rc;
    if (max_seq_len < 0) return PA_ERR_INVALID_ARGUMENT;
    if (phases <= 0 || (phases & ~(PA_PHASE_PLAN | PA_PHASE_ATTEND | PA_PHASE_REDUCE)) != 0)
        return PA_ERR_INVALID_ARGUMENT;
    if (partition_size > 0 && partition_size % block_size != 0) return PA_ERR_UNSUPPORTED;
    if (rc > 0) return PA_OK;
    if (!out) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(out, 16)) return PA_ERR_MISALIGNED;
    // The heuristic reads the device's SM count; without a device the
    // arguments are still checked (as pa_auto_workspace_bytes sizes them)
    // before the missing device is reported.
    DevInfo *di = nullptr;
    const int dev_rc = device_info(&di);
    AutoPlan a;
    if ((rc = resolve_auto(num_seqs, num_kv_heads, head_dim, block_size, max_seq_len,
                           max_total_tokens, single_pass_max_len, partition_size,
                           dev_rc == PA_OK ? di->num_sms : 1, &a)) != PA_OK)
        return rc;
    AutoLayout L{};
    if (a.form != PA_AUTO_SINGLE_PASS) {
        if (!plan_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                         max_total_tokens, a, &L))
            return PA_ERR_INVALID_ARGUMENT;
        if (!workspace) return PA_ERR_INVALID_ARGUMENT;
        if (!aligned(workspace, 256)) return PA_ERR_MISALIGNED;
        if (workspace_bytes < L.total) return PA_ERR_WORKSPACE_TOO_SMALL;
    }
    if (dev_rc != PA_OK) return dev_rc;
    CUtensorMap tk, tv;
    if ((rc = make_cache_map(&tk, key_cache, dtype, head_dim, num_kv_heads, block_size,
                             num_blocks)) != PA_OK)
        return rc;
    if ((rc = make_cache_map(&tv, value_cache, dtype, head_dim, num_kv_heads, block_size,
                             num_blocks)) != PA_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (a.form == PA_AUTO_SINGLE_PASS) {
        // Every sequence fits the single-pass limit: no work list and no
        // partials, just the single-pass grid (the plan and reduce phases have
        // nothing to do).
        if (!(phases & PA_PHASE_ATTEND)) return PA_OK;
        return launch_single_pass(s, out, query, block_tables, seq_lens, scale, dtype, tk, tv,
                                  di, st, a.uniform);
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *es = reinterpret_cast<float *>(ws + L.exp_sums);
    float *ml = reinterpret_cast<float *>(ws + L.max_logits);
    float *tmp = reinterpret_cast<float *>(ws + L.tmp_out);
    const int len_cap = max_blocks_per_seq * block_size;

    if (a.form == PA_AUTO_DENSE) {
        // Few sequences, each split at P: the partitioned grid and the dense
        // reduce, as pa_decode_partitioned + pa_partition_reduce (no planner).
        if (phases & PA_PHASE_ATTEND) {
            Params p = base_params(s, query, block_tables, seq_lens, scale, di->status);
            p.tmp_out = tmp;
            p.exp_sums = es;
            p.max_logits = ml;
            p.partition_size = a.P;
            p.max_parts = L.max_parts;
            if (attn(dtype, head_dim, kModePartitioned, tk, tv, p,
                     dim3(L.max_parts, num_kv_heads * p.hg_count, num_seqs), st) != cudaSuccess)
                return PA_ERR_CUDA;
        }
        if (phases & PA_PHASE_REDUCE) {
            ReduceParams r{};
            r.out = out;
            r.tmp_out = tmp;
            r.exp_sums = es;
            r.max_logits = ml;
            r.seq_lens = seq_lens;
            r.status = di->status;
            r.num_q_heads = num_q_heads;
            r.partition_size = a.P;
            r.max_parts = L.max_parts;
            r.single_pass_max_len = -1;
            r.len_cap = len_cap;
            if (reduce(dtype, head_dim, false, r, dim3(num_q_heads, num_seqs), st) !=
                cudaSuccess)
                return PA_ERR_CUDA;
        }
        return PA_OK;
    }

    int *counter = reinterpret_cast<int *>(ws + L.counter);
    int4 *units = reinterpret_cast<int4 *>(ws + L.units);
    int32_t *part_base = reinterpret_cast<int32_t *>(ws + L.part_base);
    int4 *pseq_list = reinterpret_cast<int4 *>(ws + L.pseq_list);

    PlanParams pp{};
    pp.seq_lens = seq_lens;
    pp.units = units;
    pp.unit_counter = counter;
    pp.unit_count = counter + 1;
    pp.part_base = part_base;
    pp.pseq_list = pseq_list;
    pp.pseq_count = counter + 2;
    pp.status = di->status;
    pp.num_seqs = num_seqs;
    pp.num_kv_heads = num_kv_heads * head_groups(head_dim, num_q_heads / num_kv_heads);
    pp.partition_size = a.P;
    pp.single_pass_max_len = a.thr;
    pp.len_cap = len_cap;
    pp.max_parts = L.max_parts;
    pp.max_slots = L.max_slots;
    if ((phases & PA_PHASE_PLAN) && launch_plan(pp, st) != cudaSuccess) return PA_ERR_CUDA;

    Params p = base_params(s, query, block_tables, seq_lens, scale, di->status);
    p.out = out;
    p.tmp_out = tmp;
    p.exp_sums = es;
    p.max_logits = ml;
    p.units = units;
    p.unit_counter = counter;
    p.unit_count = counter + 1;
    p.part_base = part_base;
    p.partition_size = a.P;
    p.max_parts = L.max_parts;
    p.single_pass_max_len = a.thr;
    const int per_sm = ctas_per_sm(dtype, head_dim, kModeWorklist, p.group);
    if (per_sm <= 0) return PA_ERR_CUDA;
    int64_t ctas = static_cast<int64_t>(per_sm) * di->num_sms;
    if (ctas > L.max_units) ctas = L.max_units;
    if (ctas < 1) ctas = 1;
    if ((phases & PA_PHASE_ATTEND) &&
        attn(dtype, head_dim, kModeWorklist, tk, tv, p, dim3(static_cast<unsigned>(ctas)), st) !=
            cudaSuccess)
        return PA_ERR_CUDA;

    if ((phases & PA_PHASE_REDUCE) && L.max_parts > 0) {
        ReduceParams r{};
        r.out = out;
        r.tmp_out = tmp;
        r.exp_sums = es;
        r.max_logits = ml;
        r.seq_lens = seq_lens;
        r.part_base = part_base;
        r.pseq_list = pseq_list;
        r.pseq_count = counter + 2;
        r.status = di->status;
        r.num_q_heads = num_q_heads;
        r.partition_size = a.P;
        r.max_parts = L.max_parts;
        r.single_pass_max_len = a.thr;
        r.len_cap = len_cap;
        // one CTA per (partitioned sequence, head): rows past the planner's
        // count exit at once
        const int rows = num_seqs;
        if (reduce(dtype, head_dim, true, r, dim3(num_q_heads, rows), st) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_decode_auto(void *out, const void *query, const void *key_cache, const void *value_cache,
                   const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                   int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                   int num_blocks, int max_blocks_per_seq, float scale, int max_seq_len,
                   long long max_total_tokens, int single_pass_max_len, int partition_size,
                   void *workspace, size_t workspace_bytes, pa_dtype_t dtype, void *stream) {
    return pa_decode_auto_phases(out, query, key_cache, value_cache, block_tables, seq_lens,
                                 num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 num_blocks, max_blocks_per_seq, scale, max_seq_len,
                                 max_total_tokens, single_pass_max_len, partition_size, workspace,
                                 workspace_bytes, dtype, stream,
                                 PA_PHASE_PLAN | PA_PHASE_ATTEND | PA_PHASE_REDUCE);
}

int pa_gather_kv(void *k_dense, void *v_dense, const void *key_cache, const void *value_cache,
                 const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                 int max_blocks_per_seq, int max_len, pa_dtype_t dtype, void *stream) {
    const Shape s{num_seqs, num_kv_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks_per_seq};
    int rc = check_attention(s, dtype, key_cache, key_cache, value_cache, block_tables, seq_lens);
    if (rc < 0) return rc;
    if (max_len < 0) return PA_ERR_INVALID_ARGUMENT;
    if (rc > 0 || max_len == 0) return PA_OK;
    if (!k_dense || !v_dense) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(k_dense, 16) || !aligned(v_dense, 16)) return PA_ERR_MISALIGNED;
    DevInfo *di = nullptr;
    if ((rc = device_info(&di)) != PA_OK) return rc;
    CUtensorMap tk, tv;
    if ((rc = make_cache_map(&tk, key_cache, dtype, head_dim, num_kv_heads, block_size,
                             num_blocks)) != PA_OK)
        return rc;
    if ((rc = make_cache_map(&tv, value_cache, dtype, head_dim, num_kv_heads, block_size,
                             num_blocks)) != PA_OK)
        return rc;
    GatherParams gp{};
    gp.k_dense = k_dense;
    gp.v_dense = v_dense;
    gp.block_tables = block_tables;
    gp.seq_lens = seq_lens;
    gp.status = di->status;
    gp.num_kv_heads = num_kv_heads;
    gp.block_size = block_size;
    gp.max_blocks = max_blocks_per_seq;
    gp.num_blocks = num_blocks;
    gp.max_len = max_len;
    const dim3 grid((max_len + kTile - 1) / kTile, num_kv_heads, num_seqs);
    return launch_gather(head_dim, tk, tv, gp, grid, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int pa_prefill(void *out, const void *query, const void *key_cache, const void *value_cache,
               const int32_t *block_tables, const int32_t *seq_lens, const int32_t *q_start,
               int num_seqs, int num_rows, int max_q_len, int num_q_heads, int num_kv_heads,
               int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
               float scale, pa_dtype_t dtype, void *stream) {
    if (num_seqs < 0 || num_rows < 0 || max_q_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks < 0 || max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARGUMENT;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARGUMENT;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARGUMENT;
    const int group = num_q_heads / num_kv_heads;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (block_size % kTile != 0 && block_size != kTile / 2) return PA_ERR_UNSUPPORTED;
    if (group > kPrefillRows) return PA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT_MAX) return PA_ERR_UNSUPPORTED;
    // the 8-token group coordinate of the cache views is a 32-bit int
    if (static_cast<int64_t>(num_blocks) * (block_size / 8) > INT_MAX) return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(num_rows) * num_q_heads * head_dim > (static_cast<int64_t>(1) << 40))
        return PA_ERR_INVALID_ARGUMENT;
    if (num_seqs == 0 || num_rows == 0 || max_q_len == 0) return PA_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !seq_lens || !q_start)
        return PA_ERR_INVALID_ARGUMENT;
    if (num_blocks == 0 || max_blocks_per_seq == 0) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(out, 16) || !aligned(query, 16) || !aligned(key_cache, 16) ||
        !aligned(value_cache, 16) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
        !aligned(q_start, 4))
        return PA_ERR_MISALIGNED;
    DevInfo *di = nullptr;
    int rc = device_info(&di);
    if (rc != PA_OK) return rc;
    // K and V move one 16-token box per copy (every piece of it a CTA holds)
    CUtensorMap tk, tv;
    if ((rc = make_cache_map_groups(&tk, key_cache, dtype, head_dim, num_kv_heads, block_size,
                                    num_blocks, head_dim / 64)) != PA_OK)
        return rc;
    if ((rc = make_cache_map_groups(&tv, value_cache, dtype, head_dim, num_kv_heads, block_size,
                                    num_blocks, prefill_v_box_pieces(head_dim))) != PA_OK)
        return rc;
    PrefillParams p{};
    p.q = query;
    p.out = out;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.q_start = q_start;
    p.status = di->status;
    p.num_seqs = num_seqs;
    p.num_rows = num_rows;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.block_size = block_size;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.tokens_per_cta = prefill_rows_per_cta(head_dim) / group;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    const dim3 grid((max_q_len + p.tokens_per_cta - 1) / p.tokens_per_cta, num_kv_heads,
                    num_seqs);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap tq;
    if ((rc = make_query_map(&tq, query, dtype, head_dim, num_q_heads, num_rows, group,
                             p.tokens_per_cta)) != PA_OK)
        return rc;
    const cudaError_t e =
        dtype == PA_BF16 ? launch_prefill_tc<__nv_bfloat16>(head_dim, tq, tk, tv, p, grid, st)
                         : launch_prefill_tc<__half>(head_dim, tq, tk, tv, p, grid, st);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_topk_softmax(float *topk_weights, int32_t *topk_ids, const void *gating_logits,
                    int num_tokens, int num_experts, int topk, int renormalize,
                    pa_logits_t logits_dtype, void *stream) {
    if (num_tokens < 0 || topk <= 0) return PA_ERR_INVALID_ARGUMENT;
    if (logits_dtype != PA_LOGITS_F16 && logits_dtype != PA_LOGITS_BF16 &&
        logits_dtype != PA_LOGITS_F32)
        return PA_ERR_INVALID_ARGUMENT;
    if (num_experts != 32 && num_experts != 64 && num_experts != 128 && num_experts != 256 &&
        num_experts != 512)
        return PA_ERR_UNSUPPORTED;
    if (topk > 32 || topk > num_experts) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!topk_weights || !topk_ids || !gating_logits) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(gating_logits, 16) || !aligned(topk_weights, 4) || !aligned(topk_ids, 4))
        return PA_ERR_MISALIGNED;
    DevInfo *di = nullptr;
    const int rc = device_info(&di);
    if (rc != PA_OK) return rc;
    TopkParams p{};
    p.logits = gating_logits;
    p.weights = topk_weights;
    p.ids = topk_ids;
    p.num_tokens = num_tokens;
    p.topk = topk;
    p.renormalize = renormalize != 0;
    return launch_topk_softmax(static_cast<int>(logits_dtype), num_experts, p,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

size_t pa_moe_sort_workspace_bytes(int num_pairs, int num_experts) {
    if (num_pairs < 0 || num_experts <= 0 || num_experts > 1024) return 0;
    return align256(static_cast<size_t>(moe_sort_chunks(num_pairs)) * num_experts *
                    sizeof(int32_t)) + 256;
}

int pa_moe_sort(int32_t *sorted_pairs, int32_t *expert_offsets, int32_t *pair_pos,
                const int32_t *expert_ids, int num_pairs, int num_experts, void *workspace,
                size_t workspace_bytes, void *stream) {
    if (num_pairs < 0 || num_experts <= 0) return PA_ERR_INVALID_ARGUMENT;
    if (num_experts > 1024) return PA_ERR_UNSUPPORTED;
    if (!expert_offsets) return PA_ERR_INVALID_ARGUMENT;
    if (num_pairs > 0 && (!sorted_pairs || !pair_pos || !expert_ids))
        return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(sorted_pairs, 4) || !aligned(expert_offsets, 4) || !aligned(pair_pos, 4) ||
        !aligned(expert_ids, 4))
        return PA_ERR_MISALIGNED;
    if (!workspace) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(workspace, 256)) return PA_ERR_MISALIGNED;
    if (workspace_bytes < pa_moe_sort_workspace_bytes(num_pairs, num_experts))
        return PA_ERR_WORKSPACE_TOO_SMALL;
    DevInfo *di = nullptr;
    const int rc = device_info(&di);
    if (rc != PA_OK) return rc;
    SortParams p{};
    p.expert_ids = expert_ids;
    p.sorted_pairs = sorted_pairs;
    p.offsets = expert_offsets;
    p.pair_pos = pair_pos;
    p.hist = static_cast<int32_t *>(workspace);
    p.status = di->status;
    p.num_pairs = num_pairs;
    p.num_experts = num_experts;
    p.num_chunks = moe_sort_chunks(num_pairs);
    if (num_pairs == 0) {   // offsets are all zero: the scan alone writes them
        p.num_chunks = 0;
    }
    return launch_moe_sort(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                : PA_ERR_CUDA;
}

int pa_moe_gather(void *sorted_hidden, const void *hidden, const int32_t *pair_pos,
                  int num_tokens, int topk, int num_rows, int hidden_size, pa_dtype_t dtype,
                  void *stream) {
    if (num_tokens < 0 || topk <= 0 || num_rows < 0 || hidden_size <= 0)
        return PA_ERR_INVALID_ARGUMENT;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARGUMENT;
    if ((hidden_size * 2) % 16 != 0 || topk > 32) return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(num_tokens) * topk > INT_MAX) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!sorted_hidden || !hidden || !pair_pos) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(sorted_hidden, 16) || !aligned(hidden, 16) || !aligned(pair_pos, 4))
        return PA_ERR_MISALIGNED;
    DevInfo *di = nullptr;
    const int rc = device_info(&di);
    if (rc != PA_OK) return rc;
    MoeGatherParams p{};
    p.out = sorted_hidden;
    p.hidden = hidden;
    p.pair_pos = pair_pos;
    p.status = di->status;
    p.num_rows = num_rows;
    p.topk = topk;
    p.num_tokens = num_tokens;
    p.row_bytes = hidden_size * 2;
    return launch_moe_gather(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                  : PA_ERR_CUDA;
}

int pa_moe_scatter_back(void *out, const void *expert_out, const int32_t *pair_pos,
                        const float *topk_weights, int num_tokens, int topk, int hidden_size,
                        pa_dtype_t dtype, void *stream) {
    if (num_tokens < 0 || topk <= 0 || hidden_size <= 0) return PA_ERR_INVALID_ARGUMENT;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARGUMENT;
    if (topk > 32 || hidden_size % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(num_tokens) * topk > INT_MAX) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!out || !expert_out || !pair_pos || !topk_weights) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(out, 16) || !aligned(expert_out, 16) || !aligned(pair_pos, 4) ||
        !aligned(topk_weights, 4))
        return PA_ERR_MISALIGNED;
    DevInfo *di = nullptr;
    const int rc = device_info(&di);
    if (rc != PA_OK) return rc;
    MoeScatterParams p{};
    p.out = out;
    p.y = expert_out;
    p.pair_pos = pair_pos;
    p.weights = topk_weights;
    p.status = di->status;
    p.num_tokens = num_tokens;
    p.topk = topk;
    p.num_pairs = num_tokens * topk;
    p.hidden_size = hidden_size;
    return launch_moe_scatter(dtype == PA_BF16, p, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int pa_selftest_wait_timeout(void *stream, int limit_us) {
    if (limit_us <= 0 || limit_us > 1000000) return PA_ERR_INVALID_ARGUMENT;
    DevInfo *di = nullptr;
    const int rc = device_info(&di);
    if (rc != PA_OK) return rc;
    return launch_wait_timeout_test(di->status, 1000ull * static_cast<unsigned>(limit_us),
                                    static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int pa_device_status(void *stream, int *flags) {
    if (!flags) return PA_ERR_INVALID_ARGUMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_pa_status_word, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                  st) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_pa_status_word, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                st) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
    *flags = v;
    return PA_OK;
}

}  // extern "C"
