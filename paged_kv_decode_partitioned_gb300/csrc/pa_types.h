// pa_types.h -- constants and launch-parameter structs shared by the host
// API and the device code of the paged-attention decode library.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace pa {

constexpr int kTile = 16;       // tokens per pipeline tile (the MMA M of S^T)
constexpr int kHeadsPad = 8;    // query heads of one MMA n-tile (the MMA N)
constexpr int kHeadsWide = 16;  // query heads a decode unit holds in registers at most
constexpr int kMaxGroup = 128;  // largest GQA group the decode kernels take (head groups)
constexpr int kPrefillRows = 128;   // largest GQA group the prefill kernel takes
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimitNs = 500ull * 1000ull * 1000ull;  // 0.5 s

// Flags of the device status word (mirrors PA_DEV_* in pa_decode.h).
enum : int {
    kBadBlock = 1, kLenClamped = 2, kWaitTimeout = 4, kTooManyParts = 8, kBadRows = 16,
    kBadExpert = 32
};

// Unit kinds.
enum : int { kOutFinal = 0, kOutPartialDense = 1, kOutPartialCompact = 2 };

// Grid modes of the attention kernel.
enum : int { kModeSingle = 0, kModePartitioned = 1, kModeWorklist = 2 };

struct Params {
    const void *q;              // [S][Hq][D]
    void *out;                  // [S][Hq][D]
    float *tmp_out;             // dense [S][Hq][max_parts][D] or compact [slot][Hq][D]
    float *exp_sums;            // dense [S][Hq][max_parts]    or compact [slot][Hq]
    float *max_logits;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    const int4 *units;          // work list (seq, kvh, part, kind)
    int *unit_counter;          // dynamic work-list cursor
    const int *unit_count;
    const int32_t *part_base;   // compact slot of partition 0 of each sequence, -1 if none
    int *status;
    int num_seqs, num_q_heads, num_kv_heads, group, block_size, max_blocks, num_blocks;
    int partition_size, max_parts, single_pass_max_len;
    int cluster;                // CTAs per unit of the single-pass grid (1..8)
    int hg_count;               // head groups per KV head: a unit's "KV head" index v is
                                // (KV head v / hg_count, head group v % hg_count)
    float scale_log2;           // scale * log2(e)
};

struct ReduceParams {
    void *out;
    const float *tmp_out;
    const float *exp_sums;
    const float *max_logits;
    const int32_t *seq_lens;
    const int32_t *part_base;   // compact layout only
    const int4 *pseq_list;      // compact layout: (sequence, first slot, partitions, -)
    const int *pseq_count;      // compact layout: number of entries
    int *status;
    int num_q_heads, partition_size, max_parts, single_pass_max_len, len_cap;
};

struct PlanParams {
    const int32_t *seq_lens;
    int4 *units;
    int *unit_counter;
    int *unit_count;
    int32_t *part_base;
    int4 *pseq_list;            // (sequence, first slot, partitions, 0) per partitioned sequence
    int *pseq_count;
    int *status;
    int num_seqs, num_kv_heads, partition_size, single_pass_max_len, len_cap, max_parts;
    int max_slots;              // partition slots the workspace holds
    int chunk;                  // sequences per planner CTA (set by the launcher)
};

struct PrefillParams {
    const void *q;              // [num_rows][Hq][D]
    void *out;                  // [num_rows][Hq][D]
    const int32_t *block_tables;
    const int32_t *seq_lens;    // cached tokens per sequence, the chunk included
    const int32_t *q_start;     // [S + 1] first chunk row of each sequence
    int *status;
    int num_seqs, num_rows, num_q_heads, num_kv_heads, group, block_size, max_blocks, num_blocks;
    int tokens_per_cta;         // chunk tokens per CTA (query rows per CTA / group)
    float scale_log2;           // scale * log2(e)
};

struct GatherParams {
    void *k_dense;
    void *v_dense;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    int *status;
    int num_kv_heads, block_size, max_blocks, num_blocks, max_len;
};

struct TopkParams {
    const void *logits;         // [T][E] f16 / bf16 / f32
    float *weights;             // [T][k]
    int32_t *ids;               // [T][k]
    int num_tokens, topk, renormalize;
};

struct SortParams {
    const int32_t *expert_ids;  // [P] (the router's ids, flattened)
    int32_t *sorted_pairs;      // [P]
    int32_t *offsets;           // [E + 1]
    int32_t *pair_pos;          // [P]
    int32_t *hist;              // workspace [num_chunks][E]
    int *status;
    int num_pairs, num_experts, num_chunks;
};

struct MoeGatherParams {
    void *out;                  // [num_rows][row_bytes]
    const void *hidden;         // [T][row_bytes]
    const int32_t *pair_pos;    // [T * topk] sorted position of each pair, -1: not placed
    int *status;
    int num_rows, topk, num_tokens, row_bytes;
};

struct MoeScatterParams {
    void *out;                  // [T][H]
    const void *y;              // [P][H], sorted order
    const int32_t *pair_pos;    // [P]
    const float *weights;       // [T][K]
    int *status;
    int num_tokens, topk, num_pairs, hidden_size;
};

}  // namespace pa
