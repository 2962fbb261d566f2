/*
 * pa_decode.h -- C ABI of the GB300 (sm_103a) paged-attention decode library
 * (libpadecode.so).
 *
 * The operation (page: project_6 commit cd0d9e1, "qwen3_6_scripts"):
 *   One query token per sequence attends over that sequence's keys and
 *   values, which live in a block-paged cache: logical block j of sequence s
 *   is the physical block block_tables[s][j] (the prefix-prefill rewrite's
 *   pre-gather of context K/V through the block table).  The result is
 *       out[s][h] = sum_t softmax_t(scale * q[s][h] . k_t) * v_t,
 *   t over the sequence's seq_lens[s] tokens.  The forward_decode heuristic
 *   runs short sequences in one pass (V1) and splits long ones into
 *   partition_size-token partitions (V2): phase 1 keeps a partial output, its
 *   maximum logit and its exp-sum per partition, and phase 2 merges the
 *   partitions with a log-sum-exp rescale.
 *
 * Conventions shared by every entry point:
 *   - All array pointers are DEVICE pointers, owned by the caller, dense and
 *     row-major in the layouts given below.  The library allocates no device
 *     memory and keeps no pointer after a call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and run on the current CUDA device.  Every argument is
 *     checked on the host before anything is launched; a call that returns an
 *     error has launched nothing (except PA_ERR_CUDA, which reports a failed
 *     launch).
 *   - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - dtype selects IEEE binary16 (PA_F16) or bfloat16 (PA_BF16) for query,
 *     caches and out.  Accumulation is fp32.  Partials are fp32.
 *   - Supported shapes (decode entry points): head_dim in {64, 128, 256};
 *     block_size 8 or a multiple of 16; GQA group num_q_heads / num_kv_heads
 *     between 1 and 128.  A group of up to 16 heads (8 at head_dim 256) is
 *     served by one unit per KV head, which reads each K/V page once; a larger
 *     group is split into head groups of 16 (8) that each read the KV head's
 *     pages.  Other shapes return PA_ERR_UNSUPPORTED.
 *   - Alignment: caches, query, out and partial buffers 16-byte aligned
 *     (PA_ERR_MISALIGNED otherwise).
 *   - block_tables contents and seq_lens values are read on the device only.
 *     A table entry outside [0, num_blocks) reads zeros (never memory outside
 *     the cache) and a length above max_blocks_per_seq * block_size is
 *     clamped; both raise a flag that pa_device_status() reports.
 *
 * Layouts:
 *   query        [num_seqs][num_q_heads][head_dim]
 *   key_cache    [num_blocks][block_size][num_kv_heads][head_dim]
 *   value_cache  [num_blocks][block_size][num_kv_heads][head_dim]
 *   block_tables int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens     int32 [num_seqs]
 *   out          [num_seqs][num_q_heads][head_dim]
 *   tmp_out      fp32 [num_seqs][num_q_heads][max_num_partitions][head_dim]
 *   exp_sums, max_logits  fp32 [num_seqs][num_q_heads][max_num_partitions]
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype_t;

/* Status codes returned by every int-valued entry point. */
enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARGUMENT = -1,   /* null pointer, negative or inconsistent size */
    PA_ERR_UNSUPPORTED = -2,        /* head_dim / block_size / GQA group not supported */
    PA_ERR_MISALIGNED = -3,         /* a pointer is not 16-byte aligned */
    PA_ERR_WORKSPACE_TOO_SMALL = -4,/* workspace_bytes below what the call needs */
    PA_ERR_CUDA = -5,               /* a CUDA runtime / driver call or launch failed */
    PA_ERR_DEVICE = -6,             /* pa_device_status: the device raised a flag */
    PA_ERR_NO_DEVICE = -7           /* no usable CUDA device / TMA entry point */
};

/* Flags that kernels raise in the device status word (pa_device_status). */
enum {
    PA_DEV_BAD_BLOCK = 1,           /* a block-table entry outside [0, num_blocks) */
    PA_DEV_LEN_CLAMPED = 2,         /* seq_len > max_blocks_per_seq*block_size or < 0 */
    PA_DEV_WAIT_TIMEOUT = 4,        /* a pipeline wait gave up; that output is not written */
    PA_DEV_TOO_MANY_PARTITIONS = 8, /* ceil(seq_len/partition_size) > max_num_partitions */
    PA_DEV_BAD_ROWS = 16            /* pa_prefill: q_start rows outside [0, num_rows] or
                                       a chunk longer than its sequence (skipped) */
};

/*
 * pa_decode -- single-pass decode (V1: the whole KV range of a sequence in
 * one launch, no partial results in global memory).
 *   out[s][h][:] = softmax(scale * q[s][h] . k_t) weighted sum of v_t over
 *   t < seq_lens[s]; a sequence with seq_len 0 gets zeros.
 * scale: the logit scale (usually 1/sqrt(head_dim)).
 */
PA_API int pa_decode(void *out, const void *query, const void *key_cache,
              const void *value_cache, const int32_t *block_tables,
              const int32_t *seq_lens, int num_seqs, int num_q_heads,
              int num_kv_heads, int head_dim, int block_size, int num_blocks,
              int max_blocks_per_seq, float scale, pa_dtype_t dtype, void *stream);

/*
 * pa_decode_partitioned -- phase 1 of the split-KV decode (V2 description,
 * phase 1; the page's partition size is 512).
 * For partition p < ceil(seq_lens[s] / partition_size) covering tokens
 * [p*P, min((p+1)*P, L)) and every query head h:
 *   max_logits[s][h][p] = m_p = max_t scale * q.k_t
 *   exp_sums[s][h][p]   = l_p = sum_t exp(scale * q.k_t - m_p)
 *   tmp_out[s][h][p][:] = sum_t exp(scale * q.k_t - m_p) v_t / l_p
 * Slots p >= ceil(L/P) are not written.  partition_size must be a positive
 * multiple of block_size; max_num_partitions >= ceil(max seq_len / P) (a
 * sequence with more partitions raises PA_DEV_TOO_MANY_PARTITIONS and has
 * only its first max_num_partitions written).
 */
PA_API int pa_decode_partitioned(float *tmp_out, float *exp_sums, float *max_logits,
                          const void *query, const void *key_cache,
                          const void *value_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, int max_blocks_per_seq, float scale,
                          int partition_size, int max_num_partitions,
                          pa_dtype_t dtype, void *stream);

/*
 * pa_partition_reduce -- phase 2 of the split-KV decode (V2 description,
 * phase 2: the log-sum-exp merge across partitions).  With n = ceil(seq_lens[s] / partition_size):
 *   M = max_p m_p,  w_p = exp(m_p - M) * l_p,
 *   out[s][h][:] = sum_{p<n} w_p * tmp_out[s][h][p][:] / sum_{p<n} w_p
 * rounded to dtype; n = 0 gives zeros.  Reads only slots p < n.
 */
PA_API int pa_partition_reduce(void *out, const float *tmp_out, const float *exp_sums,
                        const float *max_logits, const int32_t *seq_lens,
                        int num_seqs, int num_q_heads, int head_dim,
                        int partition_size, int max_num_partitions,
                        pa_dtype_t dtype, void *stream);

/*
 * pa_partition_workspace_bytes -- bytes of the phase-1 partials of
 * pa_decode_partitioned (V2 description, phase 1: a partial output, its
 * exp-sum and its maximum logit kept per partition) for num_seqs sequences,
 * num_q_heads query heads, head_dim and max_num_partitions slots, laid out in
 * one buffer as three 256-byte-aligned regions in this order:
 *   tmp_out    fp32 [num_seqs][num_q_heads][max_num_partitions][head_dim]
 *   exp_sums   fp32 [num_seqs][num_q_heads][max_num_partitions]
 *   max_logits fp32 [num_seqs][num_q_heads][max_num_partitions]
 * Region i starts at the end of region i-1 rounded up to 256 bytes.  Returns
 * 0 on bad arguments (a negative or zero size, or more than 2^40 elements).
 */
PA_API size_t pa_partition_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                           int max_num_partitions);

/*
 * pa_default_single_pass_max_len -- the launch heuristic's threshold.
 * Sequences longer than the returned length are partitioned by
 * pa_decode_auto.  It is 8192, the forward_decode heuristic's boundary
 * between V1 and V2, when there are at least as many num_seqs * num_kv_heads
 * single-pass units as SMs (the single-pass grid then splits each unit over a
 * cluster to fill the device), and partition_size otherwise (too few units:
 * split everything longer than one partition).  The crossover was measured
 * on GB300 over 1..256 sequences of 1K..64K tokens.  num_sms <= 0 queries
 * the current device.
 */
PA_API int pa_default_single_pass_max_len(int num_seqs, int num_kv_heads, int partition_size,
                                   int num_sms);

/*
 * pa_default_partition_size -- the launch heuristic's partition size (the
 * pages use 512 in one file and 256 in another).  Of 256, 512 and 1024
 * tokens (each rounded up to a multiple of block_size), returns the P that
 * minimises ceil(U_P / W) * (P + 256), where U_P = num_seqs * num_kv_heads *
 * ceil(max_seq_len / P) partition units run in waves of W = num_sms x resident
 * attention CTAs per SM, and 256 tokens stand for a unit's fixed cost; ties go
 * to the larger P (fewer partials).  Fitted to a GB300 sweep over 1..256
 * sequences of 1K..64K tokens.  num_sms <= 0 queries the current device.
 * Returns 0 on bad arguments.
 */
PA_API int pa_default_partition_size(int num_seqs, int num_kv_heads, int block_size,
                                     int head_dim, int max_seq_len, int num_sms);

/* Launch forms of pa_decode_auto (pa_auto_resolve). */
enum {
    PA_AUTO_SINGLE_PASS = 0,   /* max_seq_len <= threshold: the pa_decode grid, one launch */
    PA_AUTO_DENSE = 1,         /* few sequences, all split: pa_decode_partitioned's grid and
                                  pa_partition_reduce, partials in the workspace; two launches */
    PA_AUTO_WORKLIST = 2       /* planner + work-list attention + reduce; three launches */
};

/*
 * pa_auto_resolve -- what pa_decode_auto does for these host values, without
 * launching anything: the single-pass threshold (single_pass_max_len < 0
 * selects pa_default_single_pass_max_len, raised to max_seq_len when the
 * batch has at least one (sequence, KV head) unit per SM and the caller's
 * token bound max_total_tokens is at least 9/10 of num_seqs * max_seq_len:
 * nearly equal lengths, which one pass balances without partials), the
 * partition size (partition_size <= 0 selects pa_default_partition_size) and
 * the launch form:
 *   PA_AUTO_SINGLE_PASS when max_seq_len <= threshold;
 *   PA_AUTO_DENSE when threshold <= partition size (every sequence longer
 *     than one partition is split) and num_seqs * num_kv_heads < num_sms;
 *   PA_AUTO_WORKLIST otherwise.
 * With the default threshold, a batch that would take the dense form runs
 * single pass instead (threshold raised to max_seq_len) when its single-pass
 * grid, each unit split over a cluster of C CTAs, fits one wave of resident
 * CTAs and ceil(max_seq_len / C) <= partition size: one launch for a batch
 * that small.
 * Any output pointer may be NULL.  num_sms <= 0 queries the current device.
 * Returns PA_OK, PA_ERR_INVALID_ARGUMENT or PA_ERR_UNSUPPORTED (a partition
 * size that is not a multiple of block_size).
 */
PA_API int pa_auto_resolve(int num_seqs, int num_kv_heads, int head_dim, int block_size,
                           int max_seq_len, long long max_total_tokens, int single_pass_max_len,
                           int partition_size, int num_sms, int *out_single_pass_max_len,
                           int *out_partition_size, int *out_form);

/*
 * pa_auto_workspace_bytes -- device workspace pa_decode_auto needs (bytes),
 * for at most `max_seq_len` tokens per sequence and, when
 * max_total_tokens > 0, at most that many tokens over the whole batch
 * (0 or less: no bound beyond num_seqs * max_seq_len).  With the bound the
 * work-list form keeps at most floor((T + S_p (P - 1)) / P) partition slots,
 * S_p = min(num_seqs, T / (threshold + 1)) (the sequences that can be longer
 * than the threshold), instead of num_seqs * ceil(max_seq_len / P).
 * single_pass_max_len < 0 and partition_size <= 0 select the heuristics
 * above (resolved on the current device, as pa_decode_auto resolves them).
 * Returns 0 on bad arguments; 256 when the single-pass form needs no
 * workspace.
 */
PA_API size_t pa_auto_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int max_seq_len,
                                      long long max_total_tokens, int single_pass_max_len,
                                      int partition_size);

/*
 * pa_decode_auto -- the whole decode step with a per-sequence choice of path
 * (the forward_decode heuristic).  A sequence with
 * seq_len <= single_pass_max_len is computed in one pass and written to out
 * directly; a longer one is split into ceil(L/partition_size) partitions whose
 * partials (kept in `workspace`) are merged by the log-sum-exp reduce.  The
 * device reads seq_lens itself, so the host needs only the upper bounds
 * `max_seq_len` (every seq_len must be <= it) and `max_total_tokens` (the sum
 * of seq_lens must be <= it when it is > 0); a batch beyond either bound
 * raises PA_DEV_TOO_MANY_PARTITIONS and the partitions past the bound are
 * dropped from the output.  single_pass_max_len < 0 and partition_size <= 0
 * select the launch heuristic (pa_auto_resolve gives the values and the
 * launch form it picks).  workspace: device memory of at least
 * pa_auto_workspace_bytes(...) bytes, 256-byte aligned, owned by the caller;
 * its contents need no initialisation and are scratch after the call; it may
 * be NULL when the single-pass form is taken.  Launches, on `stream`, one
 * kernel (single-pass form), two (dense form: attention, reduce) or three
 * (work-list form: plan, attention, reduce).
 */
PA_API int pa_decode_auto(void *out, const void *query, const void *key_cache,
                   const void *value_cache, const int32_t *block_tables,
                   const int32_t *seq_lens, int num_seqs, int num_q_heads,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   int max_blocks_per_seq, float scale, int max_seq_len,
                   long long max_total_tokens, int single_pass_max_len, int partition_size,
                   void *workspace, size_t workspace_bytes, pa_dtype_t dtype, void *stream);

/* Phases of pa_decode_auto_phases (bit mask). */
enum { PA_PHASE_PLAN = 1, PA_PHASE_ATTEND = 2, PA_PHASE_REDUCE = 4 };

/*
 * pa_decode_auto_phases -- pa_decode_auto split into its launches so a caller
 * can order other stream work (events, copies) between them: PA_PHASE_PLAN
 * builds the work list in `workspace` from seq_lens; PA_PHASE_ATTEND runs the
 * attention kernel (single-pass sequences write `out`, partitioned ones write
 * their partials to `workspace`); PA_PHASE_REDUCE merges the partials into
 * `out`.  A phase the resolved launch form does not have does nothing (the
 * single-pass form has only PA_PHASE_ATTEND, the dense form no PA_PHASE_PLAN).
 * All arguments must be the same for the phases of one step and the phases
 * must run in this order on one stream.  phases = PA_PHASE_PLAN |
 * PA_PHASE_ATTEND | PA_PHASE_REDUCE is exactly pa_decode_auto.  Other masks
 * return PA_ERR_INVALID_ARGUMENT.
 */
PA_API int pa_decode_auto_phases(void *out, const void *query, const void *key_cache,
                                 const void *value_cache, const int32_t *block_tables,
                                 const int32_t *seq_lens, int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, int max_blocks_per_seq, float scale,
                                 int max_seq_len, long long max_total_tokens,
                                 int single_pass_max_len, int partition_size, void *workspace,
                                 size_t workspace_bytes, pa_dtype_t dtype, void *stream,
                                 int phases);

/*
 * pa_decode_auto_static -- pa_decode_auto for callers that cannot allocate
 * device memory.  (The source pages describe no counterpart of this entry
 * point; it exists for the calling environments below.)
 *
 * Some callers cannot hand this library a workspace: a serving engine that
 * reserves almost all device memory for its KV cache at start-up (a later
 * cudaMalloc would fail), a hot loop that must not pay for the implicit
 * device-wide synchronisation a cudaMalloc / cudaFree can cause, or a plugin
 * host that passes in its tensors but exposes no allocator.  This entry point
 * takes the same arguments as pa_decode_auto minus the workspace, and keeps
 * its scratch (work list and partition partials) in one fixed array of
 * PA_STATIC_SCRATCH_BYTES (96 MiB) in device memory that belongs to the
 * library: enough for the partials of 256 sequences of up to 64K tokens and
 * 2.9M tokens in all at partition size 512 when max_total_tokens is given.
 * Every GPU that loads the library holds that array until the process exits.
 * The call allocates nothing.
 *
 *   - Limit: a batch whose pa_auto_workspace_bytes(...) exceeds
 *     PA_STATIC_SCRATCH_BYTES is rejected with PA_ERR_WORKSPACE_TOO_SMALL
 *     before anything is launched (use pa_decode_auto with your own
 *     workspace for it).
 *   - Set-up: the first call on each device looks up the array's device
 *     address (with that device current).  Make that first call before any
 *     stream capture.
 *   - Sharing: all calls on a device share the one array, and it keeps the
 *     previous call's contents; each call re-initialises what must start at
 *     zero (the work-list cursor) in its first kernel.  Calls whose kernels
 *     overlap on the GPU (for example on two streams) race on the array:
 *     serialise them.
 */
#define PA_STATIC_SCRATCH_BYTES ((size_t)96 << 20)

PA_API int pa_decode_auto_static(void *out, const void *query, const void *key_cache,
                                 const void *value_cache, const int32_t *block_tables,
                                 const int32_t *seq_lens, int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, int max_blocks_per_seq, float scale,
                                 int max_seq_len, long long max_total_tokens,
                                 int single_pass_max_len, int partition_size, pa_dtype_t dtype,
                                 void *stream);

/*
 * pa_prefill -- prefix prefill over the paged cache (page: project_6 commit
 * cd0d9e1, "qwen3_6_scripts", the prefix-prefill part of the paged_attn.py
 * rewrite: the new chunk of each sequence attends to the sequence's whole
 * cached context, gathered through the block table, and causally to itself).
 *
 * The chunk's own K/V must already be written to the cache: sequence s holds
 * L = seq_lens[s] tokens, the last n_s = q_start[s+1] - q_start[s] of which
 * are the chunk.  Query row r = q_start[s] + i (0 <= i < n_s) sits at
 * position p = L - n_s + i and gets
 *   out[r][h][:] = softmax_{t <= p}(scale * query[r][h] . k_t) weighted sum of v_t
 * (t over the sequence's cache tokens 0..p; GQA as in pa_decode).  With
 * n_s = 1 for every sequence this is pa_decode.
 *
 * Layouts: query, out [num_rows][num_q_heads][head_dim] (the sequences'
 * chunks one after another); q_start int32 [num_seqs + 1], non-decreasing,
 * q_start[0] = 0 and q_start[num_seqs] = num_rows; caches, block_tables,
 * seq_lens as above.  max_q_len: an upper bound of every n_s; the launch
 * covers max_q_len rounded up to whole CTAs (whole CTA pairs at head_dim 256),
 * and a chunk longer than that coverage raises PA_DEV_LEN_CLAMPED with its rows
 * past the coverage not written.  q_start is read on the
 * device only: a sequence whose rows fall outside [0, num_rows], or whose
 * chunk is longer than seq_lens[s], is skipped and raises PA_DEV_BAD_ROWS.
 * Supported: head_dim 64, 128 or 256, block_size 8 or a multiple of 16, GQA
 * group 1..128.  One kernel launch on `stream`; no workspace.
 */
PA_API int pa_prefill(void *out, const void *query, const void *key_cache,
                      const void *value_cache, const int32_t *block_tables,
                      const int32_t *seq_lens, const int32_t *q_start, int num_seqs,
                      int num_rows, int max_q_len, int num_q_heads, int num_kv_heads,
                      int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                      float scale, pa_dtype_t dtype, void *stream);

/*
 * pa_gather_kv -- test entry: copies each sequence's K and V rows, fetched
 * through the block table with the same tile loader the attention kernels
 * use, into dense arrays k_dense/v_dense [num_seqs][max_len][num_kv_heads]
 * [head_dim] (rows t < seq_lens[s]; rows t >= seq_len are not written).  Bit
 * patterns are copied unchanged, so the result can be compared bit for bit.
 */
PA_API int pa_gather_kv(void *k_dense, void *v_dense, const void *key_cache,
                 const void *value_cache, const int32_t *block_tables,
                 const int32_t *seq_lens, int num_seqs, int num_kv_heads,
                 int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                 int max_len, pa_dtype_t dtype, void *stream);

/*
 * pa_selftest_wait_timeout -- test entry for the failure path: launches one
 * warp that waits on a pipeline barrier which nothing completes (no copy is
 * issued), gives up after limit_us microseconds (1 .. 1,000,000) and raises
 * PA_DEV_WAIT_TIMEOUT, as the attention kernels do when a copy does not land.
 * The device stays usable; read the flag with pa_device_status().
 */
PA_API int pa_selftest_wait_timeout(void *stream, int limit_us);

/*
 * pa_device_status -- synchronises `stream`, returns in *flags the PA_DEV_*
 * flags raised by kernels on the current device since the last call, and
 * clears them.  Returns PA_OK, or PA_ERR_CUDA if synchronisation failed.
 */
PA_API int pa_device_status(void *stream, int *flags);

/* Human-readable name of a status code (static string). */
PA_API const char *pa_status_string(int status);

/* Library version, as major * 10000 + minor * 100 + patch. */
PA_API int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
