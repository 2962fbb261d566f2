/*
 * pa_moe.h -- C ABI of the MoE router and token-regrouping kernels in
 * libpadecode.so (GB300, sm_103a).
 *
 * The operations (page: project_6 commit cd0d9e1, "qwen3_6_scripts", the MoE
 * prefill rewrite: 256 experts x top_k = 8; the T x K token-expert pairs are
 * flattened and sorted by expert id so each expert's tokens are contiguous,
 * the hidden rows are gathered in that order, and the expert outputs are
 * scattered back with index_add_; page: commit 490ff98, "Dockerfile": the
 * topk_softmax router kernel):
 *
 *   router     pa_topk_softmax      logits -> top-k expert ids and weights
 *   regroup    pa_moe_sort          ids -> expert-sorted pair order, offsets
 *              pa_moe_gather        hidden rows in that order (contiguous per expert)
 *   (the per-expert GEMMs and their activation are not part of this library)
 *   combine    pa_moe_scatter_back  per-pair outputs -> token rows, weighted
 *
 * Conventions are those of pa_decode.h: device pointers owned by the caller,
 * row-major, asynchronous on `stream`, every argument checked on the host
 * before a launch, status codes PA_OK / PA_ERR_*.  A flat pair index is
 * p = t * topk + k (token t, slot k).  Contents read only on the device
 * (expert ids, pair indices) that are out of range raise PA_DEV_BAD_EXPERT
 * in the device status word (pa_device_status) and are skipped.
 */
#ifndef PA_MOE_H
#define PA_MOE_H

#include "pa_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Router logits element type. */
typedef enum { PA_LOGITS_F16 = 0, PA_LOGITS_BF16 = 1, PA_LOGITS_F32 = 2 } pa_logits_t;

/* Device status flag of these kernels (shares the word of pa_decode.h). */
enum { PA_DEV_BAD_EXPERT = 32 };

/*
 * pa_topk_softmax -- the router.  For token t with logits x[t][0..E):
 *   p_e = exp(x_e - max x) / sum_e' exp(x_e' - max x)      (fp32)
 *   ids[t][0..k)     = the k experts with the largest logits, in descending
 *                      order, ties to the lower expert id (softmax is
 *                      monotonic, so these are the k largest p_e; choosing on
 *                      the logits makes the ids exact);
 *   weights[t][j]    = p_{ids[t][j]}, divided by their sum over j when
 *                      renormalize != 0.
 * logits [num_tokens][num_experts] (16-byte aligned), weights fp32 and ids
 * int32 [num_tokens][topk].  Supported: num_experts in {32, 64, 128, 256,
 * 512}; 1 <= topk <= min(32, num_experts).  One launch.
 */
PA_API int pa_topk_softmax(float *topk_weights, int32_t *topk_ids, const void *gating_logits,
                           int num_tokens, int num_experts, int topk, int renormalize,
                           pa_logits_t logits_dtype, void *stream);

/* Device workspace pa_moe_sort needs (bytes); 0 on bad arguments. */
PA_API size_t pa_moe_sort_workspace_bytes(int num_pairs, int num_experts);

/*
 * pa_moe_sort -- stable sort of the flat pairs by expert id:
 *   sorted_pairs [num_pairs]      pair indices, expert 0's first, and within
 *                                 one expert in increasing pair index;
 *   expert_offsets [E + 1]        first sorted position of each expert;
 *                                 expert_offsets[E] = number of pairs placed;
 *   pair_pos [num_pairs]          sorted position of each pair (the inverse
 *                                 permutation); -1 for a pair whose expert id
 *                                 is outside [0, E) (flagged, not placed).
 * expert_ids [num_pairs] int32 (the router's ids, flattened).  workspace: at
 * least pa_moe_sort_workspace_bytes(...) bytes, 256-byte aligned, scratch.
 * Supported: 1 <= num_experts <= 1024.  Three launches.
 */
PA_API int pa_moe_sort(int32_t *sorted_pairs, int32_t *expert_offsets, int32_t *pair_pos,
                       const int32_t *expert_ids, int num_pairs, int num_experts,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_moe_gather -- the hidden rows in expert-sorted order, so each expert's
 * rows are contiguous: sorted_hidden[r][:] = hidden[t][:] for the pair
 * p = t * topk + k placed at r = pair_pos[p] (bit copies; the same rows as
 * sorted_hidden[r] = hidden[sorted_pairs[r] / topk]).  It runs token-major:
 * each hidden row is read once and written to its topk positions.
 * hidden [num_tokens][hidden_size], sorted_hidden [num_rows][hidden_size]
 * (num_rows = the rows the output holds, num_tokens * topk when every pair is
 * placed), both 16-byte aligned; hidden_size * 2 bytes a multiple of 16;
 * topk <= 32.  pair_pos as written by pa_moe_sort: a pair at -1 (not placed)
 * is skipped; a position outside [0, num_rows) is skipped and flagged.  One
 * launch.
 */
PA_API int pa_moe_gather(void *sorted_hidden, const void *hidden, const int32_t *pair_pos,
                         int num_tokens, int topk, int num_rows, int hidden_size,
                         pa_dtype_t dtype, void *stream);

/*
 * pa_moe_scatter_back -- index_add_ of the weighted per-pair rows into the
 * token rows, written as a gather-reduce:
 *   out[t][:] = sum_{k < topk} topk_weights[t][k] * expert_out[pair_pos[t*topk + k]][:]
 * accumulated in fp32 in slot order and rounded once to dtype (deterministic,
 * no atomics).  expert_out [num_tokens * topk][hidden_size] in sorted order,
 * out [num_tokens][hidden_size]; pair_pos and topk_weights as produced by
 * pa_moe_sort and pa_topk_softmax.  A pair with pair_pos outside the rows adds
 * nothing (flagged).  Supported: 1 <= topk <= 32, hidden_size a multiple of
 * 8.  One launch.
 */
PA_API int pa_moe_scatter_back(void *out, const void *expert_out, const int32_t *pair_pos,
                               const float *topk_weights, int num_tokens, int topk,
                               int hidden_size, pa_dtype_t dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_MOE_H */
