// pa_launch.h -- declarations of the kernel launchers.  The attention and
// reduce launchers are templates explicitly instantiated per dtype in
// pa_inst_bf16.cu / pa_inst_f16.cu, the prefill launcher in pa_prefill.cu;
// the planner and gather launchers live in pa_aux.cu, the MoE router and
// regrouping launchers in pa_moe.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_types.h"

namespace pa {

// hp: query heads a unit holds (8, or 16 for head_dim 64 / 128)
template <typename T>
cudaError_t launch_attn(int D, int mode, int hp, const CUtensorMap &tmK, const CUtensorMap &tmV,
                        const Params &p, dim3 grid, cudaStream_t st);
template <typename T>
int attn_ctas_per_sm(int D, int mode, int hp);
template <typename T>
cudaError_t launch_reduce(int D, bool compact, const ReduceParams &r, dim3 grid, cudaStream_t st);

template <typename T>
cudaError_t launch_prefill_tc(int D, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                              const CUtensorMap &tmV, const PrefillParams &p, dim3 grid,
                              cudaStream_t st);

// Query rows (chunk token x group head) one prefill CTA covers at head_dim D.
int prefill_rows_per_cta(int D);
// 64-column pieces of a 16-token V box one prefill copy moves at head_dim D:
// every piece of the row on single CTAs, the CTA's half on CTA pairs.
int prefill_v_box_pieces(int D);

cudaError_t launch_plan(const PlanParams &pp, cudaStream_t st);
cudaError_t launch_wait_timeout_test(int *status, unsigned long long limit_ns, cudaStream_t st);
cudaError_t launch_gather(int D, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          const GatherParams &gp, dim3 grid, cudaStream_t st);

cudaError_t launch_topk_softmax(int logits_type, int num_experts, const TopkParams &p,
                                cudaStream_t st);
int moe_sort_chunks(int num_pairs);
cudaError_t launch_moe_sort(const SortParams &p, cudaStream_t st);
cudaError_t launch_moe_gather(const MoeGatherParams &p, cudaStream_t st);
cudaError_t launch_moe_scatter(bool bf16, const MoeScatterParams &p, cudaStream_t st);

}  // namespace pa
