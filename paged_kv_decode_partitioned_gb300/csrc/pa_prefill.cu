// pa_prefill.cu -- the prefix-prefill kernel instantiated for bf16 and f16.
#include "pa_prefill_tc.cuh"

namespace pa {
template cudaError_t launch_prefill_tc<__nv_bfloat16>(int, const CUtensorMap &,
                                                      const CUtensorMap &, const CUtensorMap &,
                                                      const PrefillParams &, dim3, cudaStream_t);
template cudaError_t launch_prefill_tc<__half>(int, const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, const PrefillParams &, dim3,
                                               cudaStream_t);
}  // namespace pa
