// pa_prefill.cu -- the prefix-prefill kernel instantiated for bf16 and f16.
#include "pa_prefill_tc.cuh"

namespace pa {
template cudaError_t launch_prefill_tc<__nv_bfloat16>(int, const CUtensorMap &,
                                                      const CUtensorMap &, const CUtensorMap &,
                                                      const PrefillParams &, dim3, cudaStream_t);
template cudaError_t launch_prefill_tc<__half>(int, const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, const PrefillParams &, dim3,
                                               cudaStream_t);

int prefill_rows_per_cta(int D) {
    if (D == 64) return PrefillTcCfg<64>::kRows;
    if (D == 128) return PrefillTcCfg<128>::kRows;
    if (D == 256) return PrefillTcCfg<256>::kRows;
    return 0;
}
}  // namespace pa
