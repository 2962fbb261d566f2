// pa_prefill.cu -- the prefix-prefill kernels instantiated for bf16 and f16,
// and the choice between them per head_dim: head_dim 256 runs on CTA pairs
// sharing 2-SM MMAs (pa_prefill_pair.cuh), head_dim 64 and 128 on single CTAs
// with two Q tiles each (pa_prefill_tc.cuh).
#include "pa_prefill_pair.cuh"

#ifndef PA_PREFILL_PAIR_D128
#define PA_PREFILL_PAIR_D128 0
#endif

namespace pa {

template <typename T>
cudaError_t launch_prefill_tc(int D, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                              const CUtensorMap &tmV, const PrefillParams &p, dim3 grid,
                              cudaStream_t st) {
    if (D == 64) return launch_prefill_tc_d<T, 64>(tmQ, tmK, tmV, p, grid, st);
#if PA_PREFILL_PAIR_D128
    if (D == 128) return launch_prefill_pair_d<T, 128>(tmQ, tmK, tmV, p, grid, st);
#else
    if (D == 128) return launch_prefill_tc_d<T, 128>(tmQ, tmK, tmV, p, grid, st);
#endif
    if (D == 256) return launch_prefill_pair_d<T, 256>(tmQ, tmK, tmV, p, grid, st);
    return cudaErrorInvalidValue;
}

template cudaError_t launch_prefill_tc<__nv_bfloat16>(int, const CUtensorMap &,
                                                      const CUtensorMap &, const CUtensorMap &,
                                                      const PrefillParams &, dim3, cudaStream_t);
template cudaError_t launch_prefill_tc<__half>(int, const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, const PrefillParams &, dim3,
                                               cudaStream_t);

int prefill_rows_per_cta(int D) {
    if (D == 64) return PrefillTcCfg<64>::kRows;
#if PA_PREFILL_PAIR_D128
    if (D == 128) return PrefillPairCfg<128>::kRows;
#else
    if (D == 128) return PrefillTcCfg<128>::kRows;
#endif
    if (D == 256) return PrefillPairCfg<256>::kRows;
    return 0;
}

int prefill_v_box_pieces(int D) {
    if (D == 64) return PrefillTcCfg<64>::kPieces;
#if PA_PREFILL_PAIR_D128
    if (D == 128) return PrefillPairCfg<128>::kVPieces;
#else
    if (D == 128) return PrefillTcCfg<128>::kPieces;
#endif
    if (D == 256) return PrefillPairCfg<256>::kVPieces;
    return 0;
}
}  // namespace pa
