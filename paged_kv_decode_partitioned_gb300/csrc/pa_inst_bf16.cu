// pa_inst_bf16.cu -- attention and reduce kernels instantiated for bf16.
#include "pa_launch.cuh"

namespace pa {
PA_INSTANTIATE_LAUNCHERS(__nv_bfloat16)
}  // namespace pa
