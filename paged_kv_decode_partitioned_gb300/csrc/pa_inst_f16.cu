// pa_inst_f16.cu -- attention and reduce kernels instantiated for f16.
#include "pa_launch.cuh"

namespace pa {
PA_INSTANTIATE_LAUNCHERS(__half)
}  // namespace pa
