// pa_launch.cuh -- host-side launchers of the decode kernels.  Each dtype's
// translation unit includes this file and instantiates the launchers for its
// type (explicit instantiation), so the heavy templates compile in parallel.
#pragma once

#include <atomic>

#include "pa_kernels.cuh"
#include "pa_launch.h"

namespace pa {

// CTA shape of the attention kernel per head_dim: NW warps, NS stages per warp
// (build-time overridable with -DPA_NW_D<D>=... -DPA_NS_D<D>=... for tuning).
#ifndef PA_NW_D64
#define PA_NW_D64 4
#endif
#ifndef PA_NS_D64
#define PA_NS_D64 4
#endif
#ifndef PA_NW_D128
#define PA_NW_D128 4
#endif
#ifndef PA_NS_D128
#define PA_NS_D128 2
#endif
#ifndef PA_NW_D256
#define PA_NW_D256 4
#endif
#ifndef PA_NS_D256
#define PA_NS_D256 1   // 64 KB of stages: 3 CTAs (12 warps) per SM beat 1 CTA with 2 stages
#endif
// The single-pass grid may use a deeper ring (-DPA_NS_SINGLE_D<D>=...).
#ifndef PA_NS_SINGLE_D64
#define PA_NS_SINGLE_D64 PA_NS_D64
#endif
#ifndef PA_NS_SINGLE_D128
#define PA_NS_SINGLE_D128 PA_NS_D128
#endif
#ifndef PA_NS_SINGLE_D256
#define PA_NS_SINGLE_D256 PA_NS_D256
#endif
template <int D, int MODE> struct AttnCfg;
#define PA_CFG(DD)                                                                       \
    template <int MODE> struct AttnCfg<DD, MODE> {                                       \
        static constexpr int NW = PA_NW_D##DD;                                           \
        static constexpr int NS = MODE == kModeSingle ? PA_NS_SINGLE_D##DD : PA_NS_D##DD; \
    };
PA_CFG(64)
PA_CFG(128)
PA_CFG(256)
#undef PA_CFG

constexpr int kMaxDevices = 64;

// Opt a kernel into its dynamic shared memory size once per device.
template <typename K>
inline cudaError_t ensure_smem(K kernel, int bytes, std::atomic<int> *done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
}

template <typename T, int D, int MODE>
inline cudaError_t launch_attn_d(const CUtensorMap &tmK, const CUtensorMap &tmV, const Params &p,
                                 dim3 grid, cudaStream_t st) {
    using C = AttnCfg<D, MODE>;
    using SM = Smem<D, C::NW, C::NS>;
    static std::atomic<int> done[kMaxDevices];
    auto k = pa_attn_kernel<T, D, C::NW, C::NS, MODE>;
    cudaError_t e = ensure_smem(k, SM::kLaunchBytes, done);
    if (e != cudaSuccess) return e;
    if (MODE == kModeSingle && p.cluster > 1) {
        // the p.cluster CTAs of one unit form a thread-block cluster
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(C::NW * 32);
        cfg.dynamicSmemBytes = SM::kLaunchBytes;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, k, tmK, tmV, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    k<<<grid, C::NW * 32, SM::kLaunchBytes, st>>>(tmK, tmV, p);
    return cudaGetLastError();
}

template <typename T, int D, int MODE>
inline int attn_ctas_per_sm_d() {
    using C = AttnCfg<D, MODE>;
    using SM = Smem<D, C::NW, C::NS>;
    static std::atomic<int> done[kMaxDevices];
    auto k = pa_attn_kernel<T, D, C::NW, C::NS, MODE>;
    if (ensure_smem(k, SM::kLaunchBytes, done) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, C::NW * 32, SM::kLaunchBytes) !=
        cudaSuccess)
        return 0;
    return n;
}

template <typename T>
cudaError_t launch_attn(int D, int mode, const CUtensorMap &tmK, const CUtensorMap &tmV,
                        const Params &p, dim3 grid, cudaStream_t st) {
#define PA_MODES(DD)                                                                   \
    if (D == DD) {                                                                     \
        if (mode == kModeSingle) return launch_attn_d<T, DD, kModeSingle>(tmK, tmV, p, grid, st); \
        if (mode == kModePartitioned)                                                  \
            return launch_attn_d<T, DD, kModePartitioned>(tmK, tmV, p, grid, st);      \
        if (mode == kModeWorklist)                                                     \
            return launch_attn_d<T, DD, kModeWorklist>(tmK, tmV, p, grid, st);         \
    }
    PA_MODES(64)
    PA_MODES(128)
    PA_MODES(256)
#undef PA_MODES
    return cudaErrorInvalidValue;
}

template <typename T>
int attn_ctas_per_sm(int D, int mode) {
#define PA_OCC(DD)                                                                        \
    if (D == DD) {                                                                        \
        if (mode == kModeSingle) return attn_ctas_per_sm_d<T, DD, kModeSingle>();         \
        if (mode == kModePartitioned) return attn_ctas_per_sm_d<T, DD, kModePartitioned>(); \
        return attn_ctas_per_sm_d<T, DD, kModeWorklist>();                                \
    }
    PA_OCC(64)
    PA_OCC(128)
    PA_OCC(256)
#undef PA_OCC
    return 0;
}

template <typename T>
cudaError_t launch_reduce(int D, bool compact, const ReduceParams &r, dim3 grid, cudaStream_t st) {
#define PA_RED(DD)                                                                            \
    if (D == DD) {                                                                            \
        if (compact)                                                                          \
            pa_reduce_kernel<T, DD, true><<<grid, ReduceThreads<true>::value, 0, st>>>(r);    \
        else                                                                                  \
            pa_reduce_kernel<T, DD, false><<<grid, ReduceThreads<false>::value, 0, st>>>(r);  \
        return cudaGetLastError();                                                            \
    }
    PA_RED(64)
    PA_RED(128)
    PA_RED(256)
#undef PA_RED
    return cudaErrorInvalidValue;
}

#define PA_INSTANTIATE_LAUNCHERS(T)                                                             \
    template cudaError_t launch_attn<T>(int, int, const CUtensorMap &, const CUtensorMap &,     \
                                        const Params &, dim3, cudaStream_t);                    \
    template int attn_ctas_per_sm<T>(int, int);                                                 \
    template cudaError_t launch_reduce<T>(int, bool, const ReduceParams &, dim3, cudaStream_t);

}  // namespace pa
