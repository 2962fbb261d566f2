// pa_launch.cuh -- host-side launchers of the decode kernels.  Each dtype's
// translation unit includes this file and instantiates the launchers for its
// type (explicit instantiation), so the heavy templates compile in parallel.
#pragma once

#include <atomic>
#include <utility>

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

// Launch with programmatic stream serialisation (the kernel may start while
// the previous one in the stream drains; its grid_dep_wait() orders its global
// accesses after that kernel) and, when `cluster` > 1, a thread-block cluster
// of that many CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t st, const int *cluster, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster && *cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(*cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

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

template <typename T, int D, int MODE, int HP>
inline cudaError_t launch_attn_d(const CUtensorMap &tmK, const CUtensorMap &tmV, const Params &p,
                                 dim3 grid, cudaStream_t st) {
    using C = AttnCfg<D, MODE>;
    using SM = Smem<D, C::NW, C::NS, HP>;
    static std::atomic<int> done[kMaxDevices];
    auto k = pa_attn_kernel<T, D, C::NW, C::NS, MODE, HP>;
    cudaError_t e = ensure_smem(k, SM::kLaunchBytes, done);
    if (e != cudaSuccess) return e;
    // the p.cluster CTAs of one single-pass unit form a thread-block cluster
    const int cluster = MODE == kModeSingle ? p.cluster : 1;
    e = launch_dependent(k, grid, dim3(C::NW * 32), SM::kLaunchBytes, st, &cluster, tmK, tmV, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Resident CTAs per SM of one attention kernel, asked of the occupancy
// calculator once per device (it is on the launch path of every call).
template <typename T, int D, int MODE, int HP>
inline int attn_ctas_per_sm_d() {
    using C = AttnCfg<D, MODE>;
    using SM = Smem<D, C::NW, C::NS, HP>;
    static std::atomic<int> done[kMaxDevices];
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const int c = cached[dev].load(std::memory_order_acquire);
    if (c > 0) return c;
    auto k = pa_attn_kernel<T, D, C::NW, C::NS, MODE, HP>;
    if (ensure_smem(k, SM::kLaunchBytes, done) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, C::NW * 32, SM::kLaunchBytes) !=
        cudaSuccess)
        return 0;
    if (n > 0) cached[dev].store(n, std::memory_order_release);
    return n;
}

// Heads a unit holds: 16 (two MMA n-tiles) for head_dim 64 and 128, 8 for
// head_dim 256 (two n-tiles of O^T there would not fit the register file).
constexpr int heads_wide_ok(int D) { return D <= 128; }

template <typename T>
cudaError_t launch_attn(int D, int mode, int hp, const CUtensorMap &tmK, const CUtensorMap &tmV,
                        const Params &p, dim3 grid, cudaStream_t st) {
#define PA_MODES(DD, HH)                                                                       \
    if (D == DD && hp == HH) {                                                                 \
        if (mode == kModeSingle)                                                               \
            return launch_attn_d<T, DD, kModeSingle, HH>(tmK, tmV, p, grid, st);               \
        if (mode == kModePartitioned)                                                          \
            return launch_attn_d<T, DD, kModePartitioned, HH>(tmK, tmV, p, grid, st);          \
        if (mode == kModeWorklist)                                                             \
            return launch_attn_d<T, DD, kModeWorklist, HH>(tmK, tmV, p, grid, st);             \
    }
    PA_MODES(64, 8)
    PA_MODES(64, 16)
    PA_MODES(128, 8)
    PA_MODES(128, 16)
    PA_MODES(256, 8)
#undef PA_MODES
    return cudaErrorInvalidValue;
}

template <typename T>
int attn_ctas_per_sm(int D, int mode, int hp) {
#define PA_OCC(DD, HH)                                                                        \
    if (D == DD && hp == HH) {                                                                \
        if (mode == kModeSingle) return attn_ctas_per_sm_d<T, DD, kModeSingle, HH>();         \
        if (mode == kModePartitioned) return attn_ctas_per_sm_d<T, DD, kModePartitioned, HH>(); \
        return attn_ctas_per_sm_d<T, DD, kModeWorklist, HH>();                                \
    }
    PA_OCC(64, 8)
    PA_OCC(64, 16)
    PA_OCC(128, 8)
    PA_OCC(128, 16)
    PA_OCC(256, 8)
#undef PA_OCC
    return 0;
}

template <typename T>
cudaError_t launch_reduce(int D, bool compact, const ReduceParams &r, dim3 grid, cudaStream_t st) {
#define PA_RED(DD)                                                                            \
    if (D == DD) {                                                                            \
        const cudaError_t e =                                                                 \
            compact ? launch_dependent(pa_reduce_kernel<T, DD, true>, grid,                   \
                                       dim3(ReduceThreads<true>::value), 0, st, nullptr, r)   \
                    : launch_dependent(pa_reduce_kernel<T, DD, false>, grid,                  \
                                       dim3(ReduceThreads<false>::value), 0, st, nullptr, r); \
        return e != cudaSuccess ? e : cudaGetLastError();                                     \
    }
    PA_RED(64)
    PA_RED(128)
    PA_RED(256)
#undef PA_RED
    return cudaErrorInvalidValue;
}

#define PA_INSTANTIATE_LAUNCHERS(T)                                                             \
    template cudaError_t launch_attn<T>(int, int, int, const CUtensorMap &, const CUtensorMap &, \
                                        const Params &, dim3, cudaStream_t);                    \
    template int attn_ctas_per_sm<T>(int, int, int);                                            \
    template cudaError_t launch_reduce<T>(int, bool, const ReduceParams &, dim3, cudaStream_t);

}  // namespace pa
