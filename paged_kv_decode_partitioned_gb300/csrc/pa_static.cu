// pa_static.cu -- pa_decode_auto_static: the mixed decode step with its
// scratch in a fixed device array that belongs to the library, for callers
// that cannot allocate device memory (see include/pa_decode.h).
#include <cuda_runtime.h>

#include <mutex>

#include "pa_decode.h"

namespace {

// The scratch of pa_decode_auto_static: work list and partition partials.
// Every device that loads this library holds it until the process exits.
static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void *g_addr[kMaxDev];   // device address of the array, looked up once per device

// In host code g_pa_static_scratch names a host-side stand-in, not device
// memory; the device address comes from the runtime, once per device, with
// that device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return PA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_static_scratch) != cudaSuccess || p == nullptr)
            return PA_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_auto_static(void *out, const void *query, const void *key_cache,
                                     const void *value_cache, const int32_t *block_tables,
                                     const int32_t *seq_lens, int num_seqs, int num_q_heads,
                                     int num_kv_heads, int head_dim, int block_size,
                                     int num_blocks, int max_blocks_per_seq, float scale,
                                     int max_seq_len, long long max_total_tokens,
                                     int single_pass_max_len, int partition_size,
                                     pa_dtype_t dtype, void *stream) {
    // The size check resolves the launch heuristic (threshold, partition
    // size, launch form) exactly as pa_decode_auto will on this device.
    const size_t need = pa_auto_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                block_size, max_seq_len, max_total_tokens,
                                                single_pass_max_len, partition_size);
    if (need == 0) return PA_ERR_INVALID_ARGUMENT;
    if (need > PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != PA_OK) return rc;
    // The planner (first kernel of the work-list form) resets the work-list
    // cursor and rewrites the work list; every partial is written before it
    // is read.
    return pa_decode_auto(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          max_blocks_per_seq, scale, max_seq_len, max_total_tokens,
                          single_pass_max_len, partition_size, scratch, PA_STATIC_SCRATCH_BYTES,
                          dtype, stream);
}
