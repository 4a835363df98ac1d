// pa_decode_noalloc.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// pa_decode needs a caller-provided workspace for its split-context partial
// results.  Some callers cannot obtain one: a plugin that a host framework
// hands only its input and output buffers (the framework owns every byte of
// device memory through its own allocator), or a latency-critical serving
// loop where cudaMalloc -- which may synchronise the device -- is not allowed
// once serving has started.  pa_decode_noalloc gives them the same decode
// with the workspace taken from a fixed array in the library's own device
// memory instead.
//
// The array (kNoAllocScratchBytes, 8 MiB) is a file-scope __device__
// variable: every GPU that loads the library holds it until the process
// exits.  Host code cannot use the array's name as a device address, so the
// first call on each device looks the address up with cudaGetSymbolAddress
// while that device is current and caches it; that first call should
// therefore happen before any stream capture begins.
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

// Shared by every call on a device; it keeps whatever the last call wrote.
// Nothing in it has to start at zero: each call writes every partial record
// before its reduce kernel reads it.  Two calls whose kernels overlap on the
// GPU (for example on two streams) race on this array.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices];

// Device address of this device's scratch array (looked up once per device).
void *scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace pa

extern "C" {

pa_status pa_decode_noalloc(void *out, const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_seq_len, float scale, int32_t partition_tokens,
                            cudaStream_t stream) {
    const size_t need = pa_decode_workspace_size(pool, num_seqs, num_q_heads, max_seq_len, partition_tokens);
    if (need > pa::kNoAllocScratchBytes) return PA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        scratch = pa::scratch_address();
        if (!scratch) return PA_ERR_CUDA;
    }
    return pa_decode(out, q, pool, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, max_seq_len,
                     scale, partition_tokens, scratch, need > 0 ? pa::kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"
