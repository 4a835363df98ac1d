// pa_cache.cu -- slot writer (reshape_and_cache), copy-on-write block copies,
// and the per-device error word.
//
// Slot writer: how-pagedattention-works (aiinfrainterviews.com), "A strong
// answer" -- the cache grows by one token per decode step, stored in the next
// slot of the sequence's last block; the slot is the linear form of the
// (table[t // b], t % b) address of auto-20261007-1900-en (lihaoran.work), "A
// block table maps logical order to physical storage".
// Block copies: how-pagedattention-works, feature table (beam-search row) and
// attn-paged-attention-mcq-hard (zenaique.com), the beam-search follow-up --
// forks share blocks and a diverging block is copied into a fresh one.
//
// Both kernels move 16-byte vectors (8 bf16): a (block, K/V, head) slab is
// contiguous, so each token row of d elements is d/8 coalesced 16-B accesses.
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__device__ unsigned int g_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned int *g_error_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];

// Launch with programmatic stream serialisation: the kernel's launch overlaps
// the previous kernel's tail; its griddepcontrol.wait orders the data.
template <typename Kernel, typename Arg>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, cudaStream_t stream, const Arg &arg) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, arg);
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// ---- reshape_and_cache ------------------------------------------------------

struct CacheParams {
    uint4 *pool;                 // pool base as 16-B vectors
    int64_t num_blocks;
    int64_t block_stride_v;      // in 16-B vectors
    int64_t kv_stride_v;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t row_vecs;            // head_dim / 8
    const uint4 *k;
    const uint4 *v;
    const int64_t *slots;
    int64_t num_tokens;
    unsigned int *err;
};

// One thread per 16-B vector of a (token, K/V, head) row.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const CacheParams p) {
    // inputs may come from the previous kernel; the next one may be scheduled
    // once this CTA has passed that wait (so every kernel before this one has
    // finished: a caller's promise about the kernel immediately before the
    // next call holds), and still waits for this grid to finish
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t per_token = 2ll * p.num_kv_heads * p.row_vecs;
    const int64_t total = p.num_tokens * per_token;
    const int64_t slot_limit = p.num_blocks * p.block_size;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = idx / per_token;
        int64_t r = idx - n * per_token;
        const int kv = (int)(r / ((int64_t)p.num_kv_heads * p.row_vecs));
        r -= (int64_t)kv * p.num_kv_heads * p.row_vecs;
        const int h = (int)(r / p.row_vecs);
        const int c = (int)(r - (int64_t)h * p.row_vecs);
        const int64_t slot = __ldg(p.slots + n);
        if (slot < 0) continue;  // padding
        if (slot >= slot_limit) {
            if (kv == 0 && h == 0 && c == 0) raise_error(p.err, PA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / p.block_size;
        const int off = (int)(slot - blk * p.block_size);
        const uint4 *src = (kv ? p.v : p.k) + (n * p.num_kv_heads + h) * p.row_vecs + c;
        uint4 *dst = p.pool + blk * p.block_stride_v + kv * p.kv_stride_v +
                     ((int64_t)h * p.block_size + off) * p.row_vecs + c;
        *dst = __ldg(src);
    }
}

// ---- copy_blocks --------------------------------------------------------------

struct CopyParams {
    uint4 *pool;
    int64_t num_blocks;
    int64_t block_stride_v;
    int64_t kv_stride_v;
    int64_t half_vecs;           // Hkv * b * d / 8: one K (or V) half of a block
    const int32_t *pairs;
    int32_t num_pairs;
    unsigned int *err;
};

// grid (num_pairs, 2): one CTA per (pair, K/V half); the half is contiguous.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int pair = blockIdx.x, kv = blockIdx.y;
    const int32_t src = __ldg(p.pairs + 2 * pair), dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
        if (kv == 0 && threadIdx.x == 0) raise_error(p.err, PA_DEVERR_BLOCK_ID);
        return;
    }
    const uint4 *s = p.pool + src * p.block_stride_v + kv * p.kv_stride_v;
    uint4 *d = p.pool + dst * p.block_stride_v + kv * p.kv_stride_v;
    constexpr int kUnroll = 4;
    int64_t i = threadIdx.x;
    for (; i + (kUnroll - 1) * blockDim.x < p.half_vecs; i += kUnroll * blockDim.x) {
        uint4 t[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) t[u] = s[i + u * blockDim.x];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) d[i + u * blockDim.x] = t[u];
    }
    for (; i < p.half_vecs; i += blockDim.x) d[i] = s[i];
}

struct SwapParams {
    uint4 *pool;
    int64_t num_blocks;
    int64_t block_stride_v;
    int64_t kv_stride_v;
    int64_t half_vecs;           // Hkv * b * d / 8: one K (or V) half of a block
    uint4 *host;                 // device view of the pinned host buffer [host_blocks][2][half]
    int64_t host_blocks;
    const int32_t *pairs;        // [n][2] (device block, host block)
    int32_t direction;           // PA_SWAP_OUT: pool -> host; PA_SWAP_IN: host -> pool
    unsigned int *err;
};

// grid (num_pairs, 2): one CTA per (pair, K/V half).  The host side is read or
// written directly through its device mapping, over the CPU-GPU link.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const SwapParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int pair = blockIdx.x, kv = blockIdx.y;
    const int32_t dev = __ldg(p.pairs + 2 * pair), hb = __ldg(p.pairs + 2 * pair + 1);
    if (dev < 0 || dev >= p.num_blocks || hb < 0 || hb >= p.host_blocks) {
        if (kv == 0 && threadIdx.x == 0) raise_error(p.err, PA_DEVERR_BLOCK_ID);
        return;
    }
    uint4 *pool_half = p.pool + dev * p.block_stride_v + kv * p.kv_stride_v;
    uint4 *host_half = p.host + ((int64_t)hb * 2 + kv) * p.half_vecs;
    const uint4 *s = p.direction == PA_SWAP_OUT ? pool_half : host_half;
    uint4 *d = p.direction == PA_SWAP_OUT ? host_half : pool_half;
    constexpr int kUnroll = 4;
    int64_t i = threadIdx.x;
    for (; i + (kUnroll - 1) * blockDim.x < p.half_vecs; i += kUnroll * blockDim.x) {
        uint4 t[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) t[u] = s[i + u * blockDim.x];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) d[i + u * blockDim.x] = t[u];
    }
    for (; i < p.half_vecs; i += blockDim.x) d[i] = s[i];
}

}  // namespace

unsigned int *device_error_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_error_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
        g_error_ptr[dev] = static_cast<unsigned int *>(ptr);
    }
    return g_error_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qres) ==
                cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

cudaError_t encode_pool_block_map(CUtensorMap *map, const PoolView &pool, int kv, int box_rows) {
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const int D = pool.head_dim, BS = pool.block_size;
    const char *base = static_cast<const char *>(pool.base) + (size_t)kv * pool.kv_stride * 2;
    cuuint64_t dims[5] = {64, (cuuint64_t)BS, (cuuint64_t)(D / 64), (cuuint64_t)pool.num_kv_heads,
                          (cuuint64_t)pool.num_blocks};
    cuuint64_t strides[4] = {(cuuint64_t)D * 2, 128, (cuuint64_t)BS * D * 2, (cuuint64_t)pool.block_stride * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)box_rows, (cuuint32_t)(D / 64), 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<char *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

int device_sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

// Stores the K/V of each sequence's last token (position seq_lens[s] - 1) at
// its slot through the block table: the slot writer's work for one decode
// step, with the slots derived on the device.  One thread per 16-B vector of
// a (sequence, K/V, head) row.
struct AppendParams {
    uint4 *pool;
    int64_t num_blocks;
    int64_t block_stride_v;
    int64_t kv_stride_v;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t row_vecs;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    int32_t num_seqs;
    int32_t max_len;             // lengths above this are invalid
    const uint4 *k;              // [B][Hkv][D]
    const uint4 *v;
    unsigned int *err;
};

__global__ void __launch_bounds__(256) append_last_kernel(const AppendParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // as in the slot writer
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t per_seq = 2ll * p.num_kv_heads * p.row_vecs;
    const int64_t total = (int64_t)p.num_seqs * per_seq;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int s = (int)(idx / per_seq);
        int64_t r = idx - (int64_t)s * per_seq;
        const int kv = (int)(r / ((int64_t)p.num_kv_heads * p.row_vecs));
        r -= (int64_t)kv * p.num_kv_heads * p.row_vecs;
        const int h = (int)(r / p.row_vecs), c = (int)(r % p.row_vecs);
        const int L = __ldg(p.seq_lens + s);
        if (L <= 0) continue;
        if (L > p.max_len || L > p.max_blocks * p.block_size) {
            if (kv == 0 && h == 0 && c == 0) raise_error(p.err, PA_DEVERR_SEQ_LEN);
            continue;
        }
        const int blk = __ldg(p.tables + (size_t)s * p.max_blocks + (L - 1) / p.block_size);
        if (blk < 0 || blk >= p.num_blocks) {
            if (kv == 0 && h == 0 && c == 0) raise_error(p.err, PA_DEVERR_BLOCK_ID);
            continue;
        }
        const int off = (L - 1) % p.block_size;
        const uint4 *src = (kv == 0 ? p.k : p.v) + ((size_t)s * p.num_kv_heads + h) * p.row_vecs + c;
        p.pool[blk * p.block_stride_v + kv * p.kv_stride_v + ((int64_t)h * p.block_size + off) * p.row_vecs + c] =
            *src;
    }
}

cudaError_t launch_append_last(const PoolView &pool, const int32_t *tables, int32_t max_blocks,
                               const int32_t *seq_lens, int32_t num_seqs, int32_t max_len, const void *k,
                               const void *v, cudaStream_t stream) {
    if (num_seqs == 0) return cudaSuccess;
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    AppendParams p;
    p.pool = reinterpret_cast<uint4 *>(const_cast<void *>(pool.base));
    p.num_blocks = pool.num_blocks;
    p.block_stride_v = pool.block_stride / 8;
    p.kv_stride_v = pool.kv_stride / 8;
    p.num_kv_heads = pool.num_kv_heads;
    p.block_size = pool.block_size;
    p.row_vecs = pool.head_dim / 8;
    p.tables = tables;
    p.max_blocks = max_blocks;
    p.seq_lens = seq_lens;
    p.num_seqs = num_seqs;
    p.max_len = max_len;
    p.k = static_cast<const uint4 *>(k);
    p.v = static_cast<const uint4 *>(v);
    p.err = err;
    const int64_t total = (int64_t)num_seqs * 2 * pool.num_kv_heads * p.row_vecs;
    const int threads = 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    int64_t blocks = (total + threads - 1) / threads;
    if (cap > 0 && blocks > cap) blocks = cap;
    return launch_pdl(append_last_kernel, dim3((unsigned)blocks), dim3(threads), stream, p);
}

// One CTA waits on a shared-memory barrier that no thread ever arrives at,
// through the same bounded wait every kernel uses, and gives up after
// limit_ns: the path a kernel takes when a copy or an MMA it waits for never
// completes, taken here without any fault.
__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned int *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, err, limit_ns);   // nothing arrives: records the timeout
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const PoolView &pool, const void *k, const void *v,
                                     const int64_t *slots, int64_t num_tokens, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    CacheParams p;
    p.pool = reinterpret_cast<uint4 *>(const_cast<void *>(pool.base));
    p.num_blocks = pool.num_blocks;
    p.block_stride_v = pool.block_stride / 8;
    p.kv_stride_v = pool.kv_stride / 8;
    p.num_kv_heads = pool.num_kv_heads;
    p.block_size = pool.block_size;
    p.row_vecs = pool.head_dim / 8;
    p.k = static_cast<const uint4 *>(k);
    p.v = static_cast<const uint4 *>(v);
    p.slots = slots;
    p.num_tokens = num_tokens;
    p.err = err;
    const int64_t total = num_tokens * 2 * pool.num_kv_heads * p.row_vecs;
    const int threads = 256;
    const int64_t max_blocks = (int64_t)device_sm_count() * 8;
    int64_t blocks = (total + threads - 1) / threads;
    if (max_blocks > 0 && blocks > max_blocks) blocks = max_blocks;
    return launch_pdl(reshape_and_cache_kernel, dim3((unsigned)blocks), dim3(threads), stream, p);
}

cudaError_t launch_copy_blocks(const PoolView &pool, const int32_t *pairs, int32_t num_pairs,
                               cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    CopyParams p;
    p.pool = reinterpret_cast<uint4 *>(const_cast<void *>(pool.base));
    p.num_blocks = pool.num_blocks;
    p.block_stride_v = pool.block_stride / 8;
    p.kv_stride_v = pool.kv_stride / 8;
    p.half_vecs = (int64_t)pool.num_kv_heads * pool.block_size * pool.head_dim / 8;
    p.pairs = pairs;
    p.num_pairs = num_pairs;
    p.err = err;
    return launch_pdl(copy_blocks_kernel, dim3(num_pairs, 2), dim3(256), stream, p);
}

cudaError_t launch_swap_blocks(const PoolView &pool, void *host_dev, int64_t host_blocks, const int32_t *pairs,
                               int32_t num_pairs, int32_t direction, cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    SwapParams p;
    p.pool = reinterpret_cast<uint4 *>(const_cast<void *>(pool.base));
    p.num_blocks = pool.num_blocks;
    p.block_stride_v = pool.block_stride / 8;
    p.kv_stride_v = pool.kv_stride / 8;
    p.half_vecs = (int64_t)pool.num_kv_heads * pool.block_size * pool.head_dim / 8;
    p.host = static_cast<uint4 *>(host_dev);
    p.host_blocks = host_blocks;
    p.pairs = pairs;
    p.direction = direction;
    p.err = err;
    return launch_pdl(swap_blocks_kernel, dim3(num_pairs, 2), dim3(256), stream, p);
}

}  // namespace pa
