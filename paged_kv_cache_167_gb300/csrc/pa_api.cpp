// pa_api.cpp -- the C ABI (include/pa.h): argument validation, partition
// planning and dispatch to the kernels.  Host code only; it allocates no
// device memory and launches nothing when validation fails.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cuda_runtime_api.h>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
cudaError_t launch_decode_d64(const DecodeArgs &a, cudaStream_t stream);
cudaError_t launch_decode_d128(const DecodeArgs &a, cudaStream_t stream);

namespace {

#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 4
#endif
constexpr int kDecodeWarps = PA_DECODE_WARPS;  // warps per decode CTA (must match the kernel)
#ifndef PA_DECODE_SK_CTAS_PER_SM
#define PA_DECODE_SK_CTAS_PER_SM 2
#endif
constexpr int kStreamKCtasPerSm = PA_DECODE_SK_CTAS_PER_SM;     // resident decode CTAs per SM (persistent stream-K grid)
constexpr size_t kWsAlign = 256;

// pa_set_stream_k_ctas: a fixed balanced-schedule grid size (0: two per SM).
std::atomic<int32_t> g_stream_k_ctas{0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Resolves a public pool descriptor into a PoolView; PA_OK or the reason.
pa_status resolve_pool(const pa_kv_pool *pool, PoolView *out) {
    if (!pool || !pool->base || !aligned16(pool->base)) return PA_ERR_INVALID_ARG;
    if (pool->dtype != PA_DTYPE_BF16) return PA_ERR_UNSUPPORTED;
    if (pool->num_blocks <= 0 || pool->num_kv_heads <= 0 || pool->block_size <= 0 || pool->head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (pool->head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
    const int64_t slab = (int64_t)pool->num_kv_heads * pool->block_size * pool->head_dim;
    const int64_t kv_stride = pool->kv_stride ? pool->kv_stride : slab;
    const int64_t block_stride = pool->block_stride ? pool->block_stride : 2 * slab;
    if (kv_stride < slab || block_stride < kv_stride + slab) return PA_ERR_INVALID_ARG;
    if ((kv_stride * 2) % 16 != 0 || (block_stride * 2) % 16 != 0) return PA_ERR_INVALID_ARG;
    out->base = pool->base;
    out->num_blocks = pool->num_blocks;
    out->num_kv_heads = pool->num_kv_heads;
    out->block_size = pool->block_size;
    out->head_dim = pool->head_dim;
    out->block_stride = block_stride;
    out->kv_stride = kv_stride;
    return PA_OK;
}

struct DecodePlan {
    bool stream_k;            // automatic plan: persistent balanced schedule
    int32_t partition_tokens; // split-context plan
    int32_t num_partitions;
    int32_t num_ctas;         // stream-K grid
    size_t ws_o_bytes;
    size_t ws_ml_bytes;
    size_t total_bytes() const { return ws_o_bytes + ws_ml_bytes; }
};

pa_status plan_decode(const PoolView &pool, int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                      int32_t partition_tokens, DecodePlan *plan) {
    if (num_seqs < 0 || num_q_heads <= 0 || max_seq_len < 0 || partition_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads % pool.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int group = num_q_heads / pool.num_kv_heads;
    if (!decode_supported(pool.head_dim, group, pool.block_size)) return PA_ERR_UNSUPPORTED;
    *plan = DecodePlan{};
    if (partition_tokens == 0) {
        // Persistent stream-K: two CTAs per SM share all (sequence, kv-head,
        // stage) work equally; at most two partial records per CTA.
        const int64_t stage = decode_stage_tokens(pool.block_size);
        const int64_t max_stages = (int64_t)num_seqs * pool.num_kv_heads * ceil_div(max_seq_len, stage);
        int64_t ctas = g_stream_k_ctas.load(std::memory_order_relaxed);
        if (ctas <= 0) {
            int sms = device_sm_count();
            if (sms <= 0) sms = 148;
            ctas = (int64_t)sms * kStreamKCtasPerSm;
        }
        if (ctas > max_stages) ctas = max_stages;
        if (ctas < 1) ctas = 1;
        plan->stream_k = true;
        plan->partition_tokens = max_seq_len > 0 ? max_seq_len : 1;   // length bound used by the kernel
        plan->num_partitions = 1;
        plan->num_ctas = (int32_t)ctas;
        plan->ws_o_bytes = round_up((size_t)2 * ctas * group * pool.head_dim * sizeof(float), kWsAlign);
        plan->ws_ml_bytes = round_up((size_t)2 * ctas * group * 2 * sizeof(float), kWsAlign);
        return PA_OK;
    }
    if (partition_tokens % pool.block_size != 0) return PA_ERR_INVALID_ARG;
    const int64_t parts = max_seq_len > 0 ? ceil_div(max_seq_len, partition_tokens) : 1;
    if (parts > 65535) return PA_ERR_INVALID_ARG;
    plan->partition_tokens = partition_tokens;
    plan->num_partitions = (int32_t)parts;
    if (parts > 1) {
        const size_t rows = (size_t)num_seqs * num_q_heads * (size_t)parts;
        plan->ws_o_bytes = round_up(rows * pool.head_dim * sizeof(float), kWsAlign);
        plan->ws_ml_bytes = round_up(rows * 2 * sizeof(float), kWsAlign);
    }
    return PA_OK;
}

}  // namespace

int decode_stage_tokens(int) { return 16; }

bool decode_supported(int head_dim, int group, int block_size) {
    const bool d_ok = head_dim == 64 || head_dim == 128;
    const bool g_ok = group == 1 || group == 2 || group == 4 || group == 8;
    const bool b_ok = block_size == 4 || block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64;
    return d_ok && g_ok && b_ok;
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    switch (a.pool.head_dim) {
        case 64: return launch_decode_d64(a, stream);
        case 128: return launch_decode_d128(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa

using namespace pa;

extern "C" {

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_DEVICE: return "device error word is set";
        case PA_ERR_NO_BLOCKS: return "no free block left";
        case PA_ERR_NOT_FOUND: return "unknown sequence";
        case PA_ERR_SWAPPED: return "sequence is swapped out";
    }
    return "unknown status";
}

int32_t pa_version(void) { return 10000; }

pa_status pa_reshape_and_cache(const pa_kv_pool *pool, const void *k, const void *v,
                               const int64_t *slot_mapping, int64_t num_tokens, cudaStream_t stream) {
    PoolView view;
    pa_status st = resolve_pool(pool, &view);
    if (st != PA_OK) return st;
    if (num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !aligned16(k) || !aligned16(v)) return PA_ERR_INVALID_ARG;
    return launch_reshape_and_cache(view, k, v, slot_mapping, num_tokens, stream) == cudaSuccess ? PA_OK
                                                                                                 : PA_ERR_CUDA;
}

size_t pa_decode_workspace_size(const pa_kv_pool *pool, int32_t num_seqs, int32_t num_q_heads,
                                int32_t max_seq_len, int32_t partition_tokens) {
    PoolView view;
    if (resolve_pool(pool, &view) != PA_OK) return 0;
    DecodePlan plan;
    if (plan_decode(view, num_seqs, num_q_heads, max_seq_len, partition_tokens, &plan) != PA_OK) return 0;
    return plan.total_bytes();
}

int32_t pa_decode_partition_tokens(const pa_kv_pool *pool, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t max_seq_len, int32_t partition_tokens) {
    PoolView view;
    if (resolve_pool(pool, &view) != PA_OK) return -1;
    DecodePlan plan;
    if (plan_decode(view, num_seqs, num_q_heads, max_seq_len, partition_tokens, &plan) != PA_OK) return -1;
    return plan.stream_k ? 0 : plan.partition_tokens;
}

pa_status pa_decode(void *out, const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t max_seq_len, float scale, int32_t partition_tokens, void *workspace,
                    size_t workspace_bytes, cudaStream_t stream) {
    return pa_decode_ex(out, q, pool, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_q_heads,
                        max_seq_len, scale, partition_tokens, workspace, workspace_bytes, nullptr, nullptr, 0u,
                        stream);
}

namespace {

pa_status decode_impl(void *out, const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                      int32_t max_seq_len, float scale, int32_t partition_tokens, void *workspace,
                      size_t workspace_bytes, const float *prefix_o, const float *prefix_lse, const void *new_k,
                      const void *new_v, uint32_t flags, cudaStream_t stream) {
    if ((flags & ~PA_DECODE_EARLY_METADATA) != 0) return PA_ERR_INVALID_ARG;
    if ((new_k == nullptr) != (new_v == nullptr)) return PA_ERR_INVALID_ARG;
    if (new_k && (!aligned16(new_k) || !aligned16(new_v))) return PA_ERR_INVALID_ARG;
    PoolView view;
    pa_status st = resolve_pool(pool, &view);
    if (st != PA_OK) return st;
    DecodePlan plan;
    st = plan_decode(view, num_seqs, num_q_heads, max_seq_len, partition_tokens, &plan);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !block_tables || !seq_lens || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (num_seqs > 65535) return PA_ERR_INVALID_ARG;
    if (plan.total_bytes() > 0) {
        if (!workspace || workspace_bytes < plan.total_bytes()) return PA_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0) return PA_ERR_WORKSPACE;
    }
    DecodeArgs a;
    a.out = out;
    a.q = q;
    a.pool = view;
    a.tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.max_seq_len = max_seq_len;
    a.scale = scale;
    a.partition_tokens = plan.partition_tokens;
    a.num_partitions = plan.num_partitions;
    char *ws = static_cast<char *>(workspace);
    a.ws_o = plan.ws_o_bytes ? reinterpret_cast<float *>(ws) : nullptr;
    a.ws_ml = plan.ws_ml_bytes ? reinterpret_cast<float *>(ws + plan.ws_o_bytes) : nullptr;
    a.stream_k = plan.stream_k;
    a.num_ctas = plan.num_ctas;
    a.early_meta = (flags & PA_DECODE_EARLY_METADATA) != 0;
    a.pre_o = prefix_o;
    a.pre_lse = prefix_lse;
    if (new_k) {
        if (plan.stream_k) {   // the stream-K kernel stores each last token itself
            a.new_k = new_k;
            a.new_v = new_v;
        } else if (launch_append_last(view, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                                      plan.partition_tokens * plan.num_partitions, new_k, new_v,
                                      stream) != cudaSuccess) {
            return PA_ERR_CUDA;
        }
    }
    return launch_decode(a, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

pa_status pa_decode_ex(void *out, const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                       int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t max_seq_len, float scale, int32_t partition_tokens, void *workspace,
                       size_t workspace_bytes, const void *new_k, const void *new_v, uint32_t flags,
                       cudaStream_t stream) {
    return decode_impl(out, q, pool, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_q_heads,
                       max_seq_len, scale, partition_tokens, workspace, workspace_bytes, nullptr, nullptr, new_k,
                       new_v, flags, stream);
}

pa_status pa_decode_cascade(void *out, const void *q, const pa_kv_pool *pool, const int32_t *suffix_tables,
                            int32_t max_blocks_per_seq, const int32_t *suffix_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_suffix_len, float scale, int32_t partition_tokens,
                            void *workspace, size_t workspace_bytes, const float *prefix_o,
                            const float *prefix_lse, const void *new_k, const void *new_v, uint32_t flags,
                            cudaStream_t stream) {
    if (num_seqs > 0 && (!prefix_o || !prefix_lse || !aligned16(prefix_o) ||
                         (reinterpret_cast<uintptr_t>(prefix_lse) % 4) != 0))
        return PA_ERR_INVALID_ARG;
    return decode_impl(out, q, pool, suffix_tables, max_blocks_per_seq, suffix_lens, num_seqs, num_q_heads,
                       max_suffix_len, scale, partition_tokens, workspace, workspace_bytes, prefix_o, prefix_lse,
                       new_k, new_v, flags, stream);
}

pa_status pa_copy_blocks(const pa_kv_pool *pool, const int32_t *pairs, int32_t num_pairs, cudaStream_t stream) {
    PoolView view;
    pa_status st = resolve_pool(pool, &view);
    if (st != PA_OK) return st;
    if (num_pairs < 0) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!pairs || num_pairs > (1 << 30)) return PA_ERR_INVALID_ARG;
    return launch_copy_blocks(view, pairs, num_pairs, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_swap_blocks(const pa_kv_pool *pool, void *host, int64_t host_blocks, const int32_t *pairs,
                         int32_t num_pairs, int32_t direction, cudaStream_t stream) {
    PoolView view;
    pa_status st = resolve_pool(pool, &view);
    if (st != PA_OK) return st;
    if (num_pairs < 0 || host_blocks <= 0 || (direction != PA_SWAP_OUT && direction != PA_SWAP_IN))
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!pairs || !host || !aligned16(host) || num_pairs > (1 << 30)) return PA_ERR_INVALID_ARG;
    // The kernel reaches the host buffer through its device mapping: pinned
    // (page-locked, mapped) memory only.
    void *host_dev = nullptr;
    if (cudaHostGetDevicePointer(&host_dev, host, 0) != cudaSuccess || !host_dev) {
        cudaGetLastError();   // clear the sticky-free error this query leaves
        return PA_ERR_INVALID_ARG;
    }
    return launch_swap_blocks(view, host_dev, host_blocks, pairs, num_pairs, direction, stream) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_prefill_chunk(void *out, const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *ctx_lens, int32_t num_seqs,
                           int32_t chunk_len, int32_t num_q_heads, int32_t max_ctx_len, float scale,
                           cudaStream_t stream) {
    PoolView view;
    pa_status st = resolve_pool(pool, &view);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || chunk_len < 0 || num_q_heads <= 0 || max_ctx_len < 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads % view.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!prefill_supported(view.head_dim, num_q_heads / view.num_kv_heads, view.block_size))
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || chunk_len == 0) return PA_OK;
    if (num_seqs > 65535 || (int64_t)num_seqs * chunk_len > (int64_t)INT32_MAX) return PA_ERR_INVALID_ARG;
    if (!out || !q || !block_tables || !ctx_lens || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
    if ((int64_t)max_ctx_len + chunk_len > (int64_t)max_blocks_per_seq * view.block_size) return PA_ERR_INVALID_ARG;
    PrefillArgs a;
    a.out = out;
    a.q = q;
    a.pool = view;
    a.tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.ctx_lens = ctx_lens;
    a.num_seqs = num_seqs;
    a.chunk_len = chunk_len;
    a.num_q_heads = num_q_heads;
    a.max_ctx_len = max_ctx_len;
    a.scale = scale;
    return launch_prefill(a, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_prefix_attention(float *o_part, float *lse, const void *q, const pa_kv_pool *pool,
                              const int32_t *prefix_tables, int32_t max_prefix_blocks, const int32_t *prefix_lens,
                              const int32_t *group_order, int32_t num_groups, int32_t group_size,
                              int32_t num_q_heads, int32_t max_prefix_len,
                              float scale, cudaStream_t stream) {
    PoolView view;
    pa_status st = resolve_pool(pool, &view);
    if (st != PA_OK) return st;
    if (num_groups < 0 || group_size < 0 || num_q_heads <= 0 || max_prefix_len < 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads % view.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!prefill_supported(view.head_dim, num_q_heads / view.num_kv_heads, view.block_size))
        return PA_ERR_UNSUPPORTED;
    if (num_groups == 0 || group_size == 0) return PA_OK;
    if (!o_part || !lse || !q || !prefix_tables || !prefix_lens || max_prefix_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!aligned16(o_part) || (reinterpret_cast<uintptr_t>(lse) % 4) != 0 || !aligned16(q)) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
    if ((int64_t)max_prefix_len > (int64_t)max_prefix_blocks * view.block_size) return PA_ERR_INVALID_ARG;
    // grid z is the group; the row coordinate group * group_size + j is an int32
    if (num_groups > 65535 || (int64_t)num_groups * group_size > (int64_t)INT32_MAX) return PA_ERR_INVALID_ARG;
    PrefillArgs a;
    a.out = nullptr;
    a.q = q;
    a.pool = view;
    a.tables = prefix_tables;
    a.max_blocks = max_prefix_blocks;
    a.ctx_lens = prefix_lens;
    a.num_seqs = num_groups;
    a.chunk_len = group_size;
    a.num_q_heads = num_q_heads;
    a.max_ctx_len = max_prefix_len;
    a.scale = scale;
    a.causal = false;
    a.o_part = o_part;
    a.lse = lse;
    a.order = group_order;
    return launch_prefill(a, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_grouped(void *out, const void *q, const pa_kv_pool *pool, const int32_t *prefix_tables,
                            int32_t max_prefix_blocks, const int32_t *prefix_lens, const int32_t *group_order,
                            const int32_t *suffix_tables, int32_t max_suffix_blocks, const int32_t *suffix_lens,
                            int32_t num_groups, int32_t group_size, int32_t num_q_heads, int32_t max_prefix_len,
                            int32_t max_suffix_len, float scale, const void *new_k, const void *new_v,
                            uint32_t flags, cudaStream_t stream) {
    PoolView view;
    pa_status st = resolve_pool(pool, &view);
    if (st != PA_OK) return st;
    if (num_groups < 0 || group_size < 0 || num_q_heads <= 0 || max_prefix_len < 0 || max_suffix_len < 0)
        return PA_ERR_INVALID_ARG;
    if (flags & ~PA_DECODE_EARLY_METADATA) return PA_ERR_INVALID_ARG;
    if (num_q_heads % view.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int group = num_q_heads / view.num_kv_heads;
    if (!prefill_supported(view.head_dim, group, view.block_size)) return PA_ERR_UNSUPPORTED;
    // one 128-key tile holds the suffix blocks of every member of an M-tile
    const int64_t members = std::min<int64_t>(group_size, 128 / group);
    const int64_t nb = ceil_div(max_suffix_len, view.block_size);
    if (members * nb * view.block_size > 128) return PA_ERR_UNSUPPORTED;
    if (num_groups == 0 || group_size == 0) return PA_OK;
    if (!out || !q || !prefix_tables || !prefix_lens || max_prefix_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!suffix_tables || !suffix_lens || max_suffix_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q)) return PA_ERR_INVALID_ARG;
    if ((new_k == nullptr) != (new_v == nullptr)) return PA_ERR_INVALID_ARG;
    if (new_k && (!aligned16(new_k) || !aligned16(new_v))) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
    if ((int64_t)max_prefix_len > (int64_t)max_prefix_blocks * view.block_size) return PA_ERR_INVALID_ARG;
    if ((int64_t)max_suffix_len > (int64_t)max_suffix_blocks * view.block_size) return PA_ERR_INVALID_ARG;
    if (num_groups > 65535 || (int64_t)num_groups * group_size > (int64_t)INT32_MAX) return PA_ERR_INVALID_ARG;
    PrefillArgs a;
    a.out = out;
    a.q = q;
    a.pool = view;
    a.tables = prefix_tables;
    a.max_blocks = max_prefix_blocks;
    a.ctx_lens = prefix_lens;
    a.num_seqs = num_groups;
    a.chunk_len = group_size;
    a.num_q_heads = num_q_heads;
    a.max_ctx_len = max_prefix_len;
    a.scale = scale;
    a.causal = false;
    a.order = group_order;
    a.sfx_tables = suffix_tables;
    a.sfx_max_blocks = max_suffix_blocks;
    a.sfx_lens = suffix_lens;
    a.sfx_nb = (int32_t)nb;
    a.max_sfx_len = max_suffix_len;
    a.new_k = new_k;
    a.new_v = new_v;
    a.early_meta = (flags & PA_DECODE_EARLY_METADATA) != 0;
    return launch_prefill(a, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_check_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
    if (limit_ns < 1000u || limit_ns > 1000000000u) return PA_ERR_INVALID_ARG;
    return launch_wait_timeout(limit_ns, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_set_stream_k_ctas(int32_t ctas) {
    if (ctas < 0) return PA_ERR_INVALID_ARG;
    g_stream_k_ctas.store(ctas, std::memory_order_relaxed);
    return PA_OK;
}

pa_status pa_set_prefill_ctas(int32_t ctas) {
    if (ctas < 0) return PA_ERR_INVALID_ARG;
    set_prefill_ctas(ctas);
    return PA_OK;
}

pa_status pa_get_device_error(uint32_t *err_out, int32_t clear, cudaStream_t stream) {
    if (!err_out) return PA_ERR_INVALID_ARG;
    unsigned int *word = device_error_word();
    if (!word) return PA_ERR_CUDA;
    uint32_t value = 0;
    if (cudaMemcpyAsync(&value, word, sizeof(value), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
    if (clear && value) {
        if (cudaMemsetAsync(word, 0, sizeof(value), stream) != cudaSuccess) return PA_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    *err_out = value;
    return value ? PA_ERR_DEVICE : PA_OK;
}

pa_status pa_block_layout(int64_t tokens, int32_t block_size, int64_t *blocks, int64_t *unused) {
    if (tokens < 0 || block_size <= 0 || !blocks || !unused) return PA_ERR_INVALID_ARG;
    const int64_t n = ceil_div(tokens, block_size);
    *blocks = n;
    *unused = n * block_size - tokens;
    return PA_OK;
}

pa_status pa_slot_mapping(int64_t *slots, const int32_t *tables, int32_t num_seqs, int32_t max_blocks,
                          const int32_t *seq_idx, const int64_t *positions, int64_t n, int32_t block_size,
                          int64_t num_blocks) {
    if (n < 0 || num_seqs < 0 || max_blocks <= 0 || block_size <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (n == 0) return PA_OK;
    if (!slots || !tables || !seq_idx || !positions) return PA_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t s = seq_idx[i];
        const int64_t t = positions[i];
        if (s < 0 || s >= num_seqs || t < 0 || t / block_size >= max_blocks) return PA_ERR_INVALID_ARG;
        const int32_t phys = tables[(int64_t)s * max_blocks + t / block_size];
        if (phys < 0 || phys >= num_blocks) return PA_ERR_INVALID_ARG;
        slots[i] = (int64_t)phys * block_size + t % block_size;
    }
    return PA_OK;
}

}  // extern "C"
