// pa_decode_host.cpp -- one decode step from host buffers.
//
// A serving loop that keeps a step's inputs in host memory (the new tokens'
// q, K and V, the tables and lengths it just updated) would otherwise issue a
// copy per input, the decode call and a copy back, each through its own
// binding.  pa_decode_host does all of it in one call: the inputs go into a
// caller-provided device staging buffer with one asynchronous copy each, the
// decode runs on them (storing each sequence's new token itself, as
// pa_decode_ex does), and the output comes back to host memory, all queued on
// the caller's stream.  The KV pool stays device-resident.
#include <cstdint>
#include <cuda_runtime_api.h>

#include "pa.h"

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct StagingLayout {
    size_t q, out, new_k, new_v, tables, lens, total;
};

bool staging_layout(const pa_kv_pool *pool, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks,
                    StagingLayout *l) {
    if (!pool || num_seqs < 0 || num_q_heads <= 0 || max_blocks <= 0 || pool->head_dim <= 0 ||
        pool->num_kv_heads <= 0)
        return false;
    const size_t B = (size_t)num_seqs, d = (size_t)pool->head_dim;
    const size_t q_bytes = round_up(B * (size_t)num_q_heads * d * 2);
    const size_t kv_bytes = round_up(B * (size_t)pool->num_kv_heads * d * 2);
    l->q = 0;
    l->out = l->q + q_bytes;
    l->new_k = l->out + q_bytes;
    l->new_v = l->new_k + kv_bytes;
    l->tables = l->new_v + kv_bytes;
    l->lens = l->tables + round_up(B * (size_t)max_blocks * sizeof(int32_t));
    l->total = l->lens + round_up(B * sizeof(int32_t));
    return true;
}

}  // namespace

extern "C" {

size_t pa_decode_host_staging_size(const pa_kv_pool *pool, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t max_blocks_per_seq) {
    StagingLayout l;
    return staging_layout(pool, num_seqs, num_q_heads, max_blocks_per_seq, &l) ? l.total : 0;
}

pa_status pa_decode_host(void *out_host, const void *q_host, const pa_kv_pool *pool, const int32_t *tables_host,
                         int32_t max_blocks_per_seq, const int32_t *seq_lens_host, int32_t num_seqs,
                         int32_t num_q_heads, int32_t max_seq_len, float scale, int32_t partition_tokens,
                         const void *new_k_host, const void *new_v_host, uint32_t flags, void *staging,
                         size_t staging_bytes, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    StagingLayout l;
    if (!staging_layout(pool, num_seqs, num_q_heads, max_blocks_per_seq, &l)) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out_host || !q_host || !tables_host || !seq_lens_host) return PA_ERR_INVALID_ARG;
    if ((new_k_host == nullptr) != (new_v_host == nullptr)) return PA_ERR_INVALID_ARG;
    if (!staging || staging_bytes < l.total || (reinterpret_cast<uintptr_t>(staging) % kAlign) != 0)
        return PA_ERR_WORKSPACE;
    // The tables and lengths are written by the copies just before the decode
    // kernel, so the early-metadata read is never allowed here.
    flags &= ~PA_DECODE_EARLY_METADATA;
    char *st = static_cast<char *>(staging);
    const size_t B = (size_t)num_seqs, d = (size_t)pool->head_dim;
    const size_t q_bytes = B * (size_t)num_q_heads * d * 2, kv_bytes = B * (size_t)pool->num_kv_heads * d * 2;
    auto h2d = [&](size_t off, const void *src, size_t n) {
        return cudaMemcpyAsync(st + off, src, n, cudaMemcpyHostToDevice, stream) == cudaSuccess;
    };
    if (!h2d(l.q, q_host, q_bytes) || !h2d(l.tables, tables_host, B * (size_t)max_blocks_per_seq * 4) ||
        !h2d(l.lens, seq_lens_host, B * 4))
        return PA_ERR_CUDA;
    const void *nk = nullptr, *nv = nullptr;
    if (new_k_host) {
        if (!h2d(l.new_k, new_k_host, kv_bytes) || !h2d(l.new_v, new_v_host, kv_bytes)) return PA_ERR_CUDA;
        nk = st + l.new_k;
        nv = st + l.new_v;
    }
    const pa_status s = pa_decode_ex(st + l.out, st + l.q, pool, reinterpret_cast<const int32_t *>(st + l.tables),
                                     max_blocks_per_seq, reinterpret_cast<const int32_t *>(st + l.lens), num_seqs,
                                     num_q_heads, max_seq_len, scale, partition_tokens, workspace, workspace_bytes,
                                     nk, nv, flags, stream);
    if (s != PA_OK) return s;
    return cudaMemcpyAsync(out_host, st + l.out, q_bytes, cudaMemcpyDeviceToHost, stream) == cudaSuccess ? PA_OK
                                                                                                          : PA_ERR_CUDA;
}

}  // extern "C"
