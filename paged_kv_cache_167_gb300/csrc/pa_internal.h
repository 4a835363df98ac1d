// pa_internal.h -- host-side interface between the C ABI layer (pa_api.cpp)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>

#include "pa.h"

namespace pa {

// A validated, stride-resolved view of one layer of the block pool.
struct PoolView {
    const void *base;
    int64_t num_blocks;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t head_dim;
    int64_t block_stride;  // elements
    int64_t kv_stride;     // elements
};

// Device address of the current device's error word (set up once per device);
// nullptr if the CUDA runtime failed.
unsigned int *device_error_word();
cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

// Number of SMs of the current device (cached per device); 0 on failure.
int device_sm_count();

// The driver's cuTensorMapEncodeTiled, resolved once through the runtime;
// nullptr if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Tensor map of the K (kv = 0) or V (kv = 1) half of a pool layer as (d within
// a 64-wide half, slot, half of d, kv-head, block): one box is `box_rows`
// slots (the whole block when box_rows = block_size) of one (block, K|V,
// kv-head) slab, laid out [half][slot][64] with 128-byte swizzle (head_dim 64
// or 128).  A block coordinate of num_blocks reads as zeros.
cudaError_t encode_pool_block_map(CUtensorMap *map, const PoolView &pool, int kv, int box_rows);

// ---- slot writer and block copies (pa_cache.cu) ---------------------------
cudaError_t launch_reshape_and_cache(const PoolView &pool, const void *k, const void *v,
                                     const int64_t *slots, int64_t num_tokens, cudaStream_t stream);
cudaError_t launch_append_last(const PoolView &pool, const int32_t *tables, int32_t max_blocks,
                               const int32_t *seq_lens, int32_t num_seqs, int32_t max_len, const void *k,
                               const void *v, cudaStream_t stream);
cudaError_t launch_copy_blocks(const PoolView &pool, const int32_t *pairs, int32_t num_pairs,
                               cudaStream_t stream);
// host_dev: the device address of the pinned host buffer
cudaError_t launch_swap_blocks(const PoolView &pool, void *host_dev, int64_t host_blocks, const int32_t *pairs,
                               int32_t num_pairs, int32_t direction, cudaStream_t stream);

// ---- decode (pa_decode_*.cu) -----------------------------------------------
struct DecodeArgs {
    void *out;
    const void *q;
    PoolView pool;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t max_seq_len;
    float scale;
    int32_t partition_tokens;  // resolved (> 0, multiple of block_size)
    int32_t num_partitions;    // ceil(max_seq_len / partition_tokens), >= 1
    float *ws_o;               // split: [B][Hq][P][d] when num_partitions > 1; stream-K: [2C][G][d]
    float *ws_ml;              // split: [B][Hq][P][2]; stream-K: [2C][G][2]
    bool stream_k;             // persistent balanced schedule (automatic plan)
    int32_t num_ctas;          // stream-K grid size C
    bool early_meta = false;   // stream-K: read lengths and tables before the previous kernel completes
    const void *new_k = nullptr;   // stream-K: last token's K/V per sequence, stored before attending
    const void *new_v = nullptr;
    const float *pre_o = nullptr;      // cascade: prefix partial [B][Hq][d] fp32 (normalised)
    const float *pre_lse = nullptr;    // and its log-sum-exp [B][Hq]
};

// Tokens per pipeline stage of the decode kernel for a block size (the
// granularity a partition length is rounded to).
int decode_stage_tokens(int block_size);
bool decode_supported(int head_dim, int group, int block_size);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);

// ---- prefill (pa_prefill.cu) -----------------------------------------------
struct PrefillArgs {
    void *out;
    const void *q;
    PoolView pool;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *ctx_lens;
    int32_t num_seqs;
    int32_t chunk_len;
    int32_t num_q_heads;
    int32_t max_ctx_len;
    float scale;
    bool causal = true;        // false: every query sees keys 0 .. ctx_lens[s] - 1
    float *o_part = nullptr;   // non-null: fp32 normalised output + lse instead of out
    float *lse = nullptr;
    const int32_t *order = nullptr;   // non-null: sequences in this order (a permutation)
    // grouped decode: members' suffix tables and lengths (nullptr: none)
    const int32_t *sfx_tables = nullptr;
    int32_t sfx_max_blocks = 0;
    const int32_t *sfx_lens = nullptr;
    int32_t sfx_nb = 0;        // suffix-tile blocks per member
    int32_t max_sfx_len = 0;
    const void *new_k = nullptr;
    const void *new_v = nullptr;
    bool early_meta = false;   // order, ctx_lens and tables are not written by the kernel before
};
bool prefill_supported(int head_dim, int group, int block_size);
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream);
void set_prefill_ctas(int32_t ctas);   // 0: one CTA per SM

}  // namespace pa
