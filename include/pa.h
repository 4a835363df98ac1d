/*
 * pa.h -- C ABI of the paged KV-cache attention library (libpa.so).
 *
 * A KV cache held in fixed-size physical blocks, read through per-sequence
 * block tables, on one GB300 (sm_103a).  Every device call is a hand-written
 * CUDA kernel launched asynchronously on the caller's stream.
 *
 * Conventions for every call below:
 *  - Device pointers are allocated and owned by the caller.  The library
 *    never allocates, frees or synchronises device memory, except where a
 *    function says so (pa_get_device_error synchronises its stream).
 *  - Arguments are validated on the host before anything is launched; a
 *    non-PA_OK status means nothing was launched.  A CUDA launch failure is
 *    reported as PA_ERR_CUDA.
 *  - Values that only the device can see (table entries, slots, sequence
 *    lengths, fork pairs) are bounds-checked inside the kernels.  An
 *    out-of-range value is never dereferenced: the kernel records a bit in a
 *    per-device error word (PA_DEVERR_*) and leaves the affected output
 *    undefined.  Read the word with pa_get_device_error.
 *  - Tensors are bf16, row-major, densely packed unless a stride is given,
 *    and 16-byte aligned.
 *  - Devices 0 .. 63 are supported: the library caches per-device state (the
 *    error word's and the allocation-free scratch array's addresses, the SM
 *    count) for those indices, and every device call made while a device
 *    with a higher index is current returns PA_ERR_CUDA.
 *
 * Sources (page, section) for the operations:
 *  [P1] how-pagedattention-works (aiinfrainterviews.com)
 *  [P2] attn-paged-attention-mcq-hard (zenaique.com)
 *  [P3] auto-20261007-1900-en (lihaoran.work)
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, bad stride   */
    PA_ERR_UNSUPPORTED = 2,   /* head_dim, block_size, group size or dtype not built      */
    PA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than the *_workspace_size   */
    PA_ERR_CUDA = 4,          /* the CUDA runtime reported an error                       */
    PA_ERR_DEVICE = 5,        /* pa_get_device_error found a non-zero device error word   */
    PA_ERR_NO_BLOCKS = 6,     /* block manager: the pool has no free block left           */
    PA_ERR_NOT_FOUND = 7,     /* block manager: unknown sequence id                       */
    PA_ERR_SWAPPED = 8        /* block manager: the sequence's blocks are on the host     */
} pa_status;

/* Bits of the per-device error word written by the kernels. */
#define PA_DEVERR_BLOCK_ID 0x1u /* a table entry or fork pair outside [0, num_blocks)      */
#define PA_DEVERR_SLOT     0x2u /* a slot >= num_blocks * block_size                       */
#define PA_DEVERR_SEQ_LEN  0x4u /* a length < 0, beyond the table width or the host bound  */
#define PA_DEVERR_TIMEOUT  0x8u /* a bounded wait on a shared-memory barrier gave up       */
#define PA_DEVERR_ORDER   0x10u /* a group order entry outside [0, num_groups)              */

typedef enum { PA_DTYPE_BF16 = 0 } pa_dtype;

/*
 * One layer's view of the physical block pool.  [P1] "A strong answer": the
 * cache is carved into equal blocks of block_size token slots per layer;
 * [P2] conceptual block-lookup listing: pool shaped
 * [num_blocks, 2, num_layers, num_kv_heads, block_size, d_head].
 *
 * Element (blk, kv, h, off, i) -- kv 0 for K, 1 for V -- is at element offset
 *     blk*block_stride + kv*kv_stride + (h*block_size + off)*head_dim + i
 * from base.  block_stride = 0 means 2*Hkv*b*d and kv_stride = 0 means
 * Hkv*b*d, i.e. the dense one-layer layout [NB][2][Hkv][b][d].  For the
 * layered layout [NB][2][L][Hkv][b][d] at layer l, point base at layer l's
 * first slab and set block_stride = 2*L*Hkv*b*d, kv_stride = L*Hkv*b*d.
 * Every (blk, kv, h) slab of block_size*head_dim elements is contiguous.
 * base and both strides (in bytes) must be multiples of 16.
 */
typedef struct {
    void *base;           /* device memory, owned by the caller                 */
    int64_t num_blocks;   /* NB: valid physical block ids are [0, NB)           */
    int32_t num_kv_heads; /* Hkv                                                */
    int32_t block_size;   /* b: token slots per block                           */
    int32_t head_dim;     /* d                                                  */
    int32_t dtype;        /* PA_DTYPE_BF16                                      */
    int64_t block_stride; /* elements; 0 = dense                                */
    int64_t kv_stride;    /* elements; 0 = dense                                */
} pa_kv_pool;

/* Human-readable name of a status.  Never returns NULL. */
const char *pa_status_string(pa_status status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t pa_version(void);

/*
 * Slot writer.  [P1] "A strong answer": a sequence's cache grows by one token
 * each decode step, into the next free slot of its last block.
 *   k, v          device, [num_tokens][Hkv][d] bf16 (the new tokens' K and V)
 *   slot_mapping  device, [num_tokens] int64; slot = phys*block_size + offset
 *                 (the linear form of [P3]'s (table[t//b], t%b)); a negative
 *                 slot is padding and is skipped; slot >= NB*b raises
 *                 PA_DEVERR_SLOT and is skipped
 * Writes pool[slot/b][0][h][slot%b][:] = k[n][h][:] and the same for V,
 * bit-exactly.  Two tokens with the same slot race (the result is one of them).
 */
pa_status pa_reshape_and_cache(const pa_kv_pool *pool, const void *k, const void *v,
                               const int64_t *slot_mapping, int64_t num_tokens,
                               cudaStream_t stream);

/*
 * Bytes of device workspace pa_decode needs for these shapes.  With an
 * explicit partition_tokens it is 0 when one partition covers max_seq_len;
 * with partition_tokens = 0 (the balanced schedule) it is a few MB at most:
 * two fp32 partial records of (num_q_heads / Hkv) x (head_dim + 2) per CTA of
 * a grid sized from the current device's SM count.
 */
size_t pa_decode_workspace_size(const pa_kv_pool *pool, int32_t num_seqs, int32_t num_q_heads,
                                int32_t max_seq_len, int32_t partition_tokens);

/* The partition length pa_decode will use for these shapes (a multiple of
 * block_size); 0 when partition_tokens = 0 selects the balanced schedule;
 * -1 if the shapes are invalid. */
int32_t pa_decode_partition_tokens(const pa_kv_pool *pool, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t max_seq_len, int32_t partition_tokens);

/*
 * Paged GQA decode attention.  [P1] "A strong answer": the kernel takes the
 * block table and reads each query's K/V from the physical blocks it names;
 * [P2] conceptual block-lookup listing: position t of sequence s is at
 * (block_tables[s][t // b], t % b), and attention over the gathered rows is
 * ordinary scaled dot-product attention; [P3] "A block table maps logical
 * order to physical storage".
 *
 *   out          device, [num_seqs][num_q_heads][d] bf16 (written)
 *   q            device, [num_seqs][num_q_heads][d] bf16
 *   block_tables device, [num_seqs][max_blocks_per_seq] int32 physical ids
 *   seq_lens     device, [num_seqs] int32, tokens to attend (0 gives zeros)
 *   max_seq_len  host upper bound on every seq_lens[s] (sizes the grid)
 *   scale        softmax scale, usually 1/sqrt(d)
 *   partition_tokens  0 (recommended): the balanced schedule -- a persistent
 *                grid in which every CTA takes an equal contiguous share of
 *                all (sequence, kv-head, 16-token stage) work, units cut
 *                between two CTAs being merged by a second kernel.  Else a
 *                positive multiple of block_size: split-context partitions
 *                of that many tokens, grid (partition, kv-head, sequence),
 *                merged by a reduce kernel when more than one covers
 *                max_seq_len.
 *   workspace    device scratch of pa_decode_workspace_size bytes (may be
 *                NULL when that size is 0); its contents are overwritten
 *
 * q-head h reads kv-head h / (num_q_heads / Hkv).  All query heads of a KV
 * group are served from one staged copy of each block.  Accumulation is fp32;
 * out is rounded to bf16 (round to nearest even).
 * Supported: head_dim 64 or 128; block_size 4, 8, 16, 32 or 64; group size
 * num_q_heads / Hkv of 1, 2, 4 or 8.
 */
pa_status pa_decode(void *out, const void *q, const pa_kv_pool *pool,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t max_seq_len, float scale, int32_t partition_tokens,
                    void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * pa_decode with the decode step's slot write and option flags; pa_decode is
 * pa_decode_ex with new_k = new_v = NULL and flags = 0.
 *
 * new_k, new_v (device, 16-B aligned, both NULL or both set): [num_seqs][Hkv]
 * [head_dim] bf16, the K and V of the token each sequence is decoding.  For
 * every sequence with 0 < seq_lens[s] <= its bound, the call first stores them
 * at position seq_lens[s] - 1 (slot block_tables[s][(L-1)/b] * b + (L-1) % b),
 * exactly what pa_reshape_and_cache would store there, and attention then
 * includes them.  With the automatic plan the decode kernel itself stores each
 * token just before it fetches the block holding it, which saves the slot
 * writer's launch; with an explicit partition_tokens a small kernel stores them
 * first.  An out-of-range length or table entry writes nothing and raises the
 * same error bits as decode.  ([P1] "A strong answer": each decode step adds
 * one token's K/V to the sequence's last block.)
 *
 * PA_DECODE_EARLY_METADATA: the caller promises that seq_lens and
 * block_tables are not written by the kernel this call immediately follows
 * in `stream` (host-to-device copies, or kernels before that one, are fine).
 * The decode kernel is launched with programmatic stream serialisation
 * either way; with this flag it reads the lengths and table entries and
 * plans its schedule while that previous kernel is still running, and only
 * q, the pool and the workspace wait for it to finish, which takes the
 * lengths -> schedule -> table chain off the call's start; it also brings
 * the first blocks each CTA will read into L2 (a prefetch hint, which reads
 * whatever that kernel writes there correctly).  It applies to the automatic
 * plan (partition_tokens = 0) and is otherwise ignored; results are
 * identical with and without it.  (The pool may be written by that previous
 * kernel: the slot writer is the usual one.)
 * Unknown flag bits give PA_ERR_INVALID_ARG.
 */
#define PA_DECODE_EARLY_METADATA 0x1u
pa_status pa_decode_ex(void *out, const void *q, const pa_kv_pool *pool,
                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                       const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t max_seq_len, float scale, int32_t partition_tokens,
                       void *workspace, size_t workspace_bytes, const void *new_k,
                       const void *new_v, uint32_t flags, cudaStream_t stream);

/*
 * pa_decode without a caller workspace, for callers that cannot allocate
 * device memory: e.g. a plugin that its host framework hands only input and
 * output buffers (the framework's allocator owns all device memory), or a
 * serving loop that must not call cudaMalloc (which can synchronise the
 * device) once it is running.  The pages have no counterpart to this call;
 * it is a library convenience.
 *
 * Same arguments, semantics and results as pa_decode, minus the workspace.
 * The split-context partials go to a fixed 8 MiB array in the library's own
 * device memory (a file-scope __device__ array that every GPU loading the
 * library holds until the process exits).  Shapes whose
 * pa_decode_workspace_size exceeds 8 MiB return PA_ERR_WORKSPACE and launch
 * nothing.  The call allocates and frees nothing.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture begins.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents (nothing in it needs to start at zero).  Calls whose kernels
 *    overlap on the GPU, e.g. on two streams, race on it: serialise them.
 *  - Called while a device with index 64 or more is current, it returns
 *    PA_ERR_CUDA and launches nothing.
 */
pa_status pa_decode_noalloc(void *out, const void *q, const pa_kv_pool *pool,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t max_seq_len, float scale, int32_t partition_tokens,
                            cudaStream_t stream);

/*
 * One decode step from host buffers: copies q, the tables, the lengths and
 * (optionally) the new tokens' K/V from host memory into `staging`, runs
 * pa_decode_ex on them, and copies the output back to `out_host`, all queued
 * on `stream` (one asynchronous copy per input).  The pool stays on the device.
 * The caller synchronises the stream before reading out_host; host buffers
 * should be page-locked (pinned) for the copies to run asynchronously.
 *   out_host, q_host     host, [num_seqs][num_q_heads][d] bf16
 *   tables_host          host, [num_seqs][max_blocks_per_seq] int32
 *   seq_lens_host        host, [num_seqs] int32
 *   new_k_host, new_v_host  host, [num_seqs][Hkv][d] bf16, both NULL or both set
 *                        (stored at each sequence's last position, as pa_decode_ex)
 *   staging              device, 256-byte aligned, at least
 *                        pa_decode_host_staging_size(...) bytes (else PA_ERR_WORKSPACE);
 *                        owned by the caller, not read by the step until the
 *                        copies into it have landed
 *   workspace            as pa_decode
 * flags as pa_decode_ex, except that PA_DECODE_EARLY_METADATA is ignored: the
 * tables and lengths are written by the copies just before the decode.  The
 * pages have no counterpart to this call.
 */
size_t pa_decode_host_staging_size(const pa_kv_pool *pool, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t max_blocks_per_seq);
pa_status pa_decode_host(void *out_host, const void *q_host, const pa_kv_pool *pool,
                         const int32_t *tables_host, int32_t max_blocks_per_seq,
                         const int32_t *seq_lens_host, int32_t num_seqs, int32_t num_q_heads,
                         int32_t max_seq_len, float scale, int32_t partition_tokens,
                         const void *new_k_host, const void *new_v_host, uint32_t flags, void *staging,
                         size_t staging_bytes, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * Copy-on-write block copies.  [P1] feature table, beam-search row: forks
 * share blocks and only the block that diverges is copied; [P2] interviewer
 * follow-up on beam search: a fresh block receives the diverging block's
 * content.
 *   pairs  device, [num_pairs][2] int32 (src, dst)
 * For each pair, every K and V slot of every kv-head of block src (in this
 * layer's view) is copied to block dst, bit-exactly.  An id outside
 * [0, num_blocks) raises PA_DEVERR_BLOCK_ID and that pair is skipped.  Pairs
 * are copied concurrently: a dst that is also some pair's src, or a repeated
 * dst, gives an unspecified result.
 */
/*
 * Block-granular swap between one layer of the pool and pinned host memory.
 * [P1] feature table, preemption row: under memory pressure a sequence's
 * blocks are swapped to host memory at block granularity; [P1] "What
 * interviewers probe next": when the pool runs dry mid-decode, the preempted
 * sequence's blocks go to pinned host memory.
 *   host         host memory the GPU can address -- pinned and mapped
 *                (cudaHostAlloc, or cudaHostRegister with
 *                cudaHostRegisterMapped), or any host memory where the GPU
 *                walks the host's page tables (NVLink-C2C systems) --
 *                16-byte aligned, holding host_blocks
 *                blocks as [host_blocks][2][Hkv][b][d] bf16: one block's K and
 *                V slabs for every kv-head (64 KiB at Hkv 8, b 16, d 128)
 *   pairs        device, [num_pairs][2] int32 (device block, host block)
 *   direction    PA_SWAP_OUT: host[hb] = pool[dev]; PA_SWAP_IN: pool[dev] = host[hb]
 * One kernel reads or writes the host buffer directly through its device
 * mapping (no staging copy, no per-block copy call), so it can run on its own
 * stream beside compute.  A host pointer the GPU cannot address
 * (cudaHostGetDevicePointer fails) gives PA_ERR_INVALID_ARG and nothing is
 * launched.  An id out of range raises
 * PA_DEVERR_BLOCK_ID and that pair is skipped; repeated destinations give an
 * unspecified result.  Bit-exact copies.
 */
#define PA_SWAP_OUT 0
#define PA_SWAP_IN 1
pa_status pa_swap_blocks(const pa_kv_pool *pool, void *host, int64_t host_blocks, const int32_t *pairs,
                         int32_t num_pairs, int32_t direction, cudaStream_t stream);

pa_status pa_copy_blocks(const pa_kv_pool *pool, const int32_t *pairs, int32_t num_pairs,
                         cudaStream_t stream);

/*
 * Chunked causal prefill against a paged context.  [P3] "A block table maps
 * logical order to physical storage": paging changes only where K/V live, so
 * each query still attends its whole visible (causal) history.
 *   out, q       device, [num_seqs][chunk_len][num_q_heads][d] bf16
 *   ctx_lens     device, [num_seqs] int32: tokens cached before the chunk
 *   max_ctx_len  host upper bound on every ctx_lens[s]
 *   scale        softmax scale, finite and > 0 (usually 1/sqrt(d)); else
 *                PA_ERR_INVALID_ARG
 * Query j of sequence s sits at position ctx_lens[s] + j and attends keys
 * 0 .. ctx_lens[s] + j.  The chunk's own K/V must already be in the pool
 * (pa_reshape_and_cache).  QK^T and PV run on the tcgen05 tensor cores with
 * fp32 accumulation in tensor memory.
 * Supported: head_dim 128, block_size 8, 16, 32 or 64, group size 1, 2, 4 or 8;
 * at most 65,535 sequences.
 */
pa_status pa_prefill_chunk(void *out, const void *q, const pa_kv_pool *pool,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *ctx_lens, int32_t num_seqs, int32_t chunk_len,
                           int32_t num_q_heads, int32_t max_ctx_len, float scale,
                           cudaStream_t stream);

/*
 * Cascade decode, pass 1: attention of every decode query of a group of
 * sequences over the prefix the group shares, reading the prefix's K/V once
 * for the whole group.  [P1] shared-system-prompt paragraph: the shared
 * prompt's blocks are held once and every sharer's table points at them;
 * [P3] "Shared prefixes need matching computation".  The pages share the
 * memory; reading it once is this library's design: attention over keys
 * A u B is the log-sum-exp merge of attention over A and over B.
 *   o_part        device, [num_groups][group_size][num_q_heads][d] fp32, 16-B
 *                 aligned: each row's softmax-weighted V over the prefix
 *   lse           device, [num_groups][group_size][num_q_heads] fp32: the row's
 *                 log(sum_t exp(scale * q.K_t)) over the prefix (natural log;
 *                 -inf and o_part 0 when the prefix is empty)
 *   q             device, [num_groups][group_size][num_q_heads][d] bf16: the
 *                 decode batch's q, its sequences ordered group by group
 *   prefix_tables device, [num_groups][max_prefix_blocks] int32: the group's
 *                 shared blocks
 *   prefix_lens   device, [num_groups] int32, each in [0, max_prefix_len]
 *   group_order   device, [num_groups] int32, a permutation of the groups, or
 *                 NULL: the order in which the groups' units are dealt to the
 *                 persistent CTAs (in rounds of alternating direction, so with
 *                 the longest prefix first a CTA that draws a long unit draws
 *                 a short one next; pa_cascade_plan writes that order).  It
 *                 changes no result.  An entry outside [0, num_groups) raises
 *                 PA_DEVERR_ORDER and that slot takes its own index instead
 *                 (some group is then done twice and another not at all); a
 *                 repeated entry is not detected and leaves the rows of a
 *                 missing group unwritten.
 *   max_prefix_len host bound, <= max_prefix_blocks * block_size
 *   scale         as pa_prefill_chunk
 * Every query of group i attends all prefix_lens[i] keys (no causal mask: the
 * prefix precedes every query).  Runs the pa_prefill_chunk kernel (tcgen05,
 * fp32 accumulation) without its mask; same supported shapes.  At most 65,535
 * groups.  An out-of-range length or table entry raises the device error bits
 * as prefill does.
 */
pa_status pa_prefix_attention(float *o_part, float *lse, const void *q, const pa_kv_pool *pool,
                              const int32_t *prefix_tables, int32_t max_prefix_blocks,
                              const int32_t *prefix_lens, const int32_t *group_order,
                              int32_t num_groups, int32_t group_size,
                              int32_t num_q_heads, int32_t max_prefix_len, float scale,
                              cudaStream_t stream);

/*
 * Host planning of a cascade decode over groups of group_size consecutive
 * sequences (all arrays host memory).  For each group the prefix is the
 * longest run of leading table entries that every member holds in common,
 * in whole blocks, and at most floor((min length - 1) / block_size) blocks so
 * that every member keeps at least one token of its own (the token being
 * decoded is then always in the suffix).
 *   tables         [num_seqs][max_blocks] int32; seq_lens [num_seqs]
 *   prefix_tables  out [num_seqs / group_size][max_blocks]: the shared ids, then -1
 *   prefix_lens    out [num_seqs / group_size]: shared blocks * block_size
 *   group_order    out [num_seqs / group_size] or NULL: the groups by prefix
 *                  length, longest first (ties in index order), for
 *                  pa_prefix_attention
 *   suffix_tables  out [num_seqs][max_blocks]: each row's ids after the prefix, then -1
 *   suffix_lens    out [num_seqs]: seq_lens[s] - the group's prefix length
 * PA_ERR_INVALID_ARG when num_seqs is not a multiple of group_size, a size is
 * not positive, or a length is negative or above max_blocks * block_size.
 */
pa_status pa_cascade_plan(const int32_t *tables, int32_t max_blocks, const int32_t *seq_lens,
                          int32_t num_seqs, int32_t group_size, int32_t block_size,
                          int32_t *prefix_tables, int32_t *prefix_lens, int32_t *group_order,
                          int32_t *suffix_tables, int32_t *suffix_lens);

/*
 * Cascade decode, pass 2: pa_decode_ex over each sequence's private suffix,
 * with pass 1's (prefix_o, prefix_lse) folded into every output row as one
 * more partial (weight exp(lse - M) against the suffix's own sum).  The
 * result is attention over prefix and suffix together.
 *   suffix_tables  device, [num_seqs][max_blocks_per_seq] int32: the blocks
 *                  after the shared prefix (the prefix must be whole blocks,
 *                  so suffix position 0 is offset 0 of suffix_tables[s][0])
 *   suffix_lens    device, [num_seqs] int32: tokens after the prefix (0: the
 *                  output is the prefix term alone)
 *   max_suffix_len host bound on every suffix_lens[s]
 *   prefix_o, prefix_lse  device, [num_seqs][num_q_heads]([d]) fp32 as written
 *                  by pa_prefix_attention (prefix_o 16-B aligned); both required
 *   new_k, new_v, flags   as pa_decode_ex, positions counted in the suffix
 * All other arguments, the workspace and the errors as pa_decode_ex.  The same
 * scale must be passed to both passes.
 */
pa_status pa_decode_cascade(void *out, const void *q, const pa_kv_pool *pool,
                            const int32_t *suffix_tables, int32_t max_blocks_per_seq,
                            const int32_t *suffix_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t max_suffix_len, float scale, int32_t partition_tokens,
                            void *workspace, size_t workspace_bytes, const float *prefix_o,
                            const float *prefix_lse, const void *new_k, const void *new_v,
                            uint32_t flags, cudaStream_t stream);

/*
 * Grouped decode: the cascade's two passes as one call, for groups whose
 * members' private suffixes are short (the beams of a prompt after their
 * copy-on-write fork).  [P1] feature table (beam-search row) and [P2]
 * beam/copy-on-write follow-up: beams share their prompt's blocks and each
 * owns its diverged last block; [P3] "Shared prefixes need matching
 * computation".  Each group's queries attend its shared prefix (the
 * pa_prefix_attention layout and tiling: K/V tiles read once for the whole
 * group, on the tensor cores), then one more 128-key tile that holds every
 * member's own suffix blocks, each query seeing its member's keys only; the
 * output is attention over prefix and suffix together, written as bf16, with
 * no partial results, second launch or workspace.
 *   out, q         device, [num_groups * group_size][num_q_heads][d] bf16,
 *                  sequences group by group (out written)
 *   prefix_tables, max_prefix_blocks, prefix_lens, group_order, max_prefix_len
 *                  as pa_prefix_attention (prefixes whole blocks)
 *   suffix_tables  device, [num_groups * group_size][max_suffix_blocks] int32:
 *                  each member's blocks after the prefix (pa_cascade_plan's)
 *   suffix_lens    device, [num_groups * group_size] int32, tokens after the
 *                  prefix, each <= max_suffix_len (else PA_DEVERR_SEQ_LEN)
 *   max_suffix_len host bound on every suffix length
 *   new_k, new_v   device, [num_groups * group_size][Hkv][d] bf16 or both NULL:
 *                  each member's new token, stored at its last suffix position
 *                  (as pa_decode_ex stores it) before it is attended
 *   flags          0 or PA_DECODE_EARLY_METADATA: the caller promises that
 *                  group_order, prefix_lens and prefix_tables are not written by
 *                  the kernel this call immediately follows in `stream`; they
 *                  are then read while that kernel still runs (q, the pool and
 *                  the suffix arrays still wait for it).  Results are identical
 *                  with and without it; other bits give PA_ERR_INVALID_ARG.
 * Supported when the members of one M-tile (min(group_size, 128 / (num_q_heads
 * / Hkv))) times ceil(max_suffix_len / block_size) blocks fit one 128-key
 * tile; otherwise PA_ERR_UNSUPPORTED (use pa_prefix_attention and
 * pa_decode_cascade).  head_dim 128 as pa_prefill_chunk.  The pages have no
 * counterpart to the fused form; it computes what the cascade does.
 */
pa_status pa_decode_grouped(void *out, const void *q, const pa_kv_pool *pool, const int32_t *prefix_tables,
                            int32_t max_prefix_blocks, const int32_t *prefix_lens, const int32_t *group_order,
                            const int32_t *suffix_tables, int32_t max_suffix_blocks, const int32_t *suffix_lens,
                            int32_t num_groups, int32_t group_size, int32_t num_q_heads, int32_t max_prefix_len,
                            int32_t max_suffix_len, float scale, const void *new_k, const void *new_v,
                            uint32_t flags, cudaStream_t stream);

/*
 * Check of the bounded waits: launches one CTA whose wait on a shared-memory
 * barrier that nothing arrives at gives up after limit_ns (1 us .. 1 s, else
 * PA_ERR_INVALID_ARG) through the same wait every kernel uses, records
 * PA_DEVERR_TIMEOUT and returns; read the word with pa_get_device_error.
 * Nothing faults and the context stays usable.
 */
pa_status pa_check_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

/*
 * Testing hook: the number of CTAs of the balanced (partition_tokens = 0)
 * decode grid.  ctas > 0 fixes it for every later call in the process that
 * plans that schedule (pa_decode, pa_decode_ex, pa_decode_noalloc,
 * pa_decode_host, pa_decode_cascade, pa_decode_workspace_size), still capped
 * at the batch's number of 16-token stages as the default is; 0 restores the
 * default of two CTAs per SM of the current device.  Which units a range
 * boundary cuts, and so which partial records the merge kernel combines,
 * follows from this number: sweeping it exercises every cut on one GPU,
 * whatever its SM count.  Not for production use: the setting is
 * process-wide, and a workspace sized under one setting is too small under a
 * larger one.  Negative values give PA_ERR_INVALID_ARG.  The pages have no
 * counterpart to this call.
 */
pa_status pa_set_stream_k_ctas(int32_t ctas);

/*
 * Testing hook: the number of persistent CTAs of the tensor-core kernel
 * behind pa_prefill_chunk, pa_prefix_attention and pa_decode_grouped.  That
 * kernel splits its work into units of one (M-tile, kv-head, sequence) each and
 * runs one CTA per SM by default, each CTA walking its share of the units (in
 * rounds of alternating direction) with its copy and tensor-core pipeline
 * running on from one unit into the next.  ctas > 0 fixes the grid for every
 * later call in the process (still at most one CTA per unit, and at least
 * enough CTAs that none holds more than 256 units); 0 restores the default.
 * Which units share a CTA, and so every hand-over of the pipeline from one
 * unit to the next, follows from this number: sweeping it exercises them on one
 * GPU, whatever its SM count.  The results do not depend on it.  Not for
 * production use: the setting is process-wide.  Negative values give
 * PA_ERR_INVALID_ARG.  The pages have no counterpart to this call.
 */
pa_status pa_set_prefill_ctas(int32_t ctas);

/*
 * Reads (and, if clear != 0, resets) the current device's error word after
 * synchronising `stream`.  Returns PA_ERR_DEVICE when the word is non-zero.
 */
pa_status pa_get_device_error(uint32_t *err_out, int32_t clear, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Host helpers (no GPU work).
 * ------------------------------------------------------------------------- */

/*
 * Capacity arithmetic.  [P3] "How many tail slots remain unused?": a sequence
 * of `tokens` positions needs ceil(tokens/b) blocks and leaves
 * ceil(tokens/b)*b - tokens slots idle.  tokens < 0 or block_size <= 0 is
 * PA_ERR_INVALID_ARG.
 */
pa_status pa_block_layout(int64_t tokens, int32_t block_size, int64_t *blocks, int64_t *unused);

/*
 * Slot mapping on the host.  [P3] "A block table maps logical order to
 * physical storage": position t of sequence s lives in physical block
 * tables[s][t // b] at offset t % b; its slot is that block * b + offset.
 *   slots [n] (written), tables [num_seqs][max_blocks], seq_idx [n],
 *   positions [n]; all host memory.
 * A position outside the table or an entry outside [0, num_blocks) is
 * PA_ERR_INVALID_ARG (slots then unspecified).
 */
pa_status pa_slot_mapping(int64_t *slots, const int32_t *tables, int32_t num_seqs,
                          int32_t max_blocks, const int32_t *seq_idx, const int64_t *positions,
                          int64_t n, int32_t block_size, int64_t num_blocks);

/* ---------------------------------------------------------------------------
 * Host block manager: free list, per-block reference counts, fork and
 * copy-on-write planning.  [P1] "A strong answer" (on-demand equal-size
 * blocks, one table per sequence) and its feature table (shared prefix with a
 * refcount per block; beam fork sharing blocks with copy-on-write of the
 * diverging block); [P1] "What interviewers probe next" (admission needs
 * ceil(prompt/b) + 1 free blocks, plus a watermark reserve).
 * Not thread-safe: one manager per thread or external locking.
 * ------------------------------------------------------------------------- */
typedef struct pa_bm pa_bm;

/* A manager over physical blocks [0, num_blocks) of size block_size. */
pa_status pa_bm_create(pa_bm **out, int64_t num_blocks, int32_t block_size);
void pa_bm_destroy(pa_bm *bm);

/* New empty sequence (0 tokens, no blocks). */
pa_status pa_bm_add_seq(pa_bm *bm, int32_t *seq_out);

/*
 * Appends n tokens to seq, allocating blocks on demand.  slots_out (may be
 * NULL) receives the n new slots.  If the sequence's last block is shared
 * (refcount > 1) and only partly filled, the first append forks it:
 * a fresh block is allocated, (src, dst) is written to cow_pair_out (may be
 * NULL) and *n_cow_out is set to 1 -- the caller must run pa_copy_blocks on
 * that pair before writing the new slots.  PA_ERR_NO_BLOCKS leaves the
 * sequence unchanged.
 */
pa_status pa_bm_append_tokens(pa_bm *bm, int32_t seq, int64_t n, int64_t *slots_out,
                              int32_t *cow_pair_out, int32_t *n_cow_out);

/* New sequence sharing every block of parent (refcount + 1 on each). */
pa_status pa_bm_fork(pa_bm *bm, int32_t parent, int32_t *child_out);

/* Releases a sequence; blocks whose refcount drops to 0 return to the pool. */
pa_status pa_bm_free_seq(pa_bm *bm, int32_t seq);

/* Writes seq's table into table_out[0..cap) (-1 past its blocks). */
pa_status pa_bm_get_table(const pa_bm *bm, int32_t seq, int32_t *table_out, int32_t cap,
                          int32_t *num_blocks_out, int64_t *num_tokens_out);

/* Free blocks left; reference count of one block (-1 if out of range). */
int64_t pa_bm_num_free(const pa_bm *bm);
int32_t pa_bm_refcount(const pa_bm *bm, int64_t block);

/* *admit = 1 iff free blocks >= ceil(prompt_tokens/b) + 1 + watermark_blocks. */
pa_status pa_bm_can_admit(const pa_bm *bm, int64_t prompt_tokens, int64_t watermark_blocks,
                          int32_t *admit);

/*
 * Swapping ([P1] feature table, preemption row; "What interviewers probe
 * next").  pa_bm_set_host_pool gives the manager host_blocks host slots (the
 * blocks of the pinned buffer pa_swap_blocks uses); it fails with
 * PA_ERR_INVALID_ARG while any slot is in use.
 * pa_bm_swap_out moves every block of seq to a fresh host slot: it writes one
 * (device block, host block) pair per table entry, in table order, to
 * pairs_out ([cap][2]) and *n_pairs_out; the caller runs
 * pa_swap_blocks(PA_SWAP_OUT) on them before reusing the device blocks, whose
 * references the sequence drops (a block shared with another sequence stays
 * on the device for it).  pa_bm_swap_in takes fresh device blocks from the
 * free list and writes the pairs for pa_swap_blocks(PA_SWAP_IN); the host slots
 * are free once that copy has run.  PA_ERR_NO_BLOCKS (too few free host
 * slots, or device blocks) and PA_ERR_INVALID_ARG (cap too small) leave the
 * sequence unchanged.  While swapped out, a sequence cannot be appended to,
 * forked or read as a table (PA_ERR_SWAPPED); freeing it releases its host
 * slots.  Swapping in a sequence that is not swapped out, or out one that is,
 * gives PA_ERR_SWAPPED.
 */
pa_status pa_bm_set_host_pool(pa_bm *bm, int64_t host_blocks);
pa_status pa_bm_swap_out(pa_bm *bm, int32_t seq, int32_t *pairs_out, int32_t cap, int32_t *n_pairs_out);
pa_status pa_bm_swap_in(pa_bm *bm, int32_t seq, int32_t *pairs_out, int32_t cap, int32_t *n_pairs_out);
/* Free host slots (-1 for a NULL manager); 1 if seq is swapped out, 0 if it
 * is on the device, -1 if it does not exist. */
int64_t pa_bm_num_free_host(const pa_bm *bm);
int32_t pa_bm_is_swapped(const pa_bm *bm, int32_t seq);

/*
 * Prefix cache ([P1] shared-system-prompt paragraph: a prefix many requests
 * share is stored once and every table points at its blocks; [P3] "Shared
 * prefixes need matching computation": a block's K/V depend on all the tokens
 * before it and on the conditions of the computation, so equal tokens after a
 * different context, or under another model, do not match).
 * The manager keeps an index of full blocks keyed by (the entry before it, a
 * caller-given 64-bit condition key -- model, adapter, anything else the K/V
 * depend on --, the block's b token ids), compared exactly (the chained hash
 * of the token ids only picks the bucket).  The index holds one reference on
 * every cached block.  Blocks that only the index holds are evictable: an
 * allocation that finds the free list empty, or pa_bm_prefix_evict, drops the
 * least recently used such entry together with every entry after it in its
 * chain, and blocks left unreferenced return to the free list.  Blocks
 * available to appends, swap-ins and pa_bm_can_admit are the free ones plus
 * the evictable ones; pa_bm_num_free counts free ones only.
 *
 * pa_bm_prefix_match: tokens (int32 ids) of the whole blocks at the head of
 * tokens[0..n_tokens) that are cached under condition (a multiple of b).
 * Changes nothing.
 * pa_bm_add_seq_cached: a new sequence whose table starts with those cached
 * blocks (reference + 1 each) and whose length is the matched token count,
 * written to *matched_tokens_out; the caller appends and computes the rest.
 * Pass fewer tokens than the prompt to keep some of it to compute.
 * pa_bm_cache_seq: publishes the first floor(n_tokens/b) blocks of seq, whose
 * token ids are tokens[0..n_tokens) (n_tokens <= its length), after their K/V
 * were written.  Blocks whose (context, tokens) are already cached keep the
 * existing entry; the chain continues from it.  Publishing stops at a block the
 * index already holds under other content.  *inserted_out (may be NULL) is the
 * number of new entries.  Matching and publishing count as uses for the
 * least-recently-used order, deeper blocks older than the ones before them.
 * pa_bm_prefix_evict evicts until n_blocks blocks are free or nothing is
 * evictable; *freed_out (may be NULL) is the number freed.
 * pa_bm_prefix_stats: cumulative matched and offered tokens of
 * pa_bm_add_seq_cached.
 * Errors: PA_ERR_INVALID_ARG for NULL or negative arguments or n_tokens past
 * the sequence's length, PA_ERR_NOT_FOUND / PA_ERR_SWAPPED as for the other
 * sequence calls.
 */
pa_status pa_bm_prefix_match(const pa_bm *bm, const int32_t *tokens, int64_t n_tokens, uint64_t condition,
                             int64_t *matched_tokens_out);
pa_status pa_bm_add_seq_cached(pa_bm *bm, const int32_t *tokens, int64_t n_tokens, uint64_t condition,
                               int32_t *seq_out, int64_t *matched_tokens_out);
pa_status pa_bm_cache_seq(pa_bm *bm, int32_t seq, const int32_t *tokens, int64_t n_tokens, uint64_t condition,
                          int64_t *inserted_out);
pa_status pa_bm_prefix_evict(pa_bm *bm, int64_t n_blocks, int64_t *freed_out);
/* Cached entries, evictable entries (-1 for a NULL manager). */
int64_t pa_bm_num_cached(const pa_bm *bm);
int64_t pa_bm_num_evictable(const pa_bm *bm);
pa_status pa_bm_prefix_stats(const pa_bm *bm, int64_t *hit_tokens_out, int64_t *query_tokens_out);

/* ---------------------------------------------------------------------------
 * Capacity of a KV budget, contiguous reservation against paging.
 * [P1] "A strong answer": the worked Llama 3.1 70B arithmetic (a contiguous
 * allocator reserves max_seq_len tokens a request; with b-token blocks a
 * request holds ceil(L/b) blocks, so 850 tokens take 54 blocks of 16) and the
 * shared-system-prompt paragraph (the prefix's blocks are stored once and
 * every table points at them).  [P3] "How many tail slots remain unused?":
 * ceil(T/b)*b - T idle slots per sequence.  Host arithmetic, O(n_lens).
 * ------------------------------------------------------------------------- */
typedef struct {
    int64_t contiguous_requests;   /* floor(budget / (max_seq_len * bytes_per_token))           */
    int64_t paged_requests;        /* requests admitted from lens[] in turn (see below)          */
    double contiguous_waste;       /* 1 - sum(L) / (n * max_seq_len): unused share of reservations */
    double paged_waste;            /* 1 - sum(L) / sum(ceil(L/b) * b), nothing shared            */
    double mean_tail_slots;        /* mean of ceil(L/b) * b - L                                   */
    double prefix_bytes_contiguous;/* n * prefix * bytes_per_token: a copy per request            */
    double prefix_bytes_paged;     /* (floor(prefix/b) * b + n * (prefix mod b)) * bytes_per_token */
} pa_capacity;

/*
 * lens[0..n_lens) are request lengths in tokens (each a copy of the same
 * shared_prefix_tokens-token prompt prefix followed by its own tokens, so
 * shared_prefix_tokens <= L <= max_seq_len; 0 = no shared prefix).  Paged
 * admission stores the prefix's floor(prefix/b) whole blocks once (a partial
 * last prefix block stays private: the request's first own token goes there),
 * then takes requests from lens[] in turn, cycling, each holding
 * ceil(L/b) - floor(prefix/b) blocks of b * bytes_per_token bytes, and stops at
 * the first one that does not fit in floor(budget / (b * bytes_per_token))
 * blocks.  Returns PA_ERR_INVALID_ARG for NULL pointers, n_lens <= 0,
 * block_size, max_seq_len or bytes_per_token <= 0, a negative budget or
 * prefix, a length outside [prefix, max_seq_len], a list whose requests hold
 * no private block at all, or a product that overflows int64; *out is then
 * unspecified.
 */
pa_status pa_capacity_estimate(const int64_t *lens, int64_t n_lens, int64_t shared_prefix_tokens,
                               int32_t block_size, int64_t max_seq_len, int64_t bytes_per_token,
                               int64_t budget_bytes, pa_capacity *out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
