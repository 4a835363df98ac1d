/*
 * pa_oracle.c -- CPU oracle for paged KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously correct
 * statement of what the paged attention path computes.  Only the test suite,
 * the smoke check and the bench's CPU-baseline leg may load it; the product
 * library never links, calls or falls back to it, and it shares no code,
 * header or constant with the CUDA path.
 *
 * Arithmetic is fp64 throughout.  bf16 inputs are widened exactly (a bf16 is
 * the upper half of an IEEE binary32).  Nothing here is blocked, fused or
 * reordered beyond the definitions below.
 *
 * Sources (page, section):
 *  - how-pagedattention-works (aiinfrainterviews.com), "A strong answer":
 *    per layer, K/V are stored in equal blocks of 16 token slots; each
 *    sequence owns a table from logical block number to physical block, and
 *    attention fetches every query's keys and values from the blocks that
 *    table names.
 *  - attn-paged-attention-mcq-hard (zenaique.com), the conceptual
 *    block-lookup listing: each position below seq_len is resolved to
 *    (block_table[pos // block_size], pos % block_size), its K and V are read
 *    from a pool shaped [num_blocks, 2, num_layers, num_kv_heads, block_size,
 *    d_head], and ordinary scaled dot-product attention runs on the rows so
 *    collected.
 *  - auto-20261007-1900-en (lihaoran.work), "A block table maps logical order
 *    to physical storage": logical block t // b, offset t % b, and with table
 *    [5,1,7] and b = 4 position 9 resolves to block 7, offset 1; paging moves
 *    storage only, so a causal query still attends its whole visible prefix.
 *    "How many tail slots remain unused?": ceil(T/b) blocks, ceil(T/b)*b - T
 *    idle slots, zero tokens need zero blocks, and T < 0 or b <= 0 is invalid.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - q-head h reads kv-head h / (Hq / Hkv) (consecutive GQA groups).
 *  - a slot is the linear index phys * b + offset; a negative slot is skipped.
 *  - attention over zero keys returns zeros.
 *  - a chunk query at absolute position ctx + j sees keys 0 .. ctx + j.
 *
 * Pool addressing.  One layer's view of the pool is described by
 * (num_blocks, Hkv, b, d, block_stride, kv_stride), all in elements: element
 * (blk, kv, h, off, i) sits at blk*block_stride + kv*kv_stride + (h*b+off)*d + i.
 * For the pages' layout [NB][2][L][Hkv][b][d] viewed at layer l the base is
 * offset by l*Hkv*b*d, block_stride = 2*L*Hkv*b*d and kv_stride = L*Hkv*b*d;
 * one layer gives the dense [NB][2][Hkv][b][d].
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t num_blocks;
    int64_t num_kv_heads;
    int64_t block_size;
    int64_t head_dim;
    int64_t block_stride; /* elements between consecutive physical blocks */
    int64_t kv_stride;    /* elements between the K half and the V half of a block */
} orc_pool;

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the OpenMP loops use from now on (n > 0); returns the count in force. */
int orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* bf16 bit pattern -> exact double */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* "How many tail slots remain unused?": blocks = ceil(T/b), unused = blocks*b - T.
 * Returns 0 on success, -1 for T < 0 or b <= 0. */
int orc_block_layout(int64_t tokens, int64_t block_size, int64_t *blocks, int64_t *unused)
{
    if (tokens < 0 || block_size <= 0)
        return -1;
    int64_t n = (tokens + block_size - 1) / block_size;
    *blocks = n;
    *unused = n * block_size - tokens;
    return 0;
}

/* "A block table maps logical order to physical storage": position t goes to
 * logical block t / b at offset t % b, and the table names its physical block. */
void orc_address(const int32_t *table_row, int64_t pos, int64_t block_size,
                 int64_t *phys, int64_t *offset)
{
    int64_t logical = pos / block_size;
    *offset = pos % block_size;
    *phys = table_row[logical];
}

/* Linear slot of position pos: phys * b + offset. */
int64_t orc_slot(const int32_t *table_row, int64_t pos, int64_t block_size)
{
    int64_t phys, off;
    orc_address(table_row, pos, block_size, &phys, &off);
    return phys * block_size + off;
}

/* slots[n] = slot of (sequence seq_idx[n], position positions[n]);
 * tables is [num_seqs][max_blocks]. */
void orc_slot_mapping(int64_t *slots, const int32_t *tables, int64_t max_blocks,
                      const int32_t *seq_idx, const int64_t *positions, int64_t n,
                      int64_t block_size)
{
    for (int64_t i = 0; i < n; ++i)
        slots[i] = orc_slot(tables + (int64_t)seq_idx[i] * max_blocks, positions[i], block_size);
}

static int64_t pool_elem(const orc_pool *p, int64_t blk, int64_t kv, int64_t h, int64_t off)
{
    return blk * p->block_stride + kv * p->kv_stride + (h * p->block_size + off) * p->head_dim;
}

/* Slot writer: for each new token n with slot s >= 0, K and V of every kv-head
 * go to physical block s / b, offset s % b.  k and v are [N][Hkv][d]. */
void orc_reshape_and_cache(uint16_t *pool, const orc_pool *p, const uint16_t *k,
                           const uint16_t *v, const int64_t *slots, int64_t n_tokens)
{
    const int64_t H = p->num_kv_heads, d = p->head_dim, b = p->block_size;
    for (int64_t n = 0; n < n_tokens; ++n) {
        int64_t s = slots[n];
        if (s < 0)
            continue;
        int64_t blk = s / b, off = s % b;
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < d; ++i) {
                pool[pool_elem(p, blk, 0, h, off) + i] = k[(n * H + h) * d + i];
                pool[pool_elem(p, blk, 1, h, off) + i] = v[(n * H + h) * d + i];
            }
    }
}

/* Copy-on-write fork: block dst receives block src's K and V (all kv-heads,
 * all slots).  pairs is [n][2] = (src, dst), applied in order. */
void orc_copy_blocks(uint16_t *pool, const orc_pool *p, const int32_t *pairs, int64_t n_pairs)
{
    const int64_t H = p->num_kv_heads, d = p->head_dim, b = p->block_size;
    for (int64_t j = 0; j < n_pairs; ++j) {
        int64_t src = pairs[2 * j], dst = pairs[2 * j + 1];
        for (int64_t kv = 0; kv < 2; ++kv)
            for (int64_t h = 0; h < H; ++h)
                for (int64_t off = 0; off < b; ++off)
                    for (int64_t i = 0; i < d; ++i)
                        pool[pool_elem(p, dst, kv, h, off) + i] = pool[pool_elem(p, src, kv, h, off) + i];
    }
}

/* Preemption by swapping (how-pagedattention-works, feature table, preemption
 * row; "What interviewers probe next": a preempted sequence's blocks go to
 * pinned host memory): block-granular copies between the pool and a host
 * array of host_blocks blocks laid out [hb][2][Hkv][b][d].  pairs is [n][2] =
 * (pool block, host block); direction 0 copies pool -> host, 1 host -> pool. */
void orc_swap_blocks(uint16_t *pool, const orc_pool *p, uint16_t *host, const int32_t *pairs, int64_t n_pairs,
                     int32_t direction)
{
    const int64_t H = p->num_kv_heads, d = p->head_dim, b = p->block_size;
    for (int64_t j = 0; j < n_pairs; ++j) {
        int64_t blk = pairs[2 * j], hb = pairs[2 * j + 1];
        for (int64_t half = 0; half < 2; ++half)
            for (int64_t h = 0; h < H; ++h)
                for (int64_t off = 0; off < b; ++off) {
                    uint16_t *pr = pool + pool_elem(p, blk, half, h, off);
                    uint16_t *hr = host + (((hb * 2 + half) * H + h) * b + off) * d;
                    for (int64_t i = 0; i < d; ++i) {
                        if (direction == 0)
                            hr[i] = pr[i];
                        else
                            pr[i] = hr[i];
                    }
                }
    }
}

/* Attention of one query row over the first n_keys positions of one
 * sequence, kv-head kvh.  Step 1 gathers K and V position by position
 * through the table (the conceptual lookup code); step 2 is standard scaled
 * dot-product attention on the gathered rows.  out is [d].  When lse is not
 * NULL it receives log(sum_t exp(x_t)), the log of the softmax denominator
 * (-inf over zero keys). */
static void attend_row(double *out, double *lse, const uint16_t *q_row, const uint16_t *pool,
                       const orc_pool *p, const int32_t *table_row, int64_t n_keys, int64_t kvh,
                       double scale)
{
    const int64_t d = p->head_dim, b = p->block_size;
    for (int64_t i = 0; i < d; ++i)
        out[i] = 0.0;
    if (lse)
        *lse = -INFINITY;
    if (n_keys <= 0)
        return;

    double *keys = (double *)malloc(sizeof(double) * (size_t)(n_keys * d));
    double *values = (double *)malloc(sizeof(double) * (size_t)(n_keys * d));
    double *x = (double *)malloc(sizeof(double) * (size_t)n_keys);

    /* gather */
    for (int64_t t = 0; t < n_keys; ++t) {
        int64_t phys, off;
        orc_address(table_row, t, b, &phys, &off);
        const uint16_t *krow = pool + pool_elem(p, phys, 0, kvh, off);
        const uint16_t *vrow = pool + pool_elem(p, phys, 1, kvh, off);
        for (int64_t i = 0; i < d; ++i) {
            keys[t * d + i] = bf16_to_double(krow[i]);
            values[t * d + i] = bf16_to_double(vrow[i]);
        }
    }

    /* scores x_t = scale * <q, K_t> */
    for (int64_t t = 0; t < n_keys; ++t) {
        double dot = 0.0;
        for (int64_t i = 0; i < d; ++i)
            dot += bf16_to_double(q_row[i]) * keys[t * d + i];
        x[t] = scale * dot;
    }

    /* softmax: w_t = exp(x_t - max x) / sum */
    double m = x[0];
    for (int64_t t = 1; t < n_keys; ++t)
        if (x[t] > m)
            m = x[t];
    double l = 0.0;
    for (int64_t t = 0; t < n_keys; ++t) {
        x[t] = exp(x[t] - m);
        l += x[t];
    }

    if (lse)
        *lse = m + log(l);

    /* out = sum_t w_t V_t */
    for (int64_t t = 0; t < n_keys; ++t)
        for (int64_t i = 0; i < d; ++i)
            out[i] += (x[t] / l) * values[t * d + i];

    free(keys);
    free(values);
    free(x);
}

/* Paged decode attention for selected (sequence, q-head) rows.
 *   q      [B][Hq][d] bf16 bits
 *   tables [B][max_blocks] physical block ids
 *   rows   [n_rows][2] = (s, h); out [n_rows][d]
 * Sequence s attends all seq_lens[s] cached positions; q-head h reads kv-head
 * h / (Hq / Hkv). */
void orc_paged_decode_rows(double *out, const uint16_t *q, const uint16_t *pool, const orc_pool *p,
                           const int32_t *tables, int64_t max_blocks, const int32_t *seq_lens,
                           int64_t num_q_heads, double scale, const int32_t *rows, int64_t n_rows)
{
    const int64_t d = p->head_dim;
    const int64_t group = num_q_heads / p->num_kv_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t s = rows[2 * r], h = rows[2 * r + 1];
        attend_row(out + r * d, NULL, q + (s * num_q_heads + h) * d, pool, p, tables + s * max_blocks,
                   seq_lens[s], h / group, scale);
    }
}

/* All rows: out [B][Hq][d]. */
void orc_paged_decode(double *out, const uint16_t *q, const uint16_t *pool, const orc_pool *p,
                      const int32_t *tables, int64_t max_blocks, const int32_t *seq_lens,
                      int64_t num_seqs, int64_t num_q_heads, double scale)
{
    const int64_t d = p->head_dim;
    const int64_t group = num_q_heads / p->num_kv_heads;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t s = 0; s < num_seqs; ++s)
        for (int64_t h = 0; h < num_q_heads; ++h)
            attend_row(out + (s * num_q_heads + h) * d, NULL, q + (s * num_q_heads + h) * d, pool, p,
                       tables + s * max_blocks, seq_lens[s], h / group, scale);
}

/* Decode attention of all rows with each row's log-sum-exp: out [B][Hq][d],
 * lse [B][Hq].  Attention over keys A followed by keys B equals the
 * weighted mean of the attention over A and over B with weights
 * exp(lse_A) and exp(lse_B); a cascade over a shared prefix rests on it. */
void orc_paged_decode_lse(double *out, double *lse, const uint16_t *q, const uint16_t *pool,
                          const orc_pool *p, const int32_t *tables, int64_t max_blocks,
                          const int32_t *seq_lens, int64_t num_seqs, int64_t num_q_heads, double scale)
{
    const int64_t d = p->head_dim;
    const int64_t group = num_q_heads / p->num_kv_heads;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t s = 0; s < num_seqs; ++s)
        for (int64_t h = 0; h < num_q_heads; ++h)
            attend_row(out + (s * num_q_heads + h) * d, lse + s * num_q_heads + h,
                       q + (s * num_q_heads + h) * d, pool, p, tables + s * max_blocks, seq_lens[s],
                       h / group, scale);
}

/* Chunked prefill against paged context, for selected (s, j, h) rows.
 *   q [B][C][Hq][d]; row (s, j, h) is the chunk query at absolute position
 *   ctx_lens[s] + j and, attention being causal, sees keys 0 .. ctx_lens[s] + j.
 *   The chunk's own K/V are already in the pool.  rows [n][3]; out [n][d]. */
void orc_prefill_rows(double *out, const uint16_t *q, const uint16_t *pool, const orc_pool *p,
                      const int32_t *tables, int64_t max_blocks, const int32_t *ctx_lens,
                      int64_t chunk, int64_t num_q_heads, double scale, const int32_t *rows,
                      int64_t n_rows)
{
    const int64_t d = p->head_dim;
    const int64_t group = num_q_heads / p->num_kv_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t s = rows[3 * r], j = rows[3 * r + 1], h = rows[3 * r + 2];
        int64_t visible = (int64_t)ctx_lens[s] + j + 1;
        attend_row(out + r * d, NULL, q + ((s * chunk + j) * num_q_heads + h) * d, pool, p,
                   tables + s * max_blocks, visible, h / group, scale);
    }
}

/* All rows: out [B][C][Hq][d]. */
void orc_prefill(double *out, const uint16_t *q, const uint16_t *pool, const orc_pool *p,
                 const int32_t *tables, int64_t max_blocks, const int32_t *ctx_lens,
                 int64_t num_seqs, int64_t chunk, int64_t num_q_heads, double scale)
{
    const int64_t d = p->head_dim;
    const int64_t group = num_q_heads / p->num_kv_heads;
#pragma omp parallel for collapse(3) schedule(dynamic, 4)
    for (int64_t s = 0; s < num_seqs; ++s)
        for (int64_t j = 0; j < chunk; ++j)
            for (int64_t h = 0; h < num_q_heads; ++h) {
                int64_t visible = (int64_t)ctx_lens[s] + j + 1;
                int64_t row = (s * chunk + j) * num_q_heads + h;
                attend_row(out + row * d, NULL, q + row * d, pool, p, tables + s * max_blocks, visible,
                           h / group, scale);
            }
}

/* Capacity of a KV budget (how-pagedattention-works, "A strong answer": the
 * worked Llama 3.1 70B example and the shared-system-prompt paragraph;
 * auto-20261007-1900-en, "How many tail slots remain unused?").  Every
 * quantity is obtained by simulating the two allocators request by request
 * and token by token, not from a closed form.
 *   contiguous: each admitted request reserves max_len token slots up front;
 *     requests are admitted while the next reservation still fits the budget.
 *   paged: the shared prefix's whole blocks are allocated once; then requests
 *     are taken from lens[] in turn, cycling, and each one's tokens past those
 *     shared blocks are placed slot by slot, a fresh block opening whenever a
 *     token lands at offset 0; the first request whose blocks do not all fit
 *     is returned and admission stops.
 * out[0] contiguous requests, out[1] paged requests, out[2] the unused share
 * of the contiguous reservations of lens[] (one request each), out[3] the
 * unused share of the blocks those requests hold when nothing is shared,
 * out[4] mean unused tail slots per request, out[5] bytes the prefix takes
 * when every request keeps its own copy, out[6] bytes it takes when its whole
 * blocks are shared (a partial last prefix block stays per request).
 * Returns -1 on invalid input (as the library call's argument rules). */
int orc_capacity(const int64_t *lens, int64_t n, int64_t prefix, int64_t b, int64_t max_len,
                 int64_t bytes_per_token, int64_t budget, double *out)
{
    if (n <= 0 || b <= 0 || max_len <= 0 || bytes_per_token <= 0 || budget < 0 || prefix < 0)
        return -1;
    int64_t private_total = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (lens[i] < prefix || lens[i] > max_len) return -1;
        private_total += lens[i] - (prefix / b) * b;
    }
    if (private_total == 0) return -1;

    /* contiguous allocator */
    int64_t reserved = 0, contiguous = 0;
    while (reserved + max_len * bytes_per_token <= budget) {
        reserved += max_len * bytes_per_token;
        contiguous += 1;
    }

    /* per-request slot accounting without sharing */
    double used = 0.0, reserved_slots = 0.0, held_slots = 0.0, tail = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t slots = 0;
        for (int64_t t = 0; t < lens[i]; ++t)
            if (t % b == 0) slots += b;
        used += (double)lens[i];
        reserved_slots += (double)max_len;
        held_slots += (double)slots;
        tail += (double)(slots - lens[i]);
    }

    /* paged allocator with the prefix's whole blocks shared */
    int64_t free_blocks = budget / (b * bytes_per_token);
    int64_t shared = prefix / b, paged = 0;
    if (free_blocks >= shared) {
        free_blocks -= shared;
        for (int64_t r = 0;; ++r) {
            const int64_t len = lens[r % n];
            int64_t opened = 0, ok = 1;
            for (int64_t t = shared * b; t < len; ++t) {
                if (t % b == 0) {
                    if (free_blocks == 0) { ok = 0; break; }
                    free_blocks -= 1;
                    opened += 1;
                }
            }
            if (!ok) { free_blocks += opened; break; }
            paged += 1;
        }
    }

    out[0] = (double)contiguous;
    out[1] = (double)paged;
    out[2] = 1.0 - used / reserved_slots;
    out[3] = 1.0 - used / held_slots;
    out[4] = tail / (double)n;
    out[5] = (double)n * (double)prefix * (double)bytes_per_token;
    out[6] = ((double)shared * (double)b + (double)n * (double)(prefix - shared * b)) * (double)bytes_per_token;
    return 0;
}
