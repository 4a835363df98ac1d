// pa_decode_kernel.cuh -- paged GQA decode attention (split-context partition
// kernel) and the partition reduce, for sm_103a.
//
// What it computes: for sequence s, kv-head g and every query head h of g's
// group, softmax(scale * q_h . K_t) over the positions t < seq_len, applied to
// V_t, where K_t and V_t are read through the block table:
// (table[s][t // b], t % b).  Sources: how-pagedattention-works
// (aiinfrainterviews.com), "A strong answer"; attn-paged-attention-mcq-hard
// (zenaique.com), conceptual block-lookup listing (the gather belongs inside
// the kernel's inner loop); auto-20261007-1900-en (lihaoran.work), "A block
// table maps logical order to physical storage".
//
// Design:
//  * grid (partition, kv-head, sequence); a partition is a run of
//    partition_tokens context positions of one (sequence, kv-head).
//  * Each warp owns every W-th pipeline stage of the partition and a private
//    ring of STAGES shared-memory slots.  A stage is 16 token slots (one
//    16-token block, or several smaller blocks).  Lane 0 fetches a stage's K
//    and V slabs (b*d bf16 each, contiguous in the pool) with bulk TMA copies
//    that complete on the slot's mbarrier; block ids come from a per-warp
//    register cache of the table row, so address generation never waits on a
//    dependent table load.  No data is multicast.
//  * All G query heads of the group are served from one staged copy of the
//    block.  The arithmetic is the fp32-accumulating bf16 FMA of sm_100-class
//    SMs (fma.rn.f32.bf16): K, V and q are used as stored, each product is
//    exact in fp32, and no operand needs converting.
//  * Q.K: a lane owns 8 of the d dimensions of a token row (16 B) and keeps q
//    for all G heads on those dimensions in registers (packed bf16).  Partial
//    dot products are combined across the row's lanes with a transposing
//    butterfly: at each shuffle step a lane keeps half of its values and
//    receives the other half from its partner.  When a row has exactly 2G
//    lanes, two token rows are reduced together and every lane ends with one
//    (row, head) score.  Query slots are stored in a lane-dependent order so
//    that every register index of the butterfly is static.
//  * Online softmax in the log2 domain per warp.  Probabilities are rounded
//    to bf16 once and broadcast through shared memory (one 16-byte load gives
//    a token's 8 heads); the softmax denominator sums the same rounded values,
//    so the output is an exact weighted average with those weights.  The
//    running-max correction of the accumulators is skipped when no head's
//    maximum moved.
//  * P.V: a lane owns 8 dims x G heads of fp32 accumulators.
//  * At the end the warps' (m, l, o) are merged in shared memory.  With one
//    partition the CTA writes bf16 output; otherwise it writes fp32 partials
//    (o normalised by l, m, l) and the reduce kernel merges partitions.
//  * Every table entry and length is bounds-checked; an out-of-range value is
//    reported in the error word and never dereferenced.  Every barrier wait
//    is bounded.
//  * Launched with programmatic stream serialisation: set-up that reads no
//    global memory overlaps the previous kernel's tail, and every global read
//    waits on griddepcontrol.wait.
#pragma once

#include <cfloat>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 3
#endif
#ifndef PA_DECODE_MIN_CTAS
#define PA_DECODE_MIN_CTAS 2
#endif
#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 4
#endif

namespace pa {
namespace decode {

constexpr int kWarps = PA_DECODE_WARPS;        // warps per CTA, each owning every kWarps-th stage
constexpr int kStages = PA_DECODE_STAGES;      // ring depth per warp
constexpr int kMinCtas = PA_DECODE_MIN_CTAS;   // resident CTAs per SM the register budget targets
constexpr float kLog2e = 1.4426950408889634f;

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <int D, int G, int BS>
struct Shape {
    static constexpr int LPR = D / 8;                 // lanes per token row (8 dims each)
    static constexpr int TPI = 32 / LPR;              // tokens per warp iteration
    static constexpr int TPS = BS >= 16 ? BS : 16;    // tokens per pipeline stage
    static constexpr int BPS = TPS / BS;              // blocks per stage
    static constexpr int ITERS = TPS / TPI;           // P.V iterations per stage
    static constexpr int SLAB = BS * D;               // elements of one (block, K|V, head) slab
    static constexpr int LOG_LPR = ilog2(LPR);
    static constexpr int NT = ilog2(G);               // transposing butterfly steps
    static constexpr int DUP = LPR / G;               // lanes holding the same head's score (one row)
    // Two token rows are reduced jointly when a row's lanes number exactly 2G.
    static constexpr bool JOINT = LPR == 2 * G;
    static constexpr int ROWS = JOINT ? 2 : 1;        // token rows per Q.K butterfly
    static constexpr int QK_ITERS = TPS / (ROWS * TPI);
    static constexpr int PW = G < 2 ? 1 : G / 2;      // 32-bit words of one token's bf16 probabilities
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group");
    static_assert(TPS % (ROWS * TPI) == 0 && TPS % BS == 0, "stage shape");
    static_assert(BPS <= 32, "table cache");
};

template <int D, int G, int BS>
struct alignas(16) WarpSmem {
    using S = Shape<D, G, BS>;
    __nv_bfloat16 k[kStages][S::TPS * D];
    __nv_bfloat16 v[kStages][S::TPS * D];
    uint32_t p[S::TPS][S::PW];        // bf16 probabilities by (token, head), packed in pairs
    float alpha[G < 4 ? 4 : G];       // running-max correction by head
    uint64_t bar[kStages + (kStages & 1)];
};

struct Params {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *pool;
    int64_t num_blocks;
    int64_t block_stride;
    int64_t kv_stride;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    int32_t num_q_heads;
    int32_t max_seq_len;
    float scale_log2;          // scale * log2(e)
    int32_t part_tokens;
    int32_t num_parts;
    float *ws_o;               // [B][Hq][P][D]
    float *ws_ml;              // [B][Hq][P][2]: m (log2 domain), l
    unsigned int *err;
};

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// Length actually processed for a sequence: negative lengths count as 0 and
// lengths beyond the table or the host bound are clipped (both reported).
__device__ __forceinline__ int effective_len(const Params &p, int s, int block_size, bool report) {
    int L = __ldg(p.seq_lens + s);
    const int cap = min(p.max_blocks * block_size, p.num_parts * p.part_tokens);
    if (L < 0 || L > cap) {
        if (report) raise_error(p.err, PA_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// acc += (bf16 half HA of a) * (bf16 half HB of b), fp32 accumulate; 0 = low half.
template <int HA, int HB>
__device__ __forceinline__ void bf16_fma(float &acc, uint32_t a, uint32_t b) {
    if constexpr (HA == 0 && HB == 0)
        asm("{ .reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, al, bl, %0; }" : "+f"(acc) : "r"(a), "r"(b));
    else if constexpr (HA == 0 && HB == 1)
        asm("{ .reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, al, bh, %0; }" : "+f"(acc) : "r"(a), "r"(b));
    else if constexpr (HA == 1 && HB == 0)
        asm("{ .reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, ah, bl, %0; }" : "+f"(acc) : "r"(a), "r"(b));
    else
        asm("{ .reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, ah, bh, %0; }" : "+f"(acc) : "r"(a), "r"(b));
}

// 8-dim partial dot product of a packed bf16 q chunk with a packed bf16 K chunk.
__device__ __forceinline__ float dot8(const uint32_t (&q)[4], const uint32_t (&k)[4]) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        bf16_fma<0, 0>(a, q[c], k[c]);
        bf16_fma<1, 1>(b, q[c], k[c]);
    }
    return a + b;
}

// Q.K for ROWS token rows, summed over the row's LPR lanes.
//  * one row: slot j (< G) holds head j ^ hl; NT transposing steps leave the
//    lane with head hl, plain steps finish the sum.
//  * two rows (JOINT): slot j (< 2G) holds value j ^ rl, value = row * G +
//    head; the first G slots use this lane's own row.  NT + 1 transposing
//    steps leave the lane with (row rl / G, head rl % G).
// Returns the raw dot product (scale applied by the caller).
template <int D, int G, int BS>
__device__ __forceinline__ float qk_dot(const uint32_t (&q)[G][4], const uint4 kown, const uint4 koth) {
    using S = Shape<D, G, BS>;
    const uint32_t ko[4] = {kown.x, kown.y, kown.z, kown.w};
    constexpr int NV = G * S::ROWS;
    float a[NV];
#pragma unroll
    for (int j = 0; j < G; ++j) a[j] = dot8(q[j], ko);
    if constexpr (S::JOINT) {
        const uint32_t kt[4] = {koth.x, koth.y, koth.z, koth.w};
#pragma unroll
        for (int j = 0; j < G; ++j) a[G + j] = dot8(q[j], kt);
    }
    constexpr int NTR = S::JOINT ? S::NT + 1 : S::NT;  // transposing steps
#pragma unroll
    for (int st = 0; st < NTR; ++st) {
        const int half = NV >> (st + 1);
        const int dist = S::LPR >> (st + 1);
#pragma unroll
        for (int j = 0; j < half; ++j) a[j] += __shfl_xor_sync(0xffffffffu, a[j + half], dist);
    }
    float s = a[0];
#pragma unroll
    for (int dist = S::LPR >> (NTR + 1); dist >= 1; dist >>= 1) s += __shfl_xor_sync(0xffffffffu, s, dist);
    return s;
}

template <int D, int G, int BS>
__global__ void __launch_bounds__(kWarps * 32, kMinCtas) paged_decode_kernel(const Params p) {
    using S = Shape<D, G, BS>;
    using WS = WarpSmem<D, G, BS>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WS *ws = reinterpret_cast<WS *>(smem_raw) + warp;

    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(&ws->bar[st], 1);
        fence_barrier_init();
    }
    grid_dependency_wait();   // inputs may come from the previous kernel in the stream

    const int part = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int L = effective_len(p, s, BS, part == 0 && g == 0 && threadIdx.x == 0);
    const int tok_begin = part * p.part_tokens;
    const int tok_end = min(L, tok_begin + p.part_tokens);
    const int ntok = tok_end - tok_begin;
    const size_t head0 = (size_t)s * p.num_q_heads + (size_t)g * G;

    if (ntok <= 0) {
        // Nothing to attend in this partition.  The reduce ignores partitions
        // past the sequence end; with a single partition (L == 0) the output
        // is zero by the library's reading of attention over no keys.
        if (p.num_parts == 1)
            for (int i = threadIdx.x; i < G * D / 2; i += blockDim.x)
                reinterpret_cast<uint32_t *>(p.out + head0 * D)[i] = 0u;
        return;
    }

    const int row = lane % S::LPR;                        // this lane's 8-dim chunk of a token row
    const int tsub = lane / S::LPR;                       // token within a warp iteration
    // head whose score this lane ends with, and (joint rows) which of the two rows
    const int hl = S::JOINT ? (row & (G - 1)) : (row >> (S::LOG_LPR - S::NT));
    const int rsel = S::JOINT ? (row >> S::NT) : 0;

    // q on this lane's 8 dims, packed bf16; slot j holds head j ^ hl
    uint32_t qw[G][4];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(p.q + (head0 + (j ^ hl)) * D + row * 8));
        qw[j][0] = w.x;
        qw[j][1] = w.y;
        qw[j][2] = w.z;
        qw[j][3] = w.w;
    }
    __syncwarp();

    const int nblk_seq = (L + BS - 1) / BS;
    const int blk0 = tok_begin / BS;
    const int nstages = (ntok + S::TPS - 1) / S::TPS;
    const int my_stages = nstages > warp ? (nstages - warp + kWarps - 1) / kWarps : 0;
    const int32_t *table_row = p.tables + (size_t)s * p.max_blocks;
    const __nv_bfloat16 *pool_g = p.pool + (size_t)g * S::SLAB;

    // Register cache of block ids: lane i holds warp-local block kb_base + i,
    // where warp-local block kb = k * BPS + ib is block ib of the warp's k-th stage.
    int kb_base = 0;
    auto load_ids = [&](int base) -> int {
        const int kb = base + lane;
        const int k = kb / S::BPS, ib = kb % S::BPS;
        const int logical = blk0 + (warp + k * kWarps) * S::BPS + ib;
        int id = 0;
        if (k < my_stages && logical < nblk_seq) {
            id = __ldg(table_row + logical);
            if (id < 0 || id >= p.num_blocks) {
                raise_error(p.err, PA_DEVERR_BLOCK_ID);
                id = 0;  // never dereference an out-of-range id; output is undefined
            }
        }
        return id;
    };
    int id_cache = load_ids(0);

    // Issue the copies of the warp's k-th stage into ring slot k % kStages.
    auto issue = [&](int k) {
        if (k >= my_stages) return;
        if (k * S::BPS - kb_base >= 32) {  // warp-uniform
            kb_base = k * S::BPS;
            id_cache = load_ids(kb_base);
        }
        const int slot = k % kStages;
        const int first_blk = blk0 + (warp + k * kWarps) * S::BPS;
        const int nvalid = min(S::BPS, nblk_seq - first_blk);
        int ids[S::BPS];
#pragma unroll
        for (int ib = 0; ib < S::BPS; ++ib) ids[ib] = __shfl_sync(0xffffffffu, id_cache, k * S::BPS + ib - kb_base);
        if (lane == 0) {
            mbar_arrive_expect_tx(&ws->bar[slot], (uint32_t)(nvalid * S::SLAB * 2 * 2));
#pragma unroll
            for (int ib = 0; ib < S::BPS; ++ib) {
                if (ib < nvalid) {
                    const __nv_bfloat16 *src = pool_g + (size_t)ids[ib] * p.block_stride;
                    bulk_g2s(ws->k[slot] + ib * S::SLAB, src, S::SLAB * 2, &ws->bar[slot]);
                    bulk_g2s(ws->v[slot] + ib * S::SLAB, src + p.kv_stride, S::SLAB * 2, &ws->bar[slot]);
                }
            }
        }
    };

#pragma unroll
    for (int k = 0; k < kStages; ++k) issue(k);

    float m_run = -INFINITY;   // running max (log2 domain) of head hl
    float l_run = 0.f;         // this lane's share of the softmax denominator of head hl
    float o[G][8];             // numerators: head x this lane's 8 dims
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i) o[h][i] = 0.f;

    int consumed = 0;
    bool ok = true;
    for (int k = 0; k < my_stages; ++k) {
        const int slot = k % kStages;
        const bool arrived = mbar_wait_bounded(&ws->bar[slot], (uint32_t)((k / kStages) & 1), p.err);
        if (!__all_sync(0xffffffffu, arrived)) {
            ok = false;
            break;
        }
        consumed = k + 1;
        const int tok0 = tok_begin + (warp + k * kWarps) * S::TPS;
        const bool tail = tok0 + S::TPS > tok_end;
        const __nv_bfloat16 *ks = ws->k[slot];
        const __nv_bfloat16 *vs = ws->v[slot];

        // ---- scores (log2 domain) for head hl
        float sc[S::QK_ITERS];
#pragma unroll
        for (int it = 0; it < S::QK_ITERS; ++it) {
            const int t0 = it * S::ROWS * S::TPI + tsub * S::ROWS;   // first row of this lane's group
            const int t = t0 + rsel;                                 // the row whose score this lane keeps
            const uint4 kown = *reinterpret_cast<const uint4 *>(ks + t * D + row * 8);
            uint4 koth = kown;
            if constexpr (S::JOINT) koth = *reinterpret_cast<const uint4 *>(ks + (t0 + 1 - rsel) * D + row * 8);
            sc[it] = qk_dot<D, G, BS>(qw, kown, koth) * p.scale_log2;
            if (tail && tok0 + t >= tok_end) sc[it] = -INFINITY;
        }

        // ---- online softmax for head hl over this stage
        float mb = sc[0];
#pragma unroll
        for (int it = 1; it < S::QK_ITERS; ++it) mb = fmaxf(mb, sc[it]);
        if constexpr (S::JOINT) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, G));
#pragma unroll
        for (int dist = S::LPR; dist < 32; dist <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, dist));
        const float m_new = fmaxf(m_run, mb);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m_run - m_use);
        float psum = 0.f;
        __nv_bfloat16 pb[S::QK_ITERS];
#pragma unroll
        for (int it = 0; it < S::QK_ITERS; ++it) {
            pb[it] = __float2bfloat16_rn(fast_exp2(sc[it] - m_use));
            psum += __bfloat162float(pb[it]);
        }
        l_run = l_run * alpha + psum;
        const bool moved = m_new != m_run;
        m_run = m_new;
        if (S::JOINT || (row & (S::DUP - 1)) == 0) {
            __nv_bfloat16 *pt = reinterpret_cast<__nv_bfloat16 *>(&ws->p[0][0]);
#pragma unroll
            for (int it = 0; it < S::QK_ITERS; ++it)
                pt[(it * S::ROWS * S::TPI + tsub * S::ROWS + rsel) * (2 * S::PW) + hl] = pb[it];
            if (tsub == 0 && rsel == 0) ws->alpha[hl] = alpha;
        }
        __syncwarp();

        // ---- rescale (only if some head's maximum moved) and accumulate P . V
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float a = ws->alpha[h];
#pragma unroll
                for (int i = 0; i < 8; ++i) o[h][i] *= a;
            }
        }
#pragma unroll
        for (int it = 0; it < S::ITERS; ++it) {
            const int t = it * S::TPI + tsub;
            uint4 vw = *reinterpret_cast<const uint4 *>(vs + t * D + row * 8);
            if (tail && tok0 + t >= tok_end) vw = make_uint4(0u, 0u, 0u, 0u);  // slot may hold stale data
            const uint32_t v4[4] = {vw.x, vw.y, vw.z, vw.w};
            uint32_t pw[S::PW];
            if constexpr (S::PW == 4) {
                const uint4 w = *reinterpret_cast<const uint4 *>(&ws->p[t][0]);
                pw[0] = w.x;
                pw[1] = w.y;
                pw[2] = w.z;
                pw[3] = w.w;
            } else if constexpr (S::PW == 2) {
                const uint2 w = *reinterpret_cast<const uint2 *>(&ws->p[t][0]);
                pw[0] = w.x;
                pw[1] = w.y;
            } else {
                pw[0] = ws->p[t][0];
            }
#pragma unroll
            for (int hp = 0; hp < S::PW; ++hp)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    bf16_fma<0, 0>(o[2 * hp][2 * c], pw[hp], v4[c]);
                    bf16_fma<0, 1>(o[2 * hp][2 * c + 1], pw[hp], v4[c]);
                    if constexpr (G >= 2) {
                        bf16_fma<1, 0>(o[2 * hp + 1][2 * c], pw[hp], v4[c]);
                        bf16_fma<1, 1>(o[2 * hp + 1][2 * c + 1], pw[hp], v4[c]);
                    }
                }
        }
        __syncwarp();
        issue(k + kStages);
    }

    if (!ok) {
        // A wait gave up: wait (bounded) for the copies still in flight into
        // this warp's slots before the shared memory is reused.
        const int issued = min(my_stages, consumed + kStages);
        for (int k = consumed; k < issued; ++k)
            mbar_wait_bounded(&ws->bar[k % kStages], (uint32_t)((k / kStages) & 1), p.err);
    }

    // ---- merge the lanes of different tokens (same dims, same running max)
    if constexpr (S::JOINT) l_run += __shfl_xor_sync(0xffffffffu, l_run, G);
#pragma unroll
    for (int dist = S::LPR; dist < 32; dist <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i) o[h][i] += __shfl_xor_sync(0xffffffffu, o[h][i], dist);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, dist);
    }

    // ---- merge the warps in shared memory (stage buffers are free now)
    __syncthreads();
    float *cm = reinterpret_cast<float *>(smem_raw);   // [W][G] running max
    float *cl = cm + kWarps * G;                       // [W][G] denominators
    float *co = cl + kWarps * G;                       // [W][G][D] numerators
    if (tsub == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float *dst = co + (warp * G + h) * D + row * 8;
#pragma unroll
            for (int i = 0; i < 8; i += 2) *reinterpret_cast<float2 *>(dst + i) = make_float2(o[h][i], o[h][i + 1]);
        }
        if (S::JOINT ? rsel == 0 : (row & (S::DUP - 1)) == 0) {
            cm[warp * G + hl] = my_stages > 0 ? m_run : -INFINITY;
            cl[warp * G + hl] = my_stages > 0 ? l_run : 0.f;
        }
    }
    __syncthreads();
    grid_launch_dependents();

    for (int idx = threadIdx.x; idx < G * D / 2; idx += blockDim.x) {
        const int h = idx / (D / 2);
        const int i = (idx % (D / 2)) * 2;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cm[w * G + h]);
        float lsum = 0.f, ox = 0.f, oy = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = fast_exp2(cm[w * G + h] - M);
                lsum += cl[w * G + h] * f;
                const float2 ov = *reinterpret_cast<const float2 *>(co + (w * G + h) * D + i);
                ox += ov.x * f;
                oy += ov.y * f;
            }
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        if (p.num_parts == 1) {
            reinterpret_cast<uint32_t *>(p.out + (head0 + h) * D + i)[0] = pack_bf16x2(ox * inv, oy * inv);
        } else {
            const size_t rowp = (head0 + h) * p.num_parts + part;
            *reinterpret_cast<float2 *>(p.ws_o + rowp * D + i) = make_float2(ox * inv, oy * inv);
            if (i == 0) *reinterpret_cast<float2 *>(p.ws_ml + rowp * 2) = make_float2(M, lsum);
        }
    }
}

// Merge the partitions of the G query heads of one (sequence, kv-head):
// weights l_p * 2^(m_p - M).  grid (Hkv, B), G * D / 4 threads, 4 dims each.
template <int D, int G, int BS>
__global__ void __launch_bounds__(G *D / 4) paged_decode_reduce_kernel(const Params p) {
    grid_dependency_wait();   // partials come from the partition kernel
    const int g = blockIdx.x, s = blockIdx.y;
    const int h = threadIdx.x / (D / 4);
    const int i = (threadIdx.x % (D / 4)) * 4;
    const int L = effective_len(p, s, BS, false);
    const int np = (L + p.part_tokens - 1) / p.part_tokens;
    const size_t row = (size_t)s * p.num_q_heads + (size_t)g * G + h;
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + row * p.num_parts;
    float M = -INFINITY;
    for (int q = 0; q < np; ++q) M = fmaxf(M, ml[q].x);
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
        for (int q = 0; q < np; ++q) {
            const float2 mlq = ml[q];
            const float w = mlq.y * fast_exp2(mlq.x - M);
            const float4 ov = *reinterpret_cast<const float4 *>(p.ws_o + (row * p.num_parts + q) * D + i);
            wsum += w;
            acc.x += w * ov.x;
            acc.y += w * ov.y;
            acc.z += w * ov.z;
            acc.w += w * ov.w;
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2 packed = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    *reinterpret_cast<uint2 *>(p.out + row * D + i) = packed;
}

// Launch with programmatic stream serialisation (the kernel waits on
// griddepcontrol.wait before touching global memory).
template <typename Kernel>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const Params &prm) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, prm);
}

template <int D, int G, int BS>
cudaError_t launch_shape(const Params &prm, int num_kv_heads, int num_seqs, cudaStream_t stream) {
    using WS = WarpSmem<D, G, BS>;
    constexpr size_t smem = sizeof(WS) * kWarps;
    static_assert(smem >= sizeof(float) * kWarps * G * (D + 2), "combine scratch");
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<D, G, BS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    cudaError_t e = launch_pdl(paged_decode_kernel<D, G, BS>, dim3(prm.num_parts, num_kv_heads, num_seqs),
                               dim3(kWarps * 32), smem, stream, prm);
    if (e != cudaSuccess || prm.num_parts == 1) return e;
    return launch_pdl(paged_decode_reduce_kernel<D, G, BS>, dim3(num_kv_heads, num_seqs), dim3(G * D / 4), 0,
                      stream, prm);
}

template <int D, int G>
cudaError_t launch_group(const Params &prm, int bs, int num_kv_heads, int num_seqs, cudaStream_t stream) {
    switch (bs) {
        case 4: return launch_shape<D, G, 4>(prm, num_kv_heads, num_seqs, stream);
        case 8: return launch_shape<D, G, 8>(prm, num_kv_heads, num_seqs, stream);
        case 16: return launch_shape<D, G, 16>(prm, num_kv_heads, num_seqs, stream);
        case 32: return launch_shape<D, G, 32>(prm, num_kv_heads, num_seqs, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_for_dim(const DecodeArgs &a, cudaStream_t stream) {
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    Params prm;
    prm.out = static_cast<__nv_bfloat16 *>(a.out);
    prm.q = static_cast<const __nv_bfloat16 *>(a.q);
    prm.pool = static_cast<const __nv_bfloat16 *>(a.pool.base);
    prm.num_blocks = a.pool.num_blocks;
    prm.block_stride = a.pool.block_stride;
    prm.kv_stride = a.pool.kv_stride;
    prm.tables = a.tables;
    prm.max_blocks = a.max_blocks;
    prm.seq_lens = a.seq_lens;
    prm.num_q_heads = a.num_q_heads;
    prm.max_seq_len = a.max_seq_len;
    prm.scale_log2 = a.scale * kLog2e;
    prm.part_tokens = a.partition_tokens;
    prm.num_parts = a.num_partitions;
    prm.ws_o = a.ws_o;
    prm.ws_ml = a.ws_ml;
    prm.err = err;
    const int G = a.num_q_heads / a.pool.num_kv_heads;
    const int bs = a.pool.block_size, H = a.pool.num_kv_heads, B = a.num_seqs;
    switch (G) {
        case 1: return launch_group<D, 1>(prm, bs, H, B, stream);
        case 2: return launch_group<D, 2>(prm, bs, H, B, stream);
        case 4: return launch_group<D, 4>(prm, bs, H, B, stream);
        case 8: return launch_group<D, 8>(prm, bs, H, B, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace decode
}  // namespace pa
