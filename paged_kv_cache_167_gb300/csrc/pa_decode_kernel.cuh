// pa_decode_kernel.cuh -- paged GQA decode attention for sm_103a: the
// split-context partition kernel, the persistent stream-K kernel, and the
// kernels that merge their partial results.
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
//  * The work of a (sequence, kv-head) unit is a run of pipeline stages of 16
//    token slots (one 16-token block, or several smaller blocks).  Two
//    schedules share the per-stage code:
//      - split-context partitions (explicit partition size): grid
//        (partition, kv-head, sequence), partials merged by a reduce kernel;
//      - stream-K (the automatic plan): a persistent grid of two CTAs per SM,
//        each owning an equal contiguous range of all stages in (sequence,
//        kv-head, stage) order.  A unit lying wholly inside one CTA's range is
//        written directly; a unit cut by a range boundary leaves partials in
//        the (at most two) CTAs that share it, merged by a second kernel.  This
//        removes the partly filled last wave and the per-CTA start-up of a
//        unit-per-CTA grid.
//  * Each warp owns every W-th stage of its CTA's work and a private ring of
//    STAGES shared-memory slots.  Lane 0 fetches a stage's K and V slabs (b*d
//    bf16 each, contiguous in the pool) with bulk TMA copies that complete on
//    the slot's mbarrier; block ids come from a per-warp register cache filled
//    by all lanes, so address generation never waits on a dependent table
//    load.  No data is multicast.
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
//  * The warps' (m, l, o) are merged in shared memory; bf16 output or fp32
//    partials (o normalised by l, m in the log2 domain, l) are written.
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
#ifndef PA_DECODE_SK_STAGES
#define PA_DECODE_SK_STAGES 2
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
constexpr int kStages = PA_DECODE_STAGES;      // ring depth per warp, split-context kernel
constexpr int kSkStages = PA_DECODE_SK_STAGES; // ring depth per warp, stream-K kernel
constexpr int kMinCtas = PA_DECODE_MIN_CTAS;   // resident CTAs per SM the register budget targets
constexpr int kMaxSegs = 32;                   // stream-K: units per pass of a CTA's range
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

template <int D, int G, int BS, int NS>
struct alignas(16) WarpSmem {
    using S = Shape<D, G, BS>;
    __nv_bfloat16 k[NS][S::TPS * D];
    __nv_bfloat16 v[NS][S::TPS * D];
    uint32_t p[S::TPS][S::PW];        // bf16 probabilities by (token, head), packed in pairs
    float alpha[G < 4 ? 4 : G];       // running-max correction by head
    uint64_t bar[NS + (NS & 1)];
};

// CTA-level scratch of the stream-K kernel (after the warps' rings).
template <int D, int G>
struct alignas(16) SkSmem {
    float cm[kWarps * G];             // warps' running maxima
    float cl[kWarps * G];             // warps' denominators
    float co[kWarps * G * D];         // warps' numerators
    __nv_bfloat16 q[2][G * D];        // q of the current and next unit
    int seg_s[kMaxSegs], seg_g[kMaxSegs], seg_kb[kMaxSegs], seg_ke[kMaxSegs], seg_lb[kMaxSegs + 1];
    int scan[kWarps];                 // block-scan scratch
    int found_s, found_base, nseg, more;
    uint64_t qbar[2];
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
    int32_t num_seqs;
    int32_t num_kv_heads;
    int32_t num_q_heads;
    int32_t max_seq_len;
    float scale_log2;          // scale * log2(e)
    int32_t part_tokens;       // split-context: partition length; stream-K: max_seq_len bound
    int32_t num_parts;         // split-context: partitions; stream-K: 1
    float *ws_o;               // split-context [B][Hq][P][D]; stream-K records [2C][G][D]
    float *ws_ml;              // split-context [B][Hq][P][2]; stream-K records [2C][G][2]
    int32_t *ws_cum;           // stream-K: [B + 1] exclusive prefix of stages per sequence (all kv-heads)
    int32_t num_ctas;          // stream-K grid size
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

// ---- per-lane roles and per-warp online-softmax state ------------------------

template <int D, int G, int BS>
struct Lanes {
    using S = Shape<D, G, BS>;
    int row, tsub, hl, rsel;
    __device__ __forceinline__ explicit Lanes(int lane) {
        row = lane % S::LPR;                        // this lane's 8-dim chunk of a token row
        tsub = lane / S::LPR;                       // token within a warp iteration
        // head whose score this lane ends with, and (joint rows) which of the two rows
        hl = S::JOINT ? (row & (G - 1)) : (row >> (S::LOG_LPR - S::NT));
        rsel = S::JOINT ? (row >> S::NT) : 0;
    }
};

template <int G>
struct WarpState {
    float m;          // running max (log2 domain) of head hl
    float l;          // this lane's share of the softmax denominator of head hl
    float o[G][8];    // numerators: head x this lane's 8 dims
    __device__ __forceinline__ void reset() {
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i) o[h][i] = 0.f;
    }
};

// q of one (sequence, kv-head) group on this lane's 8 dims, packed bf16; slot
// j holds head j ^ hl.  `qrows` points at the group's first head row.
template <int D, int G, int BS, bool kShared>
__device__ __forceinline__ void load_q(uint32_t (&qw)[G][4], const __nv_bfloat16 *qrows, const Lanes<D, G, BS> &ln) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const uint4 *src = reinterpret_cast<const uint4 *>(qrows + (j ^ ln.hl) * D + ln.row * 8);
        const uint4 w = kShared ? *src : __ldg(src);
        qw[j][0] = w.x;
        qw[j][1] = w.y;
        qw[j][2] = w.z;
        qw[j][3] = w.w;
    }
}

// One pipeline stage: this warp's K and V slabs of TPS tokens are in (ks, vs);
// token index tok0 + t is valid while < tok_end.
template <int D, int G, int BS, typename WS>
__device__ __forceinline__ void stage_compute(WS *ws, const __nv_bfloat16 *ks, const __nv_bfloat16 *vs,
                                              const uint32_t (&qw)[G][4], int tok0, int tok_end, float scale_log2,
                                              const Lanes<D, G, BS> &ln, WarpState<G> &st) {
    using S = Shape<D, G, BS>;
    const bool tail = tok0 + S::TPS > tok_end;
    const int row = ln.row, tsub = ln.tsub, hl = ln.hl, rsel = ln.rsel;

    // ---- scores (log2 domain) for head hl
    float sc[S::QK_ITERS];
#pragma unroll
    for (int it = 0; it < S::QK_ITERS; ++it) {
        const int t0 = it * S::ROWS * S::TPI + tsub * S::ROWS;   // first row of this lane's group
        const int t = t0 + rsel;                                 // the row whose score this lane keeps
        const uint4 kown = *reinterpret_cast<const uint4 *>(ks + t * D + row * 8);
        uint4 koth = kown;
        if constexpr (S::JOINT) koth = *reinterpret_cast<const uint4 *>(ks + (t0 + 1 - rsel) * D + row * 8);
        sc[it] = qk_dot<D, G, BS>(qw, kown, koth) * scale_log2;
        if (tail && tok0 + t >= tok_end) sc[it] = -INFINITY;
    }

    // ---- online softmax for head hl over this stage
    float mb = sc[0];
#pragma unroll
    for (int it = 1; it < S::QK_ITERS; ++it) mb = fmaxf(mb, sc[it]);
    if constexpr (S::JOINT) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, G));
#pragma unroll
    for (int dist = S::LPR; dist < 32; dist <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, dist));
    const float m_new = fmaxf(st.m, mb);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = fast_exp2(st.m - m_use);
    float psum = 0.f;
    __nv_bfloat16 pb[S::QK_ITERS];
#pragma unroll
    for (int it = 0; it < S::QK_ITERS; ++it) {
        pb[it] = __float2bfloat16_rn(fast_exp2(sc[it] - m_use));
        psum += __bfloat162float(pb[it]);
    }
    st.l = st.l * alpha + psum;
    const bool moved = m_new != st.m;
    st.m = m_new;
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
            for (int i = 0; i < 8; ++i) st.o[h][i] *= a;
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
                bf16_fma<0, 0>(st.o[2 * hp][2 * c], pw[hp], v4[c]);
                bf16_fma<0, 1>(st.o[2 * hp][2 * c + 1], pw[hp], v4[c]);
                if constexpr (G >= 2) {
                    bf16_fma<1, 0>(st.o[2 * hp + 1][2 * c], pw[hp], v4[c]);
                    bf16_fma<1, 1>(st.o[2 * hp + 1][2 * c + 1], pw[hp], v4[c]);
                }
            }
    }
    __syncwarp();
}

// Merge the lanes that held different tokens (same dims, same running max),
// then publish this warp's (m, l, o) for the G heads into CTA scratch.
template <int D, int G, int BS>
__device__ __forceinline__ void warp_publish(WarpState<G> &st, bool has_work, const Lanes<D, G, BS> &ln, int warp,
                                             float *cm, float *cl, float *co) {
    using S = Shape<D, G, BS>;
    if constexpr (S::JOINT) st.l += __shfl_xor_sync(0xffffffffu, st.l, G);
#pragma unroll
    for (int dist = S::LPR; dist < 32; dist <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i) st.o[h][i] += __shfl_xor_sync(0xffffffffu, st.o[h][i], dist);
        st.l += __shfl_xor_sync(0xffffffffu, st.l, dist);
    }
    if (ln.tsub == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float *dst = co + (warp * G + h) * D + ln.row * 8;
#pragma unroll
            for (int i = 0; i < 8; i += 2) *reinterpret_cast<float2 *>(dst + i) = make_float2(st.o[h][i], st.o[h][i + 1]);
        }
        if (S::JOINT ? ln.rsel == 0 : (ln.row & (S::DUP - 1)) == 0) {
            cm[warp * G + ln.hl] = has_work ? st.m : -INFINITY;
            cl[warp * G + ln.hl] = has_work ? st.l : 0.f;
        }
    }
}

// Combine the kWarps warps' (m, l, o) for G heads; write bf16 rows to
// `out_rows` (final) or fp32 partials: o normalised by l at o_base + h*o_hs,
// (m, l) at ml_base + h*ml_hs.
template <int D, int G>
__device__ __forceinline__ void cta_combine_store(const float *cm, const float *cl, const float *co, bool final,
                                                  __nv_bfloat16 *out_rows, float *o_base, size_t o_hs, float *ml_base,
                                                  size_t ml_hs) {
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
        if (final) {
            reinterpret_cast<uint32_t *>(out_rows + h * D + i)[0] = pack_bf16x2(ox * inv, oy * inv);
        } else {
            *reinterpret_cast<float2 *>(o_base + h * o_hs + i) = make_float2(ox * inv, oy * inv);
            if (i == 0) *reinterpret_cast<float2 *>(ml_base + h * ml_hs) = make_float2(M, lsum);
        }
    }
}

// ---- split-context partition kernel --------------------------------------------

template <int D, int G, int BS>
__global__ void __launch_bounds__(kWarps * 32, kMinCtas) paged_decode_kernel(const Params p) {
    using S = Shape<D, G, BS>;
    using WS = WarpSmem<D, G, BS, kStages>;
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

    const Lanes<D, G, BS> ln(lane);
    uint32_t qw[G][4];
    load_q<D, G, BS, false>(qw, p.q + head0 * D, ln);
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

    WarpState<G> st;
    st.reset();
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
        stage_compute<D, G, BS>(ws, ws->k[slot], ws->v[slot], qw, tok0, tok_end, p.scale_log2, ln, st);
        issue(k + kStages);
    }

    if (!ok) {
        // A wait gave up: wait (bounded) for the copies still in flight into
        // this warp's slots before the shared memory is reused.
        const int issued = min(my_stages, consumed + kStages);
        for (int k = consumed; k < issued; ++k)
            mbar_wait_bounded(&ws->bar[k % kStages], (uint32_t)((k / kStages) & 1), p.err);
    }

    // ---- merge the warps in shared memory (stage buffers are free now)
    __syncthreads();
    float *cm = reinterpret_cast<float *>(smem_raw);   // [W][G] running max
    float *cl = cm + kWarps * G;                       // [W][G] denominators
    float *co = cl + kWarps * G;                       // [W][G][D] numerators
    warp_publish<D, G, BS>(st, my_stages > 0, ln, warp, cm, cl, co);
    __syncthreads();
    grid_launch_dependents();
    const size_t rowp = head0 * p.num_parts + part;
    cta_combine_store<D, G>(cm, cl, co, p.num_parts == 1, p.out + head0 * D, p.ws_o + rowp * D,
                            (size_t)p.num_parts * D, p.ws_ml + rowp * 2, (size_t)p.num_parts * 2);
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

// ---- stream-K kernel -------------------------------------------------------------

// Stages of one sequence (one kv-head); lengths validated as in effective_len.
template <int BS>
__device__ __forceinline__ int seq_stages(const Params &p, int s, bool report) {
    constexpr int TPS = BS >= 16 ? BS : 16;
    const int L = effective_len(p, s, BS, report);
    return (L + TPS - 1) / TPS;
}

// Inclusive block-wide scan of one int per thread (kWarps * 32 threads); also
// returns the block total.  Safe to call back to back (it synchronises first).
__device__ __forceinline__ int block_inclusive_scan(int v, int *scratch, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += u;
    }
    __syncthreads();
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    int offset = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const int x = scratch[w];
        offset += w < warp ? x : 0;
        tot += x;
    }
    total = tot;
    return v + offset;
}

template <int D, int G, int BS>
__global__ void __launch_bounds__(kWarps * 32, kMinCtas) paged_decode_sk_kernel(const Params p) {
    using S = Shape<D, G, BS>;
    using WS = WarpSmem<D, G, BS, kSkStages>;
    using SK = SkSmem<D, G>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    WS *ws = reinterpret_cast<WS *>(smem_raw) + warp;
    SK *sk = reinterpret_cast<SK *>(smem_raw + sizeof(WS) * kWarps);
    constexpr int NT = kWarps * 32;
    const int Hkv = p.num_kv_heads, B = p.num_seqs, c = blockIdx.x;

    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < kSkStages; ++st) mbar_init(&ws->bar[st], 1);
        if (warp == 0) {
            mbar_init(&sk->qbar[0], 1);
            mbar_init(&sk->qbar[1], 1);
        }
        fence_barrier_init();
    }
    grid_dependency_wait();

    // ---- total work W (stages over all units) and this CTA's range [gs, ge)
    int total = 0;
    for (int base = 0; base < B; base += NT) {
        const int s = base + tid;
        const int v = s < B ? Hkv * seq_stages<BS>(p, s, c == 0) : 0;
        int chunk;
        const int inc = block_inclusive_scan(v, sk->scan, chunk);
        if (c == 0 && s < B) p.ws_cum[s] = total + inc - v;
        total += chunk;
    }
    if (c == 0 && tid == 0) p.ws_cum[B] = total;
    const int per = (total + p.num_ctas - 1) / p.num_ctas;
    const int gs = min(total, c * per), ge = min(total, gs + per);
    if (gs >= ge) return;    // nothing issued, nothing to wait for

    // ---- the sequence whose units contain gs
    {
        int run = 0;
        for (int base = 0; base < B; base += NT) {
            const int s = base + tid;
            const int v = s < B ? Hkv * seq_stages<BS>(p, s, false) : 0;
            int chunk;
            const int inc = block_inclusive_scan(v, sk->scan, chunk);
            const int excl = run + inc - v;
            if (s < B && v > 0 && excl <= gs && gs < excl + v) {
                sk->found_s = s;
                sk->found_base = excl;
            }
            run += chunk;
        }
        __syncthreads();
    }
    int cur_s = sk->found_s, cur_rem = gs - sk->found_base;   // position of the next segment to list
    int pos = gs;                                              // global stage the next segment starts at
    const Lanes<D, G, BS> ln(lane);
    int kq = 0;                  // stages this warp has consumed (ring parity counter)
    int jbase = 0;               // segments of earlier listings (q buffer parity counter)
    bool ok = true;
    bool first_seg = true;

    while (pos < ge && ok) {
        // ---- list up to kMaxSegs segments of units, starting at (cur_s, cur_rem)
        if (tid == 0) {
            int n = 0, s = cur_s, rem = cur_rem, local = 0;
            const int len = ge - pos;
            while (local < len && n < kMaxSegs && s < B) {
                const int ns = seq_stages<BS>(p, s, false);
                if (ns == 0) {
                    ++s;
                    rem = 0;
                    continue;
                }
                const int gg = rem / ns, kb = rem % ns;
                const int take = min(ns - kb, len - local);
                sk->seg_s[n] = s;
                sk->seg_g[n] = gg;
                sk->seg_kb[n] = kb;
                sk->seg_ke[n] = kb + take;
                sk->seg_lb[n] = local;
                ++n;
                local += take;
                rem += take;
                if (rem >= Hkv * ns) {
                    ++s;
                    rem = 0;
                }
            }
            sk->seg_lb[n] = local;
            sk->nseg = n;
            sk->more = (local < len && s < B) ? 1 : 0;
            sk->found_s = s;          // where the next listing resumes
            sk->found_base = rem;
        }
        __syncthreads();
        const int nseg = sk->nseg, nlocal = sk->seg_lb[nseg];
        cur_s = sk->found_s;
        cur_rem = sk->found_base;
        if (nseg == 0) break;

        // q of the first two segments
        auto issue_q = [&](int j) {
            if (j >= nseg) return;
            const int b = (jbase + j) & 1;
            const size_t head0 = (size_t)sk->seg_s[j] * p.num_q_heads + (size_t)sk->seg_g[j] * G;
            mbar_arrive_expect_tx(&sk->qbar[b], (uint32_t)(G * D * 2));
            bulk_g2s(sk->q[b], p.q + head0 * D, (uint32_t)(G * D * 2), &sk->qbar[b]);
        };
        if (tid == 0) {
            issue_q(0);
            issue_q(1);
        }

        // this warp's local stages: i = warp + kWarps * k, k < my_n
        const int my_n = nlocal > warp ? (nlocal - warp + kWarps - 1) / kWarps : 0;
        // register cache of block ids for the warp's stages: lane l holds block
        // (kbase + l) % BPS of the warp's stage (kbase + l) / BPS
        int kb_base = 0;
        auto load_ids = [&](int base) -> int {
            const int kb = base + lane;
            const int k = kb / S::BPS, ib = kb % S::BPS;
            int id = 0;
            if (k < my_n) {
                const int i = warp + k * kWarps;
                int j = 0;
                while (j + 1 < nseg && sk->seg_lb[j + 1] <= i) ++j;
                const int s = sk->seg_s[j];
                const int logical = (sk->seg_kb[j] + i - sk->seg_lb[j]) * S::BPS + ib;
                const int L = effective_len(p, s, BS, false);
                if (logical < (L + BS - 1) / BS) {
                    id = __ldg(p.tables + (size_t)s * p.max_blocks + logical);
                    if (id < 0 || id >= p.num_blocks) {
                        raise_error(p.err, PA_DEVERR_BLOCK_ID);
                        id = 0;
                    }
                } else {
                    id = -1;   // past the sequence end: not fetched
                }
            }
            return id;
        };
        int id_cache = load_ids(0);
        auto issue = [&](int k) {   // warp-uniform k
            if (k >= my_n) return;
            if (k * S::BPS - kb_base >= 32) {
                kb_base = k * S::BPS;
                id_cache = load_ids(kb_base);
            }
            const int i = warp + k * kWarps;
            int j = 0;
            while (j + 1 < nseg && sk->seg_lb[j + 1] <= i) ++j;
            const int g = sk->seg_g[j];
            const int slot = (kq + k) % kSkStages;
            int ids[S::BPS];
#pragma unroll
            for (int ib = 0; ib < S::BPS; ++ib)
                ids[ib] = __shfl_sync(0xffffffffu, id_cache, k * S::BPS + ib - kb_base);
            if (lane == 0) {
                int nvalid = 0;
#pragma unroll
                for (int ib = 0; ib < S::BPS; ++ib) nvalid += ids[ib] >= 0 ? 1 : 0;
                mbar_arrive_expect_tx(&ws->bar[slot], (uint32_t)(nvalid * S::SLAB * 2 * 2));
                const __nv_bfloat16 *pool_g = p.pool + (size_t)g * S::SLAB;
#pragma unroll
                for (int ib = 0; ib < S::BPS; ++ib) {
                    if (ids[ib] >= 0) {
                        const __nv_bfloat16 *src = pool_g + (size_t)ids[ib] * p.block_stride;
                        bulk_g2s(ws->k[slot] + ib * S::SLAB, src, S::SLAB * 2, &ws->bar[slot]);
                        bulk_g2s(ws->v[slot] + ib * S::SLAB, src + p.kv_stride, S::SLAB * 2, &ws->bar[slot]);
                    }
                }
            }
        };
#pragma unroll
        for (int k = 0; k < kSkStages; ++k) issue(k);

        int k = 0;   // this warp's next stage in this listing
        for (int j = 0; j < nseg; ++j) {
            const int s = sk->seg_s[j], g = sk->seg_g[j];
            const int L = effective_len(p, s, BS, false);
            const int ns = (L + S::TPS - 1) / S::TPS;
            const int jg = jbase + j;
            const bool qok = mbar_wait_bounded(&sk->qbar[jg & 1], (uint32_t)((jg >> 1) & 1), p.err);
            if (!__syncthreads_and(qok)) {
                ok = false;
                break;
            }
            uint32_t qw[G][4];
            load_q<D, G, BS, true>(qw, sk->q[jg & 1], ln);
            WarpState<G> st;
            st.reset();
            const int lend = sk->seg_lb[j + 1];
            int done = 0;
            while (ok && k < my_n && warp + k * kWarps < lend) {
                const int i = warp + k * kWarps;
                const int slot = (kq + k) % kSkStages;
                const bool arrived =
                    mbar_wait_bounded(&ws->bar[slot], (uint32_t)(((kq + k) / kSkStages) & 1), p.err);
                if (!__all_sync(0xffffffffu, arrived)) {
                    ok = false;
                    break;
                }
                const int tok0 = (sk->seg_kb[j] + i - sk->seg_lb[j]) * S::TPS;
                stage_compute<D, G, BS>(ws, ws->k[slot], ws->v[slot], qw, tok0, L, p.scale_log2, ln, st);
                issue(k + kSkStages);
                ++k;
                ++done;
            }
            warp_publish<D, G, BS>(st, done > 0, ln, warp, sk->cm, sk->cl, sk->co);
            if (!__syncthreads_and(ok)) {
                ok = false;
                break;
            }
            const bool complete = sk->seg_kb[j] == 0 && sk->seg_ke[j] == ns;
            const bool is_first = first_seg && j == 0;
            const int rec = 2 * c + (is_first ? 0 : 1);
            const size_t head0 = (size_t)s * p.num_q_heads + (size_t)g * G;
            cta_combine_store<D, G>(sk->cm, sk->cl, sk->co, complete, p.out + head0 * D,
                                    p.ws_o + (size_t)rec * G * D, D, p.ws_ml + (size_t)rec * G * 2, 2);
            __syncthreads();   // scratch and this q buffer are free again
            if (tid == 0) issue_q(j + 2);
        }
        if (!ok) {
            // A wait gave up: bounded waits for this warp's copies still in flight.
            const int issued = min(my_n, k + kSkStages);
            for (int kk = k; kk < issued; ++kk)
                mbar_wait_bounded(&ws->bar[(kq + kk) % kSkStages], (uint32_t)(((kq + kk) / kSkStages) & 1), p.err);
            break;
        }
        kq += my_n;
        jbase += nseg;
        pos += nlocal;
        first_seg = false;
        if (!sk->more) break;
        __syncthreads();
    }
    grid_launch_dependents();
}

// Finish the stream-K schedule for one (sequence, kv-head) unit: zero output
// for an empty sequence; merge the partial records of a unit that two or more
// CTAs shared; nothing for a unit one CTA completed.  grid (Hkv, B).
template <int D, int G, int BS>
__global__ void __launch_bounds__(G *D / 4) paged_decode_sk_merge_kernel(const Params p) {
    grid_dependency_wait();
    const int g = blockIdx.x, s = blockIdx.y;
    const int h = threadIdx.x / (D / 4);
    const int i = (threadIdx.x % (D / 4)) * 4;
    const size_t row = (size_t)s * p.num_q_heads + (size_t)g * G + h;
    const int ns = seq_stages<BS>(p, s, false);
    if (ns == 0) {
        *reinterpret_cast<uint2 *>(p.out + row * D + i) = make_uint2(0u, 0u);
        return;
    }
    const int total = p.ws_cum[p.num_seqs];
    const int per = (total + p.num_ctas - 1) / p.num_ctas;
    const int start = p.ws_cum[s] + g * ns, last = start + ns - 1;
    const int ca = start / per, cb = last / per;
    if (ca == cb) return;
    float M = -INFINITY;
    for (int cc = ca; cc <= cb; ++cc) {
        const int rec = 2 * cc + ((cc == ca && start != ca * per) ? 1 : 0);
        M = fmaxf(M, p.ws_ml[((size_t)rec * G + h) * 2]);
    }
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
        for (int cc = ca; cc <= cb; ++cc) {
            const int rec = 2 * cc + ((cc == ca && start != ca * per) ? 1 : 0);
            const float2 mlq = *reinterpret_cast<const float2 *>(p.ws_ml + ((size_t)rec * G + h) * 2);
            const float w = mlq.y * fast_exp2(mlq.x - M);
            const float4 ov = *reinterpret_cast<const float4 *>(p.ws_o + ((size_t)rec * G + h) * D + i);
            wsum += w;
            acc.x += w * ov.x;
            acc.y += w * ov.y;
            acc.z += w * ov.z;
            acc.w += w * ov.w;
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    *reinterpret_cast<uint2 *>(p.out + row * D + i) =
        make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

// ---- launchers -----------------------------------------------------------------

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

template <typename Kernel>
cudaError_t ensure_smem(Kernel kernel, size_t smem, bool *configured) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    return cudaSuccess;
}

template <int D, int G, int BS>
constexpr size_t sk_smem_bytes() {
    return sizeof(WarpSmem<D, G, BS, kSkStages>) * kWarps + sizeof(SkSmem<D, G>);
}

template <int D, int G, int BS>
cudaError_t launch_shape(const Params &prm, int num_kv_heads, int num_seqs, bool stream_k, cudaStream_t stream) {
    if (stream_k) {
        constexpr size_t smem = sk_smem_bytes<D, G, BS>();
        static bool configured[64] = {};
        cudaError_t e = ensure_smem(paged_decode_sk_kernel<D, G, BS>, smem, configured);
        if (e != cudaSuccess) return e;
        e = launch_pdl(paged_decode_sk_kernel<D, G, BS>, dim3(prm.num_ctas), dim3(kWarps * 32), smem, stream, prm);
        if (e != cudaSuccess) return e;
        return launch_pdl(paged_decode_sk_merge_kernel<D, G, BS>, dim3(num_kv_heads, num_seqs), dim3(G * D / 4), 0,
                          stream, prm);
    }
    using WS = WarpSmem<D, G, BS, kStages>;
    constexpr size_t smem = sizeof(WS) * kWarps;
    static_assert(smem >= sizeof(float) * kWarps * G * (D + 2), "combine scratch");
    static bool configured[64] = {};
    cudaError_t e = ensure_smem(paged_decode_kernel<D, G, BS>, smem, configured);
    if (e != cudaSuccess) return e;
    e = launch_pdl(paged_decode_kernel<D, G, BS>, dim3(prm.num_parts, num_kv_heads, num_seqs), dim3(kWarps * 32),
                   smem, stream, prm);
    if (e != cudaSuccess || prm.num_parts == 1) return e;
    return launch_pdl(paged_decode_reduce_kernel<D, G, BS>, dim3(num_kv_heads, num_seqs), dim3(G * D / 4), 0,
                      stream, prm);
}

template <int D, int G>
cudaError_t launch_group(const Params &prm, int bs, int num_kv_heads, int num_seqs, bool stream_k,
                         cudaStream_t stream) {
    switch (bs) {
        case 4: return launch_shape<D, G, 4>(prm, num_kv_heads, num_seqs, stream_k, stream);
        case 8: return launch_shape<D, G, 8>(prm, num_kv_heads, num_seqs, stream_k, stream);
        case 16: return launch_shape<D, G, 16>(prm, num_kv_heads, num_seqs, stream_k, stream);
        case 32: return launch_shape<D, G, 32>(prm, num_kv_heads, num_seqs, stream_k, stream);
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
    prm.num_seqs = a.num_seqs;
    prm.num_kv_heads = a.pool.num_kv_heads;
    prm.num_q_heads = a.num_q_heads;
    prm.max_seq_len = a.max_seq_len;
    prm.scale_log2 = a.scale * kLog2e;
    prm.part_tokens = a.partition_tokens;
    prm.num_parts = a.num_partitions;
    prm.ws_o = a.ws_o;
    prm.ws_ml = a.ws_ml;
    prm.ws_cum = a.ws_cum;
    prm.num_ctas = a.num_ctas;
    prm.err = err;
    const int G = a.num_q_heads / a.pool.num_kv_heads;
    const int bs = a.pool.block_size, H = a.pool.num_kv_heads, B = a.num_seqs;
    const bool sk = a.stream_k;
    switch (G) {
        case 1: return launch_group<D, 1>(prm, bs, H, B, sk, stream);
        case 2: return launch_group<D, 2>(prm, bs, H, B, sk, stream);
        case 4: return launch_group<D, 4>(prm, bs, H, B, sk, stream);
        case 8: return launch_group<D, 8>(prm, bs, H, B, sk, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace decode
}  // namespace pa
