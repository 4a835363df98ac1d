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
//        each owning an equal contiguous range of the work in (sequence,
//        kv-head, stage) order, where each unit's stages are followed by
//        kUnitCost stages of no work standing for its fixed cost (q, barrier,
//        combine, store).  A unit lying wholly inside one CTA's range is
//        written directly; a unit cut by a range boundary leaves partials in
//        the (at most two) CTAs that share it, merged by a second kernel.  This
//        removes the partly filled last wave and the per-CTA start-up of a
//        unit-per-CTA grid.
//  * Each warp owns every W-th stage of its CTA's work and a private ring of
//    STAGES shared-memory slots.  Lane 0 fetches a stage's K and V blocks with
//    tensor copies (one box of b tokens x d per block and K|V, 128-byte
//    swizzle) that complete on the slot's mbarrier; block ids come from a
//    per-warp register cache filled by all lanes, so address generation never
//    waits on a dependent table load.  No data is multicast.
//  * All G query heads of the group are served from one staged copy of the
//    block, on the tensor cores: per 16 tokens, S^T = K . Q^T is an
//    m16n8k16 bf16 MMA with fp32 accumulation (tokens on M, the group's
//    heads on N, d on K), and O^T += V^T . P^T another (d on M, heads on N,
//    tokens on K).  A lane reads whole 16-byte chunks of K and V rows from
//    shared memory; which d a chunk element stands for is a fixed
//    permutation that q (loaded once in the same order) and the output
//    write-back follow, and the 128-byte swizzle makes every read
//    bank-conflict free.  P^T is formed from the S^T accumulators with one
//    register transpose (movmatrix) per 8 x 8 tile.
//  * Online softmax in the log2 domain per warp: a head's running maximum
//    is reduced across the 8 lanes holding its tokens.  A probability enters
//    P.V as the sum of two bf16 terms (its bf16 rounding and the rounding of
//    the remainder), i.e. two MMAs per tile, so the weights carry ~16
//    significant bits; a single bf16 rounding of p alone can move an output
//    by ~2^-9 of the spread of the V values it averages.  The accumulators
//    are rescaled only when some head's maximum moved.
//  * The warps' (m, l, o) are merged in shared memory; bf16 output or fp32
//    partials (o normalised by l, m in the log2 domain, l) are written.
//  * Cascade (a prefix term given): every writer of a final output row folds
//    in the row's attention over a shared prefix, computed apart, as one more
//    record (its normalised output with l = 1 and m = its log-sum-exp).
//  * Every table entry and length is bounds-checked; an out-of-range value is
//    reported in the error word and never dereferenced.  Every barrier wait
//    is bounded.
//  * Launched with programmatic stream serialisation: set-up that reads no
//    global memory overlaps the previous kernel's tail, and every global read
//    waits on griddepcontrol.wait -- except, when the caller sets the
//    early-metadata flag (lengths and tables not written by the previous
//    kernel), the stream-K kernel's reads of lengths and table entries, the
//    planning of its first listing and L2 prefetches of its first stages'
//    blocks, which then overlap that kernel too.
//  * The stream-K merge kernel runs one block per decode CTA, so its blocks
//    wait resident beside the decode CTAs instead of holding SMs that the
//    next call's decode CTAs need.
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
constexpr int kOnePassSeqs = kWarps * 32;       // stream-K: sequences listed in one pass, one per thread
constexpr int kMaxSegs = 32;                   // stream-K: units per pass of a CTA's range
#ifndef PA_SK_PREFETCH_STAGES
#define PA_SK_PREFETCH_STAGES 2
#endif
// Stream-K with early metadata: stages per warp whose K/V boxes are prefetched
// into L2 before griddepcontrol.wait, while the previous kernel finishes.
constexpr int kSkPrefetch = PA_SK_PREFETCH_STAGES;
#ifndef PA_SK_UNIT_COST
#define PA_SK_UNIT_COST 12
#endif
// Stream-K balances work in stages plus kUnitCost stages of no work per unit:
// a unit costs a CTA more than its stages (its q, the end-of-unit barrier,
// combine and store, the pipeline refill), so ranges that hold many short
// units get fewer stages.  12 was measured best among 0, 3, 6, 9, 12, 16, 24
// on lognormal-length batches (-18% time against 0) and cost nothing on
// uniform ones.
constexpr int kUnitCost = PA_SK_UNIT_COST;
constexpr float kLog2e = 1.4426950408889634f;

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// A pipeline stage is 16 tokens: BPS whole blocks when b < 16, else a 16-row
// part of one block (one copy box of ROWS slots starting at slot_of(stage)).
template <int D, int BS>
struct Shape {
    static constexpr int TPS = 16;                    // tokens per pipeline stage
    static constexpr int ROWS = BS < 16 ? BS : 16;    // token slots per copy box
    static constexpr int BPS = TPS / ROWS;            // copy boxes (blocks) per stage
    static constexpr int KS = 1;                      // 16-token MMA steps per stage
    static constexpr int HALVES = D / 64;             // 128-byte halves of a token row
    static constexpr int BOX = ROWS * D * 2;          // bytes of one (K|V, head) copy box
    static constexpr int REGION = BOX < 1024 ? 1024 : BOX;   // its place in a slot (swizzle-atom aligned)
    static constexpr int SLOT = BPS * REGION;         // bytes of a stage's K (or V) slot
    static constexpr int NCH = D / 32;                // 16-byte chunks of a K row that one lane reads
    static constexpr int DK = D / 16;                 // Q.K steps over d = P.V tiles of d
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(BS == 4 || BS == 8 || BS == 16 || BS == 32 || BS == 64, "block size");
    // logical block of box ib of the stage starting at token tok0, and the
    // first slot the box copies (stages start on multiples of 16 tokens when
    // b >= 16, so a box never leaves its block)
    static __device__ __forceinline__ int block_of(int tok0, int ib) { return tok0 / BS + (BS < 16 ? ib : 0); }
    static __device__ __forceinline__ int slot_of(int tok0) { return BS < 16 ? 0 : tok0 % BS; }
};

// Per-warp ring of NS stage slots, K slots then V slots.  A block's box starts
// on a 1024-byte boundary, so its 128-byte swizzle pattern follows from the
// offset inside the box.
template <int D, int BS, int NS>
struct alignas(1024) WarpRing {
    unsigned char k[NS][Shape<D, BS>::SLOT];
    unsigned char v[NS][Shape<D, BS>::SLOT];
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
    int found_s, found_base, nseg, more, next_pos;
    uint64_t qbar[2];
};

// Dynamic shared memory: [slack to 1024][rings][ring barriers][extra].
template <int D, int BS, int NS>
struct SmemPlan {
    static constexpr size_t kRings = sizeof(WarpRing<D, BS, NS>) * kWarps;
    static constexpr size_t kBars = ((kWarps * NS * sizeof(uint64_t) + 127) / 128) * 128;
    static constexpr size_t bytes(size_t extra) { return 1024 + kRings + kBars + extra; }
};

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
    const uint32_t a = smem_addr(p);
    return p + (((a + 1023u) & ~1023u) - a);
}

struct Params {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    int64_t num_blocks;
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
    int32_t num_ctas;          // stream-K grid size
    int32_t early_meta;        // stream-K: lengths and tables may be read before griddepcontrol.wait
    // stream-K append: the K/V of each sequence's last token, stored at its
    // slot before the stage holding it is fetched (nullptr: no append)
    const __nv_bfloat16 *new_k;  // [B][Hkv][D]
    const __nv_bfloat16 *new_v;
    __nv_bfloat16 *pool;         // the layer's pool view (element strides below)
    int64_t block_stride;
    int64_t kv_stride;
    unsigned int *err;
    // cascade: attention of each row over a shared prefix, computed apart
    // (o normalised by its l, lse its natural-log sum of exp), folded into
    // every final output row (nullptr: none)
    const float *pre_o;          // [B][Hq][D]
    const float *pre_lse;        // [B][Hq]
};

// The prefix term of one output row: its log-sum-exp and N dims of its
// normalised output (lse = -inf: no term).  Loaded ahead of use, so that the
// load latency hides behind other work.
template <int N>
struct PrefixTerm {
    float lse;
    float o[N];
};

template <int N>
__device__ __forceinline__ PrefixTerm<N> load_prefix(const Params &p, size_t row, int D, int i, bool want = true) {
    static_assert(N == 2 || N == 4, "two or four dims");
    PrefixTerm<N> t;
    t.lse = -INFINITY;
#pragma unroll
    for (int k = 0; k < N; ++k) t.o[k] = 0.f;
    if (want && p.pre_lse != nullptr) {
        t.lse = __ldg(p.pre_lse + row);
        if constexpr (N == 2) {
            const float2 v = __ldg(reinterpret_cast<const float2 *>(p.pre_o + row * D + i));
            t.o[0] = v.x;
            t.o[1] = v.y;
        } else {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p.pre_o + row * D + i));
            t.o[0] = v.x;
            t.o[1] = v.y;
            t.o[2] = v.z;
            t.o[3] = v.w;
        }
    }
    return t;
}

// Fold a prefix term into a merge in progress: acc[] holds sum_w weight_w *
// o_w over N dims, wsum the sum of the weights, M their reference maximum
// (log2 domain).  The prefix enters as one more record with l = 1 and
// m = lse * log2(e).  Without a term nothing changes.
template <int N>
__device__ __forceinline__ void fold_prefix(const PrefixTerm<N> &t, float M, float &wsum, float (&acc)[N]) {
    if (t.lse == -INFINITY) return;
    const float mp = t.lse * 1.4426950408889634f;
    const float Mn = fmaxf(M, mp);
    const float fd = M == -INFINITY ? 0.f : fast_exp2(M - Mn);
    const float fp = fast_exp2(mp - Mn);
    wsum = wsum * fd + fp;
#pragma unroll
    for (int k = 0; k < N; ++k) acc[k] = acc[k] * fd + fp * t.o[k];
}

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

// ---- tensor-core fragments -----------------------------------------------------

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// c += A . B, m16n8k16, bf16 in, fp32 accumulate (A row-major 16 x 16, B 16 x 8).
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8 x 8 bf16 tile held one row pair per lane.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t a) {
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// Byte offset, inside a slot, of the 128-byte half row hh of the stage's
// token j, and of its 16-byte chunk c after the 128-byte swizzle.
template <int D, int BS>
__device__ __forceinline__ uint32_t row_off(int j, int hh) {
    using S = Shape<D, BS>;
    return (uint32_t)((j / S::ROWS) * S::REGION + (hh * S::ROWS + j % S::ROWS) * 128);
}
__device__ __forceinline__ uint32_t chunk_at(uint32_t row, int c) {
    return row + ((((uint32_t)c) ^ ((row >> 7) & 7u)) << 4);
}

// Lane roles: g = lane / 4 is a token row of an S^T tile / the head of a
// P^T column; t = lane % 4 picks K chunks and the head pair (2t, 2t + 1).
// K chunk idx of a lane (idx < NCH) is chunk 2t + (idx & 1) of half idx / 2;
// its 4 words are Q.K MMA operands 4 idx .. 4 idx + 3, two per d step.

// q of one (sequence, kv-head) group as the B operand of S^T = K . Q^T:
// head g (zero for g >= G), d in the lane's K chunk order.
template <int D, int G, bool kShared>
__device__ __forceinline__ void load_qf(uint32_t (&qf)[D / 8], const __nv_bfloat16 *qrows, int lane) {
    using S = Shape<D, 16>;
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int idx = 0; idx < S::NCH; ++idx) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (g < G) {
            const uint4 *src = reinterpret_cast<const uint4 *>(qrows + g * D + (idx >> 1) * 64 + (2 * t + (idx & 1)) * 8);
            w = kShared ? *src : __ldg(src);
        }
        qf[4 * idx + 0] = w.x;
        qf[4 * idx + 1] = w.y;
        qf[4 * idx + 2] = w.z;
        qf[4 * idx + 3] = w.w;
    }
}

template <int D>
struct WarpState {
    float m[2];          // running max (log2 domain) of heads 2t, 2t + 1
    float l[2];          // this lane's share of their denominators
    float o[D / 16][4];  // O^T tiles: rows d (g, g + 8 of tile), columns heads (2t, 2t + 1)
    __device__ __forceinline__ void reset() {
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }
};

// d held by row r (0 = g, 1 = g + 8) of P.V tile mt, as (half, element) of the
// lane's V chunk g: for d = 128 half r, element mt; for d = 64 element mt + 4r.
template <int D>
__host__ __device__ constexpr int pv_half(int r) { return D == 128 ? r : 0; }
template <int D>
__host__ __device__ constexpr int pv_elem(int mt, int r) { return D == 128 ? mt : mt + 4 * r; }

// One pipeline stage: this warp's K and V slots (shared-memory addresses)
// hold TPS tokens; token tok0 + j is valid while < tok_end.
template <int D, int G, int BS>
__device__ __forceinline__ void stage_compute(uint32_t kslot, uint32_t vslot, const uint32_t (&qf)[D / 8], int tok0,
                                              int tok_end, float scale_log2, int lane, WarpState<D> &st) {
    using S = Shape<D, BS>;
    const int g = lane >> 2, t = lane & 3;
    const int nvalid = tok_end - tok0;
    const bool tail = nvalid < S::TPS;

    // ---- scores (log2 domain): x[ks] = S^T of tokens 16ks + (g, g + 8), heads (2t, 2t + 1)
    float x[S::KS][4];
#pragma unroll
    for (int ks = 0; ks < S::KS; ++ks) {
        const int j0 = ks * 16 + g, j1 = j0 + 8;
        uint32_t k0[4 * S::NCH], k1[4 * S::NCH];
#pragma unroll
        for (int idx = 0; idx < S::NCH; ++idx) {
            const int hh = idx >> 1, ch = 2 * t + (idx & 1);
            const uint4 a = lds128(kslot + chunk_at(row_off<D, BS>(j0, hh), ch));
            const uint4 b = lds128(kslot + chunk_at(row_off<D, BS>(j1, hh), ch));
            k0[4 * idx + 0] = a.x;
            k0[4 * idx + 1] = a.y;
            k0[4 * idx + 2] = a.z;
            k0[4 * idx + 3] = a.w;
            k1[4 * idx + 0] = b.x;
            k1[4 * idx + 1] = b.y;
            k1[4 * idx + 2] = b.z;
            k1[4 * idx + 3] = b.w;
        }
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < S::DK; ++s) mma_bf16(c, k0[2 * s], k1[2 * s], k0[2 * s + 1], k1[2 * s + 1], qf[2 * s], qf[2 * s + 1]);
        const bool v0 = !tail || j0 < nvalid, v1 = !tail || j1 < nvalid;
        x[ks][0] = v0 ? c[0] * scale_log2 : -INFINITY;
        x[ks][1] = v0 ? c[1] * scale_log2 : -INFINITY;
        x[ks][2] = v1 ? c[2] * scale_log2 : -INFINITY;
        x[ks][3] = v1 ? c[3] * scale_log2 : -INFINITY;
    }

    // ---- online softmax for heads 2t, 2t + 1 (maxima reduced over the 8 lanes g)
    float mh0 = -INFINITY, mh1 = -INFINITY;
#pragma unroll
    for (int ks = 0; ks < S::KS; ++ks) {
        mh0 = fmaxf(mh0, fmaxf(x[ks][0], x[ks][2]));
        mh1 = fmaxf(mh1, fmaxf(x[ks][1], x[ks][3]));
    }
#pragma unroll
    for (int dist = 4; dist < 32; dist <<= 1) {
        mh0 = fmaxf(mh0, __shfl_xor_sync(0xffffffffu, mh0, dist));
        mh1 = fmaxf(mh1, __shfl_xor_sync(0xffffffffu, mh1, dist));
    }
    const float mn0 = fmaxf(st.m[0], mh0), mn1 = fmaxf(st.m[1], mh1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(st.m[0] - mu0), al1 = fast_exp2(st.m[1] - mu1);
    const bool moved = mn0 != st.m[0] || mn1 != st.m[1];
    // p as the sum of two bf16 terms, hi = bf16(p) and lo = bf16(p - hi): the
    // weights the P.V MMAs apply then agree with the fp32 probabilities to
    // about 2^-17 instead of bf16's 2^-9, and the denominator sums the fp32 p.
    uint32_t pb[S::KS][2][2];   // [ks][token row g | g + 8][hi | lo]: bf16 pairs of heads (2t, 2t + 1)
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int ks = 0; ks < S::KS; ++ks) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float pa = fast_exp2(x[ks][2 * r] - mu0), pc = fast_exp2(x[ks][2 * r + 1] - mu1);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(pa, pc);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(pa - __low2float(hi), pc - __high2float(hi));
            ps0 += pa;
            ps1 += pc;
            pb[ks][r][0] = *reinterpret_cast<const uint32_t *>(&hi);
            pb[ks][r][1] = *reinterpret_cast<const uint32_t *>(&lo);
        }
    }
    st.l[0] = st.l[0] * al0 + ps0;
    st.l[1] = st.l[1] * al1 + ps1;
    st.m[0] = mn0;
    st.m[1] = mn1;
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
        for (int mt = 0; mt < S::DK; ++mt) {
            st.o[mt][0] *= al0;
            st.o[mt][1] *= al1;
            st.o[mt][2] *= al0;
            st.o[mt][3] *= al1;
        }
    }

    // ---- O^T += V^T . P^T per 16 tokens
#pragma unroll
    for (int ks = 0; ks < S::KS; ++ks) {
        const uint32_t b0 = transpose8x8(pb[ks][0][0]), b1 = transpose8x8(pb[ks][1][0]);
        const uint32_t c0 = transpose8x8(pb[ks][0][1]), c1 = transpose8x8(pb[ks][1][1]);
        // V chunk g (each half) of tokens 16ks + 2t, +1, +8, +9; tokens past the
        // end read as zero (their slots may hold stale or non-finite data)
        uint32_t vw[4][S::HALVES][4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int j = ks * 16 + 2 * t + (kk & 1) + 8 * (kk >> 1);
            const bool valid = !tail || j < nvalid;
#pragma unroll
            for (int hh = 0; hh < S::HALVES; ++hh) {
                uint4 w = lds128(vslot + chunk_at(row_off<D, BS>(j, hh), g));
                if (!valid) w = make_uint4(0u, 0u, 0u, 0u);
                vw[kk][hh][0] = w.x;
                vw[kk][hh][1] = w.y;
                vw[kk][hh][2] = w.z;
                vw[kk][hh][3] = w.w;
            }
        }
#pragma unroll
        for (int mt = 0; mt < S::DK; ++mt) {
            const int hA = pv_half<D>(0), eA = pv_elem<D>(mt, 0);
            const int hB = pv_half<D>(1), eB = pv_elem<D>(mt, 1);
            const uint32_t sA = (eA & 1) ? 0x7632u : 0x5410u, sB = (eB & 1) ? 0x7632u : 0x5410u;
            const uint32_t a0 = __byte_perm(vw[0][hA][eA >> 1], vw[1][hA][eA >> 1], sA);
            const uint32_t a1 = __byte_perm(vw[0][hB][eB >> 1], vw[1][hB][eB >> 1], sB);
            const uint32_t a2 = __byte_perm(vw[2][hA][eA >> 1], vw[3][hA][eA >> 1], sA);
            const uint32_t a3 = __byte_perm(vw[2][hB][eB >> 1], vw[3][hB][eB >> 1], sB);
            mma_bf16(st.o[mt], a0, a1, a2, a3, b0, b1);
            mma_bf16(st.o[mt], a0, a1, a2, a3, c0, c1);
        }
    }
}

// Reduce the denominators over the lanes of a head pair, then publish this
// warp's (m, l, o) for the G heads into CTA scratch.
template <int D, int G>
__device__ __forceinline__ void warp_publish(WarpState<D> &st, bool has_work, int lane, int warp, float *cm,
                                             float *cl, float *co) {
    const int g = lane >> 2, t = lane & 3;
    float l[2] = {st.l[0], st.l[1]};
#pragma unroll
    for (int dist = 4; dist < 32; dist <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], dist);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], dist);
    }
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        const int h = 2 * t + hi;
        if (h < G) {
            float *dst = co + (warp * G + h) * D;
            float r[2][8];
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) r[pv_half<D>(rr)][pv_elem<D>(mt, rr)] = st.o[mt][2 * rr + hi];
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh) {
                float4 *d4 = reinterpret_cast<float4 *>(dst + hh * 64 + g * 8);
                d4[0] = make_float4(r[hh][0], r[hh][1], r[hh][2], r[hh][3]);
                d4[1] = make_float4(r[hh][4], r[hh][5], r[hh][6], r[hh][7]);
            }
            if (g == 0) {
                cm[warp * G + h] = has_work ? st.m[hi] : -INFINITY;
                cl[warp * G + h] = has_work ? l[hi] : 0.f;
            }
        }
    }
}

// The prefix terms of the (head, dim pair) items a thread finishes in
// cta_combine_store: item idx = threadIdx.x + it * kWarps * 32.
template <int D, int G>
struct CombinePrefix {
    static constexpr int kItems = G * D / 2;
    static constexpr int kIt = (kItems + kWarps * 32 - 1) / (kWarps * 32);
    PrefixTerm<2> t[kIt];
    __device__ __forceinline__ void load(const Params &p, size_t row0, bool want) {
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int idx = threadIdx.x + it * kWarps * 32;
            t[it] = load_prefix<2>(p, row0 + idx / (D / 2), D, (idx % (D / 2)) * 2, want && idx < kItems);
        }
    }
};

// Combine the kWarps warps' (m, l, o) for G heads (blockDim.x = kWarps * 32);
// write bf16 rows to `out_rows` (final, with the prefix terms folded in) or
// fp32 partials: o normalised by l at o_base + h*o_hs, (m, l) at ml_base + h*ml_hs.
template <int D, int G>
__device__ __forceinline__ void cta_combine_store(const CombinePrefix<D, G> &pre, const float *cm, const float *cl,
                                                  const float *co, bool final, __nv_bfloat16 *out_rows, float *o_base,
                                                  size_t o_hs, float *ml_base, size_t ml_hs) {
    using CP = CombinePrefix<D, G>;
#pragma unroll
    for (int it = 0; it < CP::kIt; ++it) {
        const int idx = threadIdx.x + it * kWarps * 32;
        if (idx >= CP::kItems) break;
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
        if (final) {
            float acc[2] = {ox, oy};
            fold_prefix<2>(pre.t[it], M, lsum, acc);
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            reinterpret_cast<uint32_t *>(out_rows + h * D + i)[0] = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        } else {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            *reinterpret_cast<float2 *>(o_base + h * o_hs + i) = make_float2(ox * inv, oy * inv);
            if (i == 0) *reinterpret_cast<float2 *>(ml_base + h * ml_hs) = make_float2(M, lsum);
        }
    }
}

// ---- split-context partition kernel --------------------------------------------

template <int D, int G, int BS>
__global__ void __launch_bounds__(kWarps * 32, kMinCtas)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const Params p) {
    using S = Shape<D, BS>;
    using WR = WarpRing<D, BS, kStages>;
    using SP = SmemPlan<D, BS, kStages>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = align1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring = smem_addr(smem) + warp * (uint32_t)sizeof(WR);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + SP::kRings) + warp * kStages;

    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(&bar[st], 1);
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
            for (int i = threadIdx.x; i < G * D / 2; i += blockDim.x) {
                float acc[2] = {0.f, 0.f}, wsum = 0.f;
                fold_prefix<2>(load_prefix<2>(p, head0 + i / (D / 2), D, (i % (D / 2)) * 2), -INFINITY, wsum, acc);
                const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
                reinterpret_cast<uint32_t *>(p.out + head0 * D)[i] = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            }
        return;
    }

    uint32_t qf[D / 8];
    load_qf<D, G, false>(qf, p.q + head0 * D, lane);
    __syncwarp();
    CombinePrefix<D, G> pre;   // loaded now, used after the last stage
    pre.load(p, head0, p.num_parts == 1);

    const int nblk_seq = (L + BS - 1) / BS;
    const int nstages = (ntok + S::TPS - 1) / S::TPS;
    const int my_stages = nstages > warp ? (nstages - warp + kWarps - 1) / kWarps : 0;
    const int32_t *table_row = p.tables + (size_t)s * p.max_blocks;

    // Register cache of block ids: lane i holds warp-local block kb_base + i,
    // where warp-local block kb = k * BPS + ib is block ib of the warp's k-th stage.
    int kb_base = 0;
    auto load_ids = [&](int base) -> int {
        const int kb = base + lane;
        const int k = kb / S::BPS, ib = kb % S::BPS;
        const int logical = S::block_of(tok_begin + (warp + k * kWarps) * S::TPS, ib);
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
        const int stok = tok_begin + (warp + k * kWarps) * S::TPS;   // the stage's first token
        const int nvalid = min(S::BPS, nblk_seq - S::block_of(stok, 0));
        const int c_slot = S::slot_of(stok);
        int ids[S::BPS];
#pragma unroll
        for (int ib = 0; ib < S::BPS; ++ib) ids[ib] = __shfl_sync(0xffffffffu, id_cache, k * S::BPS + ib - kb_base);
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar[slot], (uint32_t)(nvalid * S::BOX * 2));
            const uint32_t kslot = ring + slot * S::SLOT, vslot = ring + (kStages + slot) * S::SLOT;
#pragma unroll
            for (int ib = 0; ib < S::BPS; ++ib) {
                if (ib < nvalid) {
                    tensor_copy_5d(kslot + ib * S::REGION, &tmk, 0, c_slot, 0, g, ids[ib], &bar[slot]);
                    tensor_copy_5d(vslot + ib * S::REGION, &tmv, 0, c_slot, 0, g, ids[ib], &bar[slot]);
                }
            }
        }
    };

#pragma unroll
    for (int k = 0; k < kStages; ++k) issue(k);

    WarpState<D> st;
    st.reset();
    int consumed = 0;
    bool ok = true;
    for (int k = 0; k < my_stages; ++k) {
        const int slot = k % kStages;
        const bool arrived = mbar_wait_bounded(&bar[slot], (uint32_t)((k / kStages) & 1), p.err);
        if (!__all_sync(0xffffffffu, arrived)) {
            ok = false;
            break;
        }
        consumed = k + 1;
        const int tok0 = tok_begin + (warp + k * kWarps) * S::TPS;
        stage_compute<D, G, BS>(ring + slot * S::SLOT, ring + (kStages + slot) * S::SLOT, qf, tok0, tok_end,
                                p.scale_log2, lane, st);
        __syncwarp();   // every lane is done with the slot before it is refilled
        issue(k + kStages);
    }

    if (!ok) {
        // A wait gave up: wait (bounded) for the copies still in flight into
        // this warp's slots before the shared memory is reused.
        const int issued = min(my_stages, consumed + kStages);
        for (int k = consumed; k < issued; ++k)
            mbar_wait_bounded(&bar[k % kStages], (uint32_t)((k / kStages) & 1), p.err);
    }

    // ---- merge the warps in shared memory (stage buffers are free now)
    __syncthreads();
    float *cm = reinterpret_cast<float *>(smem);       // [W][G] running max
    float *cl = cm + kWarps * G;                       // [W][G] denominators
    float *co = cl + kWarps * G;                       // [W][G][D] numerators
    warp_publish<D, G>(st, my_stages > 0, lane, warp, cm, cl, co);
    __syncthreads();
    grid_launch_dependents();
    const size_t rowp = head0 * p.num_parts + part;
    cta_combine_store<D, G>(pre, cm, cl, co, p.num_parts == 1, p.out + head0 * D, p.ws_o + rowp * D,
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
    const PrefixTerm<4> pre = load_prefix<4>(p, row, D, i);
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
    float a4[4] = {acc.x, acc.y, acc.z, acc.w};
    fold_prefix<4>(pre, M, wsum, a4);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2 packed = make_uint2(pack_bf16x2(a4[0] * inv, a4[1] * inv), pack_bf16x2(a4[2] * inv, a4[3] * inv));
    *reinterpret_cast<uint2 *>(p.out + row * D + i) = packed;
}

// ---- stream-K kernel -------------------------------------------------------------

// Stages of one sequence (one kv-head); lengths validated as in effective_len.
template <int BS>
__device__ __forceinline__ int seq_stages(const Params &p, int s, bool report) {
    constexpr int TPS = 16;
    const int L = effective_len(p, s, BS, report);
    return (L + TPS - 1) / TPS;
}

// Length of one unit of a sequence with ns stages in the balanced schedule's
// work order: its stages, then kUnitCost stages of no work (none if empty).
__device__ __forceinline__ int unit_span(int ns) { return ns > 0 ? ns + kUnitCost : 0; }

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
__global__ void __launch_bounds__(kWarps * 32, kMinCtas)
    paged_decode_sk_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                           const Params p) {
    using S = Shape<D, BS>;
    using WR = WarpRing<D, BS, kSkStages>;
    using SP = SmemPlan<D, BS, kSkStages>;
    using SK = SkSmem<D, G>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = align1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const uint32_t ring = smem_addr(smem) + warp * (uint32_t)sizeof(WR);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + SP::kRings) + warp * kSkStages;
    SK *sk = reinterpret_cast<SK *>(smem + SP::kRings + SP::kBars);
    constexpr int NT = kWarps * 32;
    const int Hkv = p.num_kv_heads, B = p.num_seqs, c = blockIdx.x;

    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < kSkStages; ++st) mbar_init(&bar[st], 1);
        if (warp == 0) {
            mbar_init(&sk->qbar[0], 1);
            mbar_init(&sk->qbar[1], 1);
        }
        fence_barrier_init();
    }
    // With early_meta (one-pass listing only) the lengths and the table are
    // read, and the first listing made, while the previous kernel in the
    // stream finishes; q, the pool and the workspace are touched only after
    // griddepcontrol.wait.
    const bool one_pass = B <= NT;
    bool waited = !p.early_meta;
    if (waited) grid_dependency_wait();

    // ---- total work W (unit spans over all units) and this CTA's range [gs, ge)
    // With at most NT sequences (one per thread) each thread keeps its
    // sequence's stage count and first global stage for the listing below.
    int my_ns = 0, my_first = 0;
    int total = 0;
    for (int base = 0; base < B; base += NT) {
        const int s = base + tid;
        const int ns = s < B ? seq_stages<BS>(p, s, c == 0) : 0;
        const int v = Hkv * unit_span(ns);
        int chunk;
        const int inc = block_inclusive_scan(v, sk->scan, chunk);
        my_ns = ns;
        my_first = total + inc - v;
        total += chunk;
    }
    auto wait_inputs = [&]() {   // the deferred wait (early_meta)
        if (waited) return;
        grid_dependency_wait();
        waited = true;
    };
    const int per = (total + p.num_ctas - 1) / p.num_ctas;
    const int gs = min(total, c * per), ge = min(total, gs + per);
    if (gs >= ge) {          // nothing issued, nothing to wait for
        wait_inputs();       // the kernels before this one finish before the merge kernel starts
        return;
    }

    // ---- the sequence whose units contain gs (the serial listing's start)
    if (!one_pass) {
        int run = 0;
        for (int base = 0; base < B; base += NT) {
            const int s = base + tid;
            const int v = s < B ? Hkv * unit_span(seq_stages<BS>(p, s, false)) : 0;
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
    int pos = gs;                                              // work position the next listing starts at
    int kq = 0;                  // stages this warp has consumed (ring parity counter)
    int jbase = 0;               // segments of earlier listings (q buffer parity counter)
    bool ok = true;
    bool first_seg = true;

    while (pos < ge && ok) {
        // ---- list up to kMaxSegs segments of units covering [pos, ge)
        if (one_pass) {
            // every thread lists the units of its own sequence whose stages
            // meet [pos, ge); block scans of their counts and stage counts
            // give the slots and the local stage offsets
            const int span = unit_span(my_ns), v = Hkv * span;
            int g_lo = 0, n = 0;
            if (my_ns > 0 && my_first < ge && my_first + v > pos) {
                const int off = max(pos, my_first) - my_first;
                g_lo = off / span;
                if (off - g_lo * span >= my_ns) ++g_lo;   // pos inside a unit's tail of no work
                const int g_hi = (min(ge, my_first + v) - 1 - my_first) / span;
                n = max(0, g_hi - g_lo + 1);
            }
            int r = 0;   // stages of those units inside [pos, ge)
            for (int k = 0; k < n; ++k) {
                const int u0 = my_first + (g_lo + k) * span;
                r += min(ge, u0 + my_ns) - max(pos, u0);
            }
            int nall, rall;
            const int base = block_inclusive_scan(n, sk->scan, nall) - n;
            int local = block_inclusive_scan(r, sk->scan, rall) - r;
            for (int k = 0; k < n; ++k) {
                const int idx = base + k;
                if (idx > kMaxSegs) break;
                const int u0 = my_first + (g_lo + k) * span;   // work position of the unit's start
                const int a = max(pos, u0), b = min(ge, u0 + my_ns);
                if (idx == kMaxSegs) {        // first unit of the next listing
                    sk->seg_lb[kMaxSegs] = local;
                    sk->next_pos = a;
                    break;
                }
                sk->seg_s[idx] = tid;   // one pass: thread tid holds sequence tid
                sk->seg_g[idx] = g_lo + k;
                sk->seg_kb[idx] = a - u0;
                sk->seg_ke[idx] = b - u0;
                sk->seg_lb[idx] = local;
                local += b - a;
            }
            if (tid == 0) {
                sk->nseg = min(nall, kMaxSegs);
                sk->more = nall > kMaxSegs ? 1 : 0;
                if (nall <= kMaxSegs) {
                    sk->seg_lb[nall] = rall;
                    sk->next_pos = ge;
                }
            }
        } else if (tid == 0) {
            // walk the units from the one holding pos: `done` counts work
            // positions consumed (stages and unit tails), `local` stages listed
            int n = 0, s = cur_s, rem = cur_rem, local = 0, done = 0;
            const int len = ge - pos;
            while (done < len && n < kMaxSegs && s < B) {
                const int ns = seq_stages<BS>(p, s, false);
                if (ns == 0) {
                    ++s;
                    rem = 0;
                    continue;
                }
                const int span = unit_span(ns);
                const int gg = rem / span, kb = rem % span;
                int step;
                if (kb >= ns) {          // inside the unit's tail of no work
                    step = min(span - kb, len - done);
                } else {
                    const int take = min(ns - kb, len - done);
                    sk->seg_s[n] = s;
                    sk->seg_g[n] = gg;
                    sk->seg_kb[n] = kb;
                    sk->seg_ke[n] = kb + take;
                    sk->seg_lb[n] = local;
                    ++n;
                    local += take;
                    step = take;
                }
                done += step;
                rem += step;
                if (rem >= Hkv * span) {
                    ++s;
                    rem = 0;
                }
            }
            sk->seg_lb[n] = local;
            sk->nseg = n;
            sk->more = (done < len && s < B) ? 1 : 0;
            sk->next_pos = pos + done;
            sk->found_s = s;          // where the next listing resumes
            sk->found_base = rem;
        }
        __syncthreads();
        const int nseg = sk->nseg, nlocal = sk->seg_lb[nseg];
        cur_s = sk->found_s;
        cur_rem = sk->found_base;
        if (nseg == 0) break;

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
                const int logical = S::block_of((sk->seg_kb[j] + i - sk->seg_lb[j]) * S::TPS, ib);
                const int L = effective_len(p, s, BS, false);
                if (logical < (L + BS - 1) / BS) {
                    id = __ldg(p.tables + (size_t)s * p.max_blocks + logical);
                    if (id < 0 || id >= p.num_blocks) {
                        raise_error(p.err, PA_DEVERR_BLOCK_ID);
                        id = -2;   // not fetched, not written
                    }
                } else {
                    id = -1;   // past the sequence end: not fetched
                }
            }
            return id;
        };
        int id_cache = load_ids(0);
        if (!waited) {
            // The previous kernel may still be writing the pool (the slot
            // writer does) or q: the first segments' q rows and the first
            // stages' boxes go to L2 now, as a hint, and their copies after the
            // wait find them there.
            if (tid < 2 && tid < nseg) {
                const size_t head0 = (size_t)sk->seg_s[tid] * p.num_q_heads + (size_t)sk->seg_g[tid] * G;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.q + head0 * D),
                             "r"((uint32_t)(G * D * 2))
                             : "memory");
            }
#pragma unroll 1
            for (int k = 0; k < kSkPrefetch && k < my_n && (k + 1) * S::BPS <= 32; ++k) {
                const int i = warp + k * kWarps;
                int j = 0;
                while (j + 1 < nseg && sk->seg_lb[j + 1] <= i) ++j;
                const int g = sk->seg_g[j];
                const int c_slot = S::slot_of((sk->seg_kb[j] + i - sk->seg_lb[j]) * S::TPS);
#pragma unroll
                for (int ib = 0; ib < S::BPS; ++ib) {
                    const int id = __shfl_sync(0xffffffffu, id_cache, k * S::BPS + ib);
                    if (lane == 0 && id >= 0) {
                        tensor_prefetch_l2_5d(&tmk, 0, c_slot, 0, g, id);
                        tensor_prefetch_l2_5d(&tmv, 0, c_slot, 0, g, id);
                    }
                }
            }
        }
        wait_inputs();

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
            const int tok0 = (sk->seg_kb[j] + i - sk->seg_lb[j]) * S::TPS;
            const int c_slot = S::slot_of(tok0);
            const int slot = (kq + k) % kSkStages;
            int ids[S::BPS];
#pragma unroll
            for (int ib = 0; ib < S::BPS; ++ib)
                ids[ib] = __shfl_sync(0xffffffffu, id_cache, k * S::BPS + ib - kb_base);
            if (p.new_k != nullptr) {
                // the stage holding the sequence's last token stores that token's
                // K and V first; the copy below then reads them back from the pool
                const int s = sk->seg_s[j];
                const int L = __ldg(p.seq_lens + s), last = L - 1;   // an out-of-range length writes nothing
                if (L <= min(p.max_blocks * BS, p.num_parts * p.part_tokens) && last >= tok0 &&
                    last < tok0 + S::TPS) {
                    const int ib = BS < 16 ? last / BS - tok0 / BS : 0;
                    int blk = 0;
#pragma unroll
                    for (int x = 0; x < S::BPS; ++x) blk = x == ib ? ids[x] : blk;
                    if (blk >= 0) {
                        constexpr int CH = D / 8;   // 16-byte chunks per row
                        const int half = lane / CH, c16 = lane % CH;
                        if (half < 2) {
                            const __nv_bfloat16 *src = (half == 0 ? p.new_k : p.new_v) +
                                                       ((size_t)s * p.num_kv_heads + g) * D + c16 * 8;
                            __nv_bfloat16 *dst = p.pool + (size_t)blk * p.block_stride + half * p.kv_stride +
                                                 ((size_t)g * BS + last % BS) * D + c16 * 8;
                            *reinterpret_cast<uint4 *>(dst) = __ldg(reinterpret_cast<const uint4 *>(src));
                        }
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        __syncwarp();
                    }
                }
            }
            if (lane == 0) {
                int nvalid = 0;
#pragma unroll
                for (int ib = 0; ib < S::BPS; ++ib) nvalid += ids[ib] >= 0 ? 1 : 0;
                mbar_arrive_expect_tx(&bar[slot], (uint32_t)(nvalid * S::BOX * 2));
                const uint32_t kslot = ring + slot * S::SLOT, vslot = ring + (kSkStages + slot) * S::SLOT;
#pragma unroll
                for (int ib = 0; ib < S::BPS; ++ib) {
                    if (ids[ib] >= 0) {
                        tensor_copy_5d(kslot + ib * S::REGION, &tmk, 0, c_slot, 0, g, ids[ib], &bar[slot]);
                        tensor_copy_5d(vslot + ib * S::REGION, &tmv, 0, c_slot, 0, g, ids[ib], &bar[slot]);
                    }
                }
            }
        };
#pragma unroll
        for (int k = 0; k < kSkStages; ++k) issue(k);
        // the merge kernel may start now: it sums the lengths, then waits for this grid
        grid_launch_dependents();

        int k = 0;   // this warp's next stage in this listing
        for (int j = 0; j < nseg; ++j) {
            const int s = sk->seg_s[j], g = sk->seg_g[j];
            const int L = effective_len(p, s, BS, false);
            const int ns = (L + S::TPS - 1) / S::TPS;
            const bool complete = sk->seg_kb[j] == 0 && sk->seg_ke[j] == ns;
            const size_t head0 = (size_t)s * p.num_q_heads + (size_t)g * G;
            CombinePrefix<D, G> pre;   // loaded now, used at the segment's end
            pre.load(p, head0, complete);
            const int jg = jbase + j;
            const bool qok = mbar_wait_bounded(&sk->qbar[jg & 1], (uint32_t)((jg >> 1) & 1), p.err);
            if (!__syncthreads_and(qok)) {
                ok = false;
                break;
            }
            uint32_t qf[D / 8];
            load_qf<D, G, true>(qf, sk->q[jg & 1], lane);
            WarpState<D> st;
            st.reset();
            const int lend = sk->seg_lb[j + 1];
            int done = 0;
            while (ok && k < my_n && warp + k * kWarps < lend) {
                const int i = warp + k * kWarps;
                const int slot = (kq + k) % kSkStages;
                const bool arrived =
                    mbar_wait_bounded(&bar[slot], (uint32_t)(((kq + k) / kSkStages) & 1), p.err);
                if (!__all_sync(0xffffffffu, arrived)) {
                    ok = false;
                    break;
                }
                const int tok0 = (sk->seg_kb[j] + i - sk->seg_lb[j]) * S::TPS;
                stage_compute<D, G, BS>(ring + slot * S::SLOT, ring + (kSkStages + slot) * S::SLOT, qf, tok0, L,
                                        p.scale_log2, lane, st);
                __syncwarp();   // every lane is done with the slot before it is refilled
                issue(k + kSkStages);
                ++k;
                ++done;
            }
            warp_publish<D, G>(st, done > 0, lane, warp, sk->cm, sk->cl, sk->co);
            if (!__syncthreads_and(ok)) {
                ok = false;
                break;
            }
            const bool is_first = first_seg && j == 0;
            const int rec = 2 * c + (is_first ? 0 : 1);
            cta_combine_store<D, G>(pre, sk->cm, sk->cl, sk->co, complete, p.out + head0 * D,
                                    p.ws_o + (size_t)rec * G * D, D, p.ws_ml + (size_t)rec * G * 2, 2);
            __syncthreads();   // scratch and this q buffer are free again
            if (tid == 0) issue_q(j + 2);
        }
        if (!ok) {
            // A wait gave up: bounded waits for this warp's copies still in flight.
            const int issued = min(my_n, k + kSkStages);
            for (int kk = k; kk < issued; ++kk)
                mbar_wait_bounded(&bar[(kq + kk) % kSkStages], (uint32_t)(((kq + kk) / kSkStages) & 1), p.err);
            break;
        }
        kq += my_n;
        jbase += nseg;
        pos = sk->next_pos;
        first_seg = false;
        if (!sk->more) break;
        __syncthreads();
    }
    wait_inputs();   // only if no segment was listed
    grid_launch_dependents();
}

// Finish the stream-K schedule.  grid (num_ctas), kWarps * 32 threads: block c
// merges the unit that the start of decode CTA c's range cuts, when that is
// the unit's first cut (a unit cut several times is merged by the block of its
// first cut, from the records of every CTA it spans), and writes the rows of
// the sequences with no keys among s = c, c + num_ctas, ...: zeros, or the
// prefix term alone.  A unit that one CTA completed needs nothing here.
// The unit is located from the lengths, before griddepcontrol.wait: each
// thread sums the unit spans of a slice of the sequences and a block scan
// gives the slices' starts.  The decode kernel this one follows never writes
// the lengths, and every decode CTA waited for the kernels before it.
// With one block per decode CTA (at most two per SM) the whole grid fits
// beside the running decode CTAs, so its blocks wait resident and release no
// SM late; the next kernel's CTAs take the SMs the decode CTAs leave.
#ifndef PA_MERGE_THREADS
#define PA_MERGE_THREADS 128
#endif
#ifndef PA_MERGE_MIN_BLOCKS
#define PA_MERGE_MIN_BLOCKS 10
#endif
constexpr int kMergeThreads = PA_MERGE_THREADS;
// Registers: two stream-K CTAs leave 65536 - 2 * 128 * 200 = 14336 per SM,
// room for two merge blocks of 128 threads at 56 registers.  The bound of 10
// blocks a SM caps them at 48 (one spilled word), which leaves slack for an
// uneven placement of warps: at 56, some SMs kept the next call's decode CTAs
// waiting for merge blocks to exit (34.93 against 34.43 us a call on the
// Llama-shaped batch).
template <int D, int G, int BS>
__global__ void __launch_bounds__(kMergeThreads, PA_MERGE_MIN_BLOCKS) paged_decode_sk_merge_kernel(const Params p) {
    grid_launch_dependents();   // the next kernel waits for this grid's completion before using its data
    constexpr int NT = kMergeThreads, NW = NT / 32;
    __shared__ int scan[NW];
    __shared__ int found[3];    // sequence, kv-head and work position of the unit to merge (sequence -1: none)
    const int c = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.num_seqs, Hkv = p.num_kv_heads, C = p.num_ctas;
    const int per_thread = (B + NT - 1) / NT;
    const int s0 = min(B, tid * per_thread), s1 = min(B, s0 + per_thread);
    int mine = 0;
    for (int s = s0; s < s1; ++s) mine += Hkv * unit_span(seq_stages<BS>(p, s, false));
    int inc = mine;   // block scan of the slices' spans
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += u;
    }
    if (lane == 31) scan[warp] = inc;
    if (tid == 0) found[0] = -1;
    __syncthreads();
    int total = 0, excl = inc - mine;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        total += scan[w];
        excl += w < warp ? scan[w] : 0;
    }
    const int per = (total + C - 1) / C;
    const int P = c * per;   // the start of decode CTA c's range
    if (c > 0 && P < total && excl <= P && P < excl + mine) {
        int run = excl;
        for (int s = s0; s < s1; ++s) {
            const int ns = seq_stages<BS>(p, s, false);
            const int span = unit_span(ns), v = Hkv * span;
            if (P < run + v) {
                const int g = (P - run) / span, kb = (P - run) % span, u0 = run + g * span;
                // P falls after the unit's first stage and on one of its stages,
                // and the unit starts in CTA c - 1's range: its first cut
                if (kb >= 1 && kb < ns && u0 >= (c - 1) * per) {
                    found[0] = s;
                    found[1] = g;
                    found[2] = u0;
                }
                break;
            }
            run += v;
        }
    }
    __syncthreads();
    grid_dependency_wait();
    if (found[0] >= 0) {
        const int s = found[0], g = found[1], u0 = found[2];
        const int ns = seq_stages<BS>(p, s, false);
        const int ca = u0 / per, cb = (u0 + ns - 1) / per;
        // the unit is CTA ca's first segment unless a stage of the unit before
        // it (which ends kUnitCost positions before u0) lies in that CTA's range
        const int first_rec = (u0 - ca * per > kUnitCost) ? 1 : 0;
        const size_t row0 = (size_t)s * p.num_q_heads + (size_t)g * G;
        // A thread's items (head, four dims) and up to kR records per pass are
        // loaded before any is combined, so a pass costs one memory round trip;
        // passes merge online (running maximum, rescaled sums).
        constexpr int kItems = G * D / 4, kAll = (kItems + NT - 1) / NT, kIt = kAll < 2 ? kAll : 2, kR = 2;
#pragma unroll 1
        for (int t0 = 0; t0 < kAll; t0 += kIt) {
        float M[kIt], wsum[kIt], acc[kIt][4];
#pragma unroll
        for (int t = 0; t < kIt; ++t) {
            M[t] = -INFINITY;
            wsum[t] = 0.f;
            acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
        }
        for (int c0 = ca; c0 <= cb; c0 += kR) {
            float2 ml[kIt][kR];
            float4 ov[kIt][kR];
#pragma unroll
            for (int t = 0; t < kIt; ++t) {
                const int it = tid + (t0 + t) * NT, h = it / (D / 4), i = (it % (D / 4)) * 4;
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const int cc = c0 + r;
                    ml[t][r] = make_float2(-INFINITY, 0.f);
                    ov[t][r] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (it < kItems && cc <= cb) {
                        const size_t rec = 2 * (size_t)cc + (cc == ca ? first_rec : 0);
                        ml[t][r] = *reinterpret_cast<const float2 *>(p.ws_ml + (rec * G + h) * 2);
                        ov[t][r] = *reinterpret_cast<const float4 *>(p.ws_o + (rec * G + h) * D + i);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kIt; ++t) {
                float Mn = M[t];
#pragma unroll
                for (int r = 0; r < kR; ++r) Mn = fmaxf(Mn, ml[t][r].x);
                if (Mn == -INFINITY) continue;
                const float f = M[t] == -INFINITY ? 0.f : fast_exp2(M[t] - Mn);
                wsum[t] *= f;
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[t][k] *= f;
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const float w = ml[t][r].x == -INFINITY ? 0.f : ml[t][r].y * fast_exp2(ml[t][r].x - Mn);
                    wsum[t] += w;
                    acc[t][0] += w * ov[t][r].x;
                    acc[t][1] += w * ov[t][r].y;
                    acc[t][2] += w * ov[t][r].z;
                    acc[t][3] += w * ov[t][r].w;
                }
                M[t] = Mn;
            }
        }
#pragma unroll
        for (int t = 0; t < kIt; ++t) {
            const int it = tid + (t0 + t) * NT;
            if (it >= kItems) continue;
            const int h = it / (D / 4), i = (it % (D / 4)) * 4;
            const size_t row = row0 + h;
            fold_prefix<4>(load_prefix<4>(p, row, D, i), M[t], wsum[t], acc[t]);
            const float inv = wsum[t] > 0.f ? 1.f / wsum[t] : 0.f;
            *reinterpret_cast<uint2 *>(p.out + row * D + i) =
                make_uint2(pack_bf16x2(acc[t][0] * inv, acc[t][1] * inv), pack_bf16x2(acc[t][2] * inv, acc[t][3] * inv));
        }
        }
    }
    // sequences with no keys of their own: zero rows, or the prefix term alone
    for (int s = c; s < B; s += C) {
        if (seq_stages<BS>(p, s, false) != 0) continue;
        for (int it = tid; it < p.num_q_heads * (D / 4); it += NT) {
            const size_t row = (size_t)s * p.num_q_heads + it / (D / 4);
            const int i = (it % (D / 4)) * 4;
            float a4[4] = {0.f, 0.f, 0.f, 0.f}, wsum = 0.f;
            fold_prefix<4>(load_prefix<4>(p, row, D, i), -INFINITY, wsum, a4);
            const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
            *reinterpret_cast<uint2 *>(p.out + row * D + i) =
                make_uint2(pack_bf16x2(a4[0] * inv, a4[1] * inv), pack_bf16x2(a4[2] * inv, a4[3] * inv));
        }
    }
}

// ---- launchers -----------------------------------------------------------------

// Launch with programmatic stream serialisation (the kernel waits on
// griddepcontrol.wait before touching global memory).
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const Args &...args) {
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
    return cudaLaunchKernelEx(&cfg, kernel, args...);
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
    return SmemPlan<D, BS, kSkStages>::bytes(sizeof(SkSmem<D, G>));
}

template <int D, int G, int BS>
cudaError_t launch_shape(const CUtensorMap &tmk, const CUtensorMap &tmv, const Params &prm, int num_kv_heads,
                         int num_seqs, bool stream_k, cudaStream_t stream) {
    if (stream_k) {
        constexpr size_t smem = sk_smem_bytes<D, G, BS>();
        static bool configured[64] = {};
        cudaError_t e = ensure_smem(paged_decode_sk_kernel<D, G, BS>, smem, configured);
        if (e != cudaSuccess) return e;
        e = launch_pdl(paged_decode_sk_kernel<D, G, BS>, dim3(prm.num_ctas), dim3(kWarps * 32), smem, stream, tmk,
                       tmv, prm);
        if (e != cudaSuccess) return e;
        return launch_pdl(paged_decode_sk_merge_kernel<D, G, BS>, dim3(prm.num_ctas), dim3(kMergeThreads), 0, stream,
                          prm);
    }
    using SP = SmemPlan<D, BS, kStages>;
    constexpr size_t smem = SP::bytes(0);
    static_assert(SP::kRings >= sizeof(float) * kWarps * G * (D + 2), "combine scratch");
    static bool configured[64] = {};
    cudaError_t e = ensure_smem(paged_decode_kernel<D, G, BS>, smem, configured);
    if (e != cudaSuccess) return e;
    e = launch_pdl(paged_decode_kernel<D, G, BS>, dim3(prm.num_parts, num_kv_heads, num_seqs), dim3(kWarps * 32),
                   smem, stream, tmk, tmv, prm);
    if (e != cudaSuccess || prm.num_parts == 1) return e;
    return launch_pdl(paged_decode_reduce_kernel<D, G, BS>, dim3(num_kv_heads, num_seqs), dim3(G * D / 4), 0,
                      stream, prm);
}

template <int D, int G>
cudaError_t launch_group(const CUtensorMap &tmk, const CUtensorMap &tmv, const Params &prm, int bs, int num_kv_heads,
                         int num_seqs, bool stream_k, cudaStream_t stream) {
    switch (bs) {
        case 4: return launch_shape<D, G, 4>(tmk, tmv, prm, num_kv_heads, num_seqs, stream_k, stream);
        case 8: return launch_shape<D, G, 8>(tmk, tmv, prm, num_kv_heads, num_seqs, stream_k, stream);
        case 16: return launch_shape<D, G, 16>(tmk, tmv, prm, num_kv_heads, num_seqs, stream_k, stream);
        case 32: return launch_shape<D, G, 32>(tmk, tmv, prm, num_kv_heads, num_seqs, stream_k, stream);
        case 64: return launch_shape<D, G, 64>(tmk, tmv, prm, num_kv_heads, num_seqs, stream_k, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_for_dim(const DecodeArgs &a, cudaStream_t stream) {
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    CUtensorMap tmk, tmv;
    const int rows = a.pool.block_size < 16 ? a.pool.block_size : 16;   // slots per copy box
    cudaError_t e = encode_pool_block_map(&tmk, a.pool, 0, rows);
    if (e != cudaSuccess) return e;
    e = encode_pool_block_map(&tmv, a.pool, 1, rows);
    if (e != cudaSuccess) return e;
    Params prm;
    prm.out = static_cast<__nv_bfloat16 *>(a.out);
    prm.q = static_cast<const __nv_bfloat16 *>(a.q);
    prm.num_blocks = a.pool.num_blocks;
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
    prm.num_ctas = a.num_ctas;
    prm.early_meta = a.early_meta ? 1 : 0;
    prm.new_k = static_cast<const __nv_bfloat16 *>(a.new_k);
    prm.pre_o = a.pre_o;
    prm.pre_lse = a.pre_lse;
    prm.new_v = static_cast<const __nv_bfloat16 *>(a.new_v);
    prm.pool = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.pool.base));
    prm.block_stride = a.pool.block_stride;
    prm.kv_stride = a.pool.kv_stride;
    prm.err = err;
    const int G = a.num_q_heads / a.pool.num_kv_heads;
    const int bs = a.pool.block_size, H = a.pool.num_kv_heads, B = a.num_seqs;
    const bool sk = a.stream_k;
    switch (G) {
        case 1: return launch_group<D, 1>(tmk, tmv, prm, bs, H, B, sk, stream);
        case 2: return launch_group<D, 2>(tmk, tmv, prm, bs, H, B, sk, stream);
        case 4: return launch_group<D, 4>(tmk, tmv, prm, bs, H, B, sk, stream);
        case 8: return launch_group<D, 8>(tmk, tmv, prm, bs, H, B, sk, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace decode
}  // namespace pa
