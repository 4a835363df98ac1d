// pa_prefill.cu -- chunked causal prefill against a paged context on the
// tcgen05 tensor cores (sm_103a).
//
// What it computes: for sequence s with ctx cached tokens and a chunk of C new
// query tokens at positions ctx .. ctx + C - 1 (whose K/V are already in the
// pool), query j of head h attends keys 0 .. ctx + j of kv-head h / G, read
// through the block table (table[s][t / b], t % b).  Sources:
// auto-20261007-1900-en (lihaoran.work), "A block table maps logical order to
// physical storage" (paging changes where K/V live, not what a causal query
// sees); attn-paged-attention-mcq-hard (zenaique.com), conceptual block-lookup
// listing (the gather belongs inside the kernel's tiling loop).
//
// The same kernel, without the causal mask, runs the shared-prefix pass of a
// cascade decode: sequence s stands for a group of C sequences that share
// their first ctx_lens[s] tokens (whole blocks, one table), its "chunk" holds
// the C sequences' decode queries, and every query sees all ctx_lens[s] keys.
// That pass writes fp32 output normalised by l together with each row's
// log-sum-exp, which the decode of the private suffixes folds in.
//
// Design:
//  * Work comes in units of one 128-row M-tile of one (sequence, kv-head): row
//    r is query j0 + r / G of head g*G + r % G, so every K/V tile staged in
//    shared memory serves the whole query group.  The grid is persistent (one
//    CTA per SM); each CTA walks its units in rounds of alternating direction,
//    its copy and tensor-core pipeline running on from one unit into the next.
//  * Twelve warps: eight softmax warps in two warpgroups each own 64 of a
//    row's 128 keys (tensor-memory lanes follow warp % 4); lane 0 of one warp
//    issues the Q.K MMAs and lane 0 of another the P.V MMAs, so each runs
//    ahead as far as its own inputs allow; a K warp and a V warp issue the
//    tensor copies, one lane per box.
//  * TMA (cp.async.bulk.tensor, 128-byte swizzle) brings Q and the K/V tiles.
//    A K tile of 128 keys is 8 blocks x 2 halves of d, one box of 16 rows x
//    64 dims per (block, half) through a 5-D tensor map of the pool's
//    (d, slot, head, K|V, block) view, laid out [half][128 keys][128 B] (the
//    Q.K operand needs a uniform 8-row stride over the tile).  A V tile is one
//    4 KiB box per block, laid out [block][half][16 keys][128 B] (each 16-key
//    P.V step is one block).  Blocks past the sequence end, or with an
//    out-of-range table entry, are fetched from an out-of-bounds coordinate,
//    which TMA fills with zeros.  No multicast.
//  * S = Q.K^T and O += P.V are tcgen05.mma kind::f16 (bf16 in, fp32 out)
//    with M = N = 128, K = 16 per instruction, accumulators in tensor memory
//    (two S buffers, and one O accumulator per key half: 512 columns),
//    tracked with tcgen05.commit on mbarriers.  Q.K runs up to two tiles ahead
//    of P.V.
//  * Softmax: each thread owns half of one row's keys and its own accumulator.
//    It reads S with tcgen05.ld, applies the mask, keeps its own reference
//    maximum in the log2 domain that only moves when a tile's maximum exceeds
//    it by more than 8 (so p <= 2^8 and O needs rescaling rarely), writes P as
//    bf16 back into the first half of the S columns it read (tcgen05.st, two
//    bf16 per column), from where P.V takes its A operand, and sums the fp32
//    probabilities into its l.  The two halves meet once, in the epilogue:
//    (O0 f0 + O1 f1) / (l0 f0 + l1 f1), f = 2^(m - max(m0, m1)).
//  * Two Q buffers, two-stage K and V rings; a K slot is refilled once its Q.K
//    has completed, a V slot once its P.V has.  A full M-tile of bf16 output is
//    staged in its unit's Q buffer and leaves by tensor stores.
//  * Every wait is bounded; on expiry the kernel records PA_DEVERR_TIMEOUT,
//    waits (bounded) for its outstanding work and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace prefill {

constexpr int kSoftWarps = 8;               // softmax warps: two per TMEM lane quadrant
constexpr int kParts = kSoftWarps / 4;      // warps sharing a row: each owns kPK of its 128 keys
constexpr int kPK = 128 / kParts;           // keys of a row per softmax thread (64)
constexpr int kPC = kPK / 32;               // 32-column TMEM accesses per thread and tile
constexpr int kMmaWarp = kSoftWarps;        // lane 0 issues the P.V MMAs
constexpr int kKWarp = kSoftWarps + 1;      // copies Q and the K tiles
constexpr int kVWarp = kSoftWarps + 2;      // copies the V tiles
constexpr int kQkWarp = kSoftWarps + 3;     // lane 0 issues the Q.K MMAs
constexpr int kThreads = (kSoftWarps + 4) * 32;
constexpr int kRows = 128;                  // M tile
constexpr int kKeys = 128;                  // N tile of Q.K (keys per iteration)
constexpr int kD = 128;                     // head_dim
constexpr uint32_t kHalf = 128u * 128u;     // one [128 rows][64 bf16] swizzled half tile, bytes
constexpr uint32_t kTile = 2u * kHalf;      // [2 halves][128 rows][128 B]
constexpr uint32_t kOffQ = 0;               // two Q buffers (a unit's Q lands while the previous one finishes)
#ifndef PA_PREFILL_KV_STAGES
#define PA_PREFILL_KV_STAGES 2
#endif
constexpr int kKV = PA_PREFILL_KV_STAGES;    // K and V ring depth (2 and 3 measured alike)
constexpr uint32_t kOffK = kOffQ + 2 * kTile;   // kKV stages, [half][128 keys][128 B]
constexpr uint32_t kOffV = kOffK + kKV * kTile; // kKV stages, [block][half][16 keys][128 B]
constexpr uint32_t kOffBar = kOffV + kKV * kTile;
constexpr uint32_t kBarBytes = 256;
constexpr uint32_t kOffX = kOffBar + kBarBytes;   // epilogue: each part's (m, l, done) per row
constexpr int kMaxUnits = 256;                    // units per CTA (the launcher adds CTAs beyond)
constexpr uint32_t kOffUnits = kOffX + (uint32_t)kParts * 128u * 12u;
constexpr uint32_t kSmemBytes = kOffUnits + kMaxUnits * 8 + 1024;   // + alignment slack
constexpr int kSBufs = 2;                   // S accumulators in tensor memory
constexpr uint32_t kTmemCols = 512;         // S0, S1, O0, O1 (128 columns each)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 domain
#ifndef PA_PREFILL_PRECISE_KEYS
#define PA_PREFILL_PRECISE_KEYS 512
#endif
constexpr int kPreciseKeys = PA_PREFILL_PRECISE_KEYS;   // fewer visible keys: probabilities as two bf16 terms
static_assert(kSmemBytes <= 232448, "shared memory");

struct Params {
    __nv_bfloat16 *out;          // [B][C][Hq][D]
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *ctx_lens;
    int32_t max_ctx_len;
    int32_t chunk;
    int32_t num_q_heads;
    int64_t num_blocks;
    float scale_log2;
    unsigned int *err;
    int32_t causal;              // 0: every query of sequence s sees keys 0 .. ctx_lens[s] - 1
    float *o_part;               // non-null: fp32 output normalised by l, [B][C][Hq][D], instead of out
    float *lse;                  // with o_part: [B][C][Hq] natural-log sum of exp(scale * q.k)
    const int32_t *order;        // non-null: sequence slot z holds sequence order[z] (a permutation of 0 .. B-1)
    int32_t num_mt;              // M-tiles per sequence
    int32_t num_kv;              // kv-heads
    int32_t num_seqs;            // sequences (B)
    int32_t early_meta;          // order, ctx_lens and tables are not written by the kernel before
    // Grouped decode (sfx_tables non-null): sequence s stands for a group of
    // `chunk` members that share its ctx_lens[s] prefix tokens; after the
    // prefix tiles one more tile holds every member's own suffix blocks (member
    // m of the M-tile in blocks m * sfx_nb .. m * sfx_nb + sfx_nb - 1), and each
    // row attends the prefix plus its member's suffix keys only.
    const int32_t *sfx_tables;   // [groups * chunk][sfx_max_blocks]
    int32_t sfx_max_blocks;
    const int32_t *sfx_lens;     // [groups * chunk]
    int32_t sfx_nb;              // tail-tile blocks per member
    int32_t max_sfx_len;
    // with sfx_tables: each member's new token, stored at its last suffix
    // position before that tile is read (nullptr: none)
    const __nv_bfloat16 *new_k;  // [groups * chunk][Hkv][D]
    const __nv_bfloat16 *new_v;
    __nv_bfloat16 *pool;         // the layer's pool view (element strides below)
    int64_t block_stride;
    int64_t kv_stride;
};


// ---- PTX wrappers -----------------------------------------------------------

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Shared -> global copy of one box of a 4-D tensor map at (c0 .. c3), in this
// thread's current bulk group (coordinates >= 0, c0 * 2 B a multiple of 16 B).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(map),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have finished reading shared memory / have completed
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Hint: bring one box of a 4-D tensor map at (c0 .. c3) into L2 (changes no
// data and orders nothing, so it may run before the data's writer finishes).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(map), "r"(c0),
                 "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5, %6}], [%7];" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int *err) {
    return mbar_wait_bounded(reinterpret_cast<uint64_t *>(__cvta_shared_to_generic(bar)), parity, err);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: 128-byte swizzle, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, A K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// A operand from tensor memory (M rows in lanes, K along columns, two bf16 per column).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

#define PA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                 "=r"(r[i + 6]), "=r"(r[i + 7])
#define PA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                 "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : PA_R8(0), PA_R8(8), PA_R8(16), PA_R8(24)
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        PA_W8(0), PA_W8(8), PA_W8(16), PA_W8(24)
        : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[N]) {   // r[0..15]
    static_assert(N >= 16, "16 words");
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        PA_W8(0), PA_W8(8)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- the kernel ---------------------------------------------------------------

__device__ __forceinline__ void mbar_arrive_u32(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Tensor-memory column of keys kk*16 .. kk*16+15 of P in S buffer sb: each
// part of a row's keys is written, two bf16 per column, by the warp that read
// it, into the first half of the S columns it read.
__device__ __forceinline__ uint32_t p_col(int sb, int kk) {
    constexpr int kSteps = kPK / 16;   // 16-key P.V steps per softmax thread
    return (uint32_t)(sb * 128 + (kk / kSteps) * kPK + (kk % kSteps) * 8);
}

__device__ __forceinline__ void part_sync(int warp) {   // warps w, w + 4, ... own the same rows
    asm volatile("bar.sync %0, %1;" ::"r"(1 + (warp & 3)), "r"(kParts * 32) : "memory");
}

__device__ __forceinline__ void soft_sync() {   // all softmax warps
    asm volatile("bar.sync 5, %0;" ::"n"(kSoftWarps * 32) : "memory");
}

__device__ __forceinline__ float max_tree32(const uint32_t (&a)[32]) {
    float m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = fmaxf(__uint_as_float(a[i]), __uint_as_float(a[i + 16]));
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    return m[0];
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Maximum of 64 values by three-input steps: 64 -> 22 -> 8 -> 4 -> 2 -> 1
// (32 instructions, five deep, against 63 and six with two-input steps).
__device__ __forceinline__ float max_tree64(const uint32_t (&a)[32], const uint32_t (&b)[32]) {
    float v[64];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v[i] = __uint_as_float(a[i]);
        v[32 + i] = __uint_as_float(b[i]);
    }
    float m1[22];
#pragma unroll
    for (int i = 0; i < 21; ++i) m1[i] = max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
    m1[21] = v[63];
    float m2[8];
#pragma unroll
    for (int i = 0; i < 7; ++i) m2[i] = max3(m1[3 * i], m1[3 * i + 1], m1[3 * i + 2]);
    m2[7] = m1[21];
    const float x = max3(m2[0], m2[1], m2[2]), y = max3(m2[3], m2[4], m2[5]);
    return fmaxf(max3(x, y, m2[6]), m2[7]);
}

// Work units: one (M-tile mt, kv-head g, sequence slot z) each, numbered
// u = mt + num_mt * (g + num_kv * z).  The grid is persistent (one CTA per SM
// at most): CTA c takes units k * C + c for even rounds k and k * C + C - 1 - c
// for odd ones, so when the caller orders the sequences longest first a CTA
// that drew a long unit in one round draws a short one in the next.  Each
// role walks the same unit list; the CTA's tiles are numbered T = 0, 1, ...
// across its units, and every ring (K / V slots, S buffers, P and P.V
// barriers) is indexed by T, so the next unit's copies stream while the
// current one finishes.
//
// Timeline of tile T (kKV = kSBufs = 2):
//   K warp   : Q of unit k -> Q buffer k % 2 once the Q.K of unit k - 2 are done;
//              K(T) -> K slot T % 2 once Q.K(T - 2) has completed
//   V warp   : V(T) -> V slot T % 2 once P.V(T - 2) has completed
//   Q.K lane : Q.K(T) -> S[T % 2] once K(T) and the unit's Q have landed and
//              P.V(T - 2) has completed
//   P.V lane : P.V(T) once P(T) and V(T) are in place (a unit's first once the
//              previous unit's epilogue has read O)
//   softmax  : S[T % 2] -> registers ; P(T) into S[T % 2] ; O rescale when the
//              reference moved ; signal P(T) ; after a unit's last tile its
//              epilogue, then O is released to the next unit
// Barriers: Q landed / Q free per buffer, K / V landed (TMA), S ready, P.V done
// per P buffer and per S buffer, K / V slot free (MMA commit), P ready and O
// read (256 arrivals), unit's P.V done, suffix tile's V ready (grouped), one
// drain per MMA lane (MMA commit, used once).
// A parity wait is exact only while the barrier's previous phase is known to
// have completed; each wait below names the completion that guarantees it.
template <int G, int BS, bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                   const Params p) {
    constexpr int QPT = kRows / G;   // queries per M-tile
    constexpr int NBT = kKeys / BS;  // blocks per 128-key tile
    constexpr uint32_t kVBlock = 2u * BS * 128u;   // one block's V box: [half][BS keys][128 B]
    static_assert(BS == 8 || BS == 16 || BS == 32 || BS == 64, "block size");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - smem_addr(smem_raw));
    const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV;
    const uint32_t barQ = base + kOffBar;
    // barriers: Q landed[2] | K[kKV] | V[kKV] | S[2] | P[2] | P.V done[2] | P.V done per S buffer[2] |
    // K slot free[kKV] | V slot free[kKV] | Q free[2] | unit's P.V done | O read | suffix V ready[2] |
    // drain (P.V, Q.K issuers)
    const uint32_t barK = barQ + 16, barV = barK + 8 * kKV, barS = barV + 8 * kKV, barP = barS + 16,
                   barOP = barP + 16, barSdone = barOP + 16, barKfree = barSdone + 16, barVfree = barKfree + 8 * kKV,
                   barQfree = barVfree + 8 * kKV, barUnit = barQfree + 16, barOfree = barUnit + 8,
                   barVsfx = barOfree + 8, barEnd = barVsfx + 16, barEndQk = barEnd + 8;
    constexpr int kNumBars = 2 + 2 * kKV + 2 + 2 + 2 + 2 + 2 * kKV + 2 + 1 + 1 + 2 + 2;
    static_assert(8 * kNumBars + 8 <= kBarBytes, "barrier area");
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffBar + 8 * kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kOffBar + 8 * kNumBars + 4);
    int2 *utab = reinterpret_cast<int2 *>(gbase + kOffUnits);   // this CTA's units: (sequence, context length)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const uint32_t b = barQ + 8 * i;
            const bool softmax_arrivals = (b >= barP && b < barOP) || b == barOfree;   // P[2], O read
            // Q free: the Q.K lane's commit and the softmax's release of the
            // buffer, which may stage the unit's output tile for a tensor store
            const bool q_free = b >= barQfree && b < barQfree + 16;
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b),
                         "r"(softmax_arrivals ? (uint32_t)(kSoftWarps * 32) : (q_free ? 2u : 1u))
                         : "memory");
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();   // the barriers, before unit 0's Q copy below

    // The kernel is launched with programmatic stream serialisation: what it
    // reads waits for the kernel before it to finish here, except, when the
    // caller promises that kernel does not write them, the sequence order,
    // context lengths and tables, read below while it still runs.  Each CTA
    // lets the kernel after this one be scheduled once it has passed that
    // wait (so every kernel before this one has finished, and every CTA of
    // this grid has started): that kernel's CTAs set up on the SMs this grid's
    // CTAs leave as they finish, and wait for the whole grid before they read
    // what it wrote.
    if (!p.early_meta) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }

    // ---- this CTA's units, read once into shared memory
    const int C = (int)gridDim.x, cta = (int)blockIdx.x;
    const int per_seq = p.num_mt * p.num_kv;
    const int n_units = per_seq * p.num_seqs;
    auto unit_index = [&](int k) { return k * C + ((k & 1) ? C - 1 - cta : cta); };
    const int rounds = (n_units + C - 1) / C;
    int my_units = rounds > 0 ? rounds - 1 + (unit_index(rounds - 1) < n_units ? 1 : 0) : 0;
    if (my_units > kMaxUnits) {   // the launcher sizes the grid so that this cannot happen
        if (tid == 0) raise_error(p.err, PA_DEVERR_SEQ_LEN);
        my_units = kMaxUnits;
    }
    // Copy warps: unit 0's sequence and its first 64 block ids, read beside the
    // table below instead of after it (an id is checked against the unit's
    // blocks when first used, so the ids need not wait for the context
    // length); the K warp copies unit 0's Q as soon as its sequence is known.
    int ids0_a = 0, ids0_b = 0, s0 = 0;
    if ((warp == kKWarp || warp == kVWarp) && my_units > 0) {
        const int z0 = unit_index(0) / per_seq;
        s0 = z0;
        if (p.order != nullptr) {   // a bad entry is reported by the table fill
            const int o = __ldg(p.order + z0);
            if (o >= 0 && o < p.num_seqs) s0 = o;
        }
        const int32_t *row0 = p.tables + (size_t)s0 * p.max_blocks;
        if (lane < p.max_blocks) ids0_a = __ldg(row0 + lane);
        if (32 + lane < p.max_blocks) ids0_b = __ldg(row0 + 32 + lane);
        if (p.early_meta) {
            // While the kernel before still runs: unit 0's Q and first two K/V
            // tiles into L2 (hints; an id past the unit's blocks only warms an
            // unused block, one out of range is skipped)
            const int u0 = unit_index(0);
            if (warp == kKWarp && lane < 2)
                tma_prefetch_4d(&tmap_q, lane * 64, 0, (u0 / p.num_mt) % p.num_kv, s0 * p.chunk + (u0 % p.num_mt) * QPT);
            if (lane < kKV * NBT && ids0_a >= 0 && ids0_a < p.num_blocks) {
                const int g0 = (u0 / p.num_mt) % p.num_kv;
                if (warp == kKWarp) {
                    tensor_prefetch_l2_5d(&tmap_k, 0, 0, g0, 0, ids0_a);
                    tensor_prefetch_l2_5d(&tmap_k, 64, 0, g0, 0, ids0_a);
                } else {
                    tensor_prefetch_l2_5d(&tmap_v, 0, 0, 0, g0, ids0_a);
                }
            }
        }
        if (warp == kKWarp && !p.early_meta) {
            const int u0 = unit_index(0);
            if (lane == 0) mbar_expect(barQ, kTile);
            __syncwarp();
            if (lane < 2)
                tma_load_4d(sQ + lane * kHalf, &tmap_q, lane * 64, 0, (u0 / p.num_mt) % p.num_kv,
                            s0 * p.chunk + (u0 % p.num_mt) * QPT, barQ);
        }
    }
    for (int k = tid; k < my_units; k += kThreads) {
        const int z = unit_index(k) / per_seq;
        int s = z;
        if (p.order != nullptr) {   // the caller's order: units start in it, so the longest work can go first
            const int o = __ldg(p.order + z);
            if (o >= 0 && o < p.num_seqs) s = o;
            else raise_error(p.err, PA_DEVERR_ORDER);
        }
        int ctx = __ldg(p.ctx_lens + s);
        if (ctx < 0 || ctx > p.max_ctx_len) {
            raise_error(p.err, PA_DEVERR_SEQ_LEN);
            ctx = ctx < 0 ? 0 : p.max_ctx_len;
        }
        utab[k] = make_int2(s, ctx);
    }
    if (p.early_meta) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (warp == kKWarp && my_units > 0) {   // q may come from the kernel before
            const int u0 = unit_index(0);
            if (lane == 0) mbar_expect(barQ, kTile);
            __syncwarp();
            if (lane < 2)
                tma_load_4d(sQ + lane * kHalf, &tmap_q, lane * 64, 0, (u0 / p.num_mt) % p.num_kv,
                            s0 * p.chunk + (u0 % p.num_mt) * QPT, barQ);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + kSBufs * 128;

    // grouped decode is a separate instantiation: its code in the plain
    // kernel, even when idle, cost the causal prefill 20% (1.18 against 0.98 ms)
    const bool grouped = kGrouped && p.sfx_tables != nullptr && p.sfx_nb > 0;
    struct Unit {
        int s, g, j0, ctx, seq_end, nblk_seq, n_pre, n_tiles, members;
        bool precise;
    };
    auto unit = [&](int k) {
        Unit U;
        const int u = unit_index(k);
        const int2 e = utab[k];
        U.s = e.x;
        U.ctx = e.y;
        U.g = (u / p.num_mt) % p.num_kv;
        U.j0 = (u % p.num_mt) * QPT;
        // causal: keys 0 .. ctx + C - 1 exist and query j sees 0 .. ctx + j;
        // otherwise keys 0 .. ctx - 1 exist and every query sees all of them
        U.seq_end = p.causal ? U.ctx + p.chunk : U.ctx;
        U.nblk_seq = (U.seq_end + BS - 1) / BS;
        const int last_q = min(U.j0 + QPT, p.chunk) - 1;   // last valid query of the M-tile
        U.n_pre = ((p.causal ? U.ctx + last_q + 1 : U.ctx) + kKeys - 1) / kKeys;   // 0 only without causal
        U.n_tiles = U.n_pre + (grouped ? 1 : 0);   // grouped: the members' suffix tile last
        // members of the M-tile (grouped): queries j0 .. j0 + members - 1
        U.members = max(0, min(QPT, p.chunk - U.j0));
        // Grouped rows that may see fewer than kPreciseKeys keys carry each
        // probability as two bf16 terms, hi = bf16(p) and lo = bf16(p - hi), and
        // P.V runs once for each: with few keys a single rounding of p (relative
        // error 2^-9) does not average down (one output of an eight-key beam row
        // moved by 1.0% of its value); with many it does, and one term is kept.
        // The plain kernel has no second term at all: even idle, it cost the
        // causal prefill 13% (1.09 against 0.96 ms).
        U.precise = kGrouped && U.ctx + p.max_sfx_len < kPreciseKeys;
        return U;
    };
    constexpr uint32_t idesc_qk = idesc_bf16(kRows, kKeys, false);
    constexpr uint32_t idesc_pv = idesc_bf16(kRows, kD, true);

    if (warp == kKWarp || warp == kVWarp) {
        // ---- copy warps: a lane per box.  Block ids sit in registers: one
        // load of the 32 lanes holds blocks c * 32 + lane, i.e. tiles c * TPC ..
        // c * TPC + TPC - 1, and the next load is issued a whole load ahead (the
        // next unit's first two at the start of this one), so no copy waits on
        // a table read (a dependent read per tile held the copies ~1,800 cycles
        // apart, slower than the MMAs consume tiles).  An id is checked when its
        // load becomes the current one.
        constexpr int TPC = 32 / NBT;
        const bool is_k = warp == kKWarp;
        const uint32_t bar0 = is_k ? barK : barV;
        const uint32_t slot0 = is_k ? sK : sV;
        auto ids_load = [&](const Unit &U, int c) -> int {
            const int bi = c * 32 + lane;
            int v = 0;
            if (bi < U.nblk_seq && bi < U.n_pre * NBT) v = __ldg(p.tables + (size_t)U.s * p.max_blocks + bi);
            return v;
        };
        auto ids_check = [&](int v, const Unit &U, int c) -> int {   // out-of-bounds coordinate: zero fill
            const int bi = c * 32 + lane;
            if (!(bi < U.nblk_seq && bi < U.n_pre * NBT)) return (int)p.num_blocks;
            if (v < 0 || v >= p.num_blocks) {
                raise_error(p.err, PA_DEVERR_BLOCK_ID);
                return (int)p.num_blocks;
            }
            return v;
        };
        bool ok = true;
        int T = 0;                 // tiles issued so far
        Unit U;
        int raw_cur = ids0_a, raw_next = ids0_b;   // unit 0's, read above
        if (my_units > 0) U = unit(0);
        for (int k = 0; k < my_units && ok; ++k) {
            Unit N = U;            // the next unit, and its first ids
            int nraw_cur = 0, nraw_next = 0;
            if (k + 1 < my_units) {
                N = unit(k + 1);
                nraw_cur = ids_load(N, 0);
                nraw_next = ids_load(N, 1);
            }
            if (is_k && k > 0) {   // (unit 0's Q was copied above)
                // Q buffer k % 2 held unit k - 2's Q: its Q.K must have completed
                // and the store of the output tile staged there must have read it
                // (the phase before, unit k - 4's, was waited for here two units ago)
                const int qb = k & 1;
                if (k >= 2) ok = __all_sync(0xffffffffu, mbar_wait(barQfree + 8 * qb, (uint32_t)(((k >> 1) - 1) & 1), p.err));
                if (!ok) {
                    *abort_flag = 1;
                    break;
                }
                if (lane == 0) mbar_expect(barQ + 8 * qb, kTile);
                __syncwarp();
                if (lane < 2)
                    tma_load_4d(sQ + qb * kTile + lane * kHalf, &tmap_q, lane * 64, 0, U.g, U.s * p.chunk + U.j0,
                                barQ + 8 * qb);
            }
            int ids_cur = ids_check(raw_cur, U, 0);
            int tail_id = (int)p.num_blocks;   // grouped: this lane's block of the suffix tile (out of bounds: zeros)
            // grouped: lane m < members holds member m's suffix length, loaded here
            // and first used once the unit's first tiles are in flight (members <=
            // NBT: each member owns at least one block of the suffix tile)
            int len_m = 0;
            if (grouped && lane < U.members) len_m = __ldg(p.sfx_lens + U.s * p.chunk + U.j0 + lane);
            // Each member's new token goes into the pool (K warp: K rows, V warp: V
            // rows), then a proxy fence: this warp's tensor copy of the suffix tile
            // is issued after it in program order.  The work runs in three stages,
            // one before each of three consecutive slot waits once the unit's first
            // tiles are in flight, each only issuing the reads the next one
            // consumes, so the chain of dependent reads (length, block, token)
            // overlaps waits the warp makes anyway; stages not yet run by the
            // suffix tile run there.
            constexpr int kPass = (NBT + 1) / 2;   // two members a pass: 16 lanes x 16 B = one row of d = 128
            int L = 0, nblk = -1, tv = 0;
            bool tv_read = false;   // this lane read a block of the suffix tile into tv
            uint4 tok[kPass];
            auto prep_lengths = [&]() {   // clip the lengths; read each token's block and this lane's tail block
                const int cap = min(p.max_sfx_len, min(p.sfx_max_blocks, p.sfx_nb) * BS);
                L = len_m;
                if (lane < U.members && (L < 0 || L > cap)) {
                    if (is_k && U.g == 0) raise_error(p.err, PA_DEVERR_SEQ_LEN);
                    L = L < 0 ? 0 : cap;
                }
                if (p.new_k != nullptr && lane < U.members && L > 0)
                    nblk = __ldg(p.sfx_tables + (size_t)(U.s * p.chunk + U.j0 + lane) * p.sfx_max_blocks + (L - 1) / BS);
                // this lane's block of the suffix tile: member lane / sfx_nb, its block lane % sfx_nb
                const int mt_ = lane / p.sfx_nb, bt = lane % p.sfx_nb;
                const int Lt = __shfl_sync(0xffffffffu, L, mt_ & 31);
                tv_read = lane < NBT && mt_ < U.members && bt * BS < Lt;
                if (tv_read) tv = __ldg(p.sfx_tables + (size_t)(U.s * p.chunk + U.j0 + mt_) * p.sfx_max_blocks + bt);
            };
            auto prep_tokens = [&]() {    // check the tail blocks; read the tokens
                if (tv_read) {
                    if (tv < 0 || tv >= p.num_blocks) raise_error(p.err, PA_DEVERR_BLOCK_ID);
                    else tail_id = tv;
                }
                if (p.new_k == nullptr) return;
#pragma unroll
                for (int ps = 0; ps < kPass; ++ps) {
                    const int m = ps * 2 + (lane >> 4), c16 = lane & 15;
                    const int bm = __shfl_sync(0xffffffffu, nblk, m & 31), Lm = __shfl_sync(0xffffffffu, L, m & 31);
                    tok[ps] = make_uint4(0u, 0u, 0u, 0u);
                    if (m < U.members && Lm > 0 && bm >= 0 && bm < p.num_blocks) {   // a bad id is reported above
                        const size_t seq = (size_t)U.s * p.chunk + U.j0 + m;
                        tok[ps] = __ldg(reinterpret_cast<const uint4 *>((is_k ? p.new_k : p.new_v) +
                                                                        (seq * p.num_kv + U.g) * kD + c16 * 8));
                    }
                }
            };
            auto prep_store = [&]() {     // store the tokens, then the proxy fence
                if (p.new_k == nullptr) return;
#pragma unroll
                for (int ps = 0; ps < kPass; ++ps) {
                    const int m = ps * 2 + (lane >> 4), c16 = lane & 15;
                    const int bm = __shfl_sync(0xffffffffu, nblk, m & 31), Lm = __shfl_sync(0xffffffffu, L, m & 31);
                    if (m < U.members && Lm > 0 && bm >= 0 && bm < p.num_blocks)
                        *reinterpret_cast<uint4 *>(p.pool + (size_t)bm * p.block_stride + (is_k ? 0 : p.kv_stride) +
                                                   ((size_t)U.g * BS + (Lm - 1) % BS) * kD + c16 * 8) = tok[ps];
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
            };
            const int prep0 = min(U.n_pre, kKV);   // the first stage's tile
            for (int t = 0; t < U.n_tiles; ++t) {
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                const int st = T % kKV;
                if (t > 0 && t % TPC == 0) {
                    ids_cur = ids_check(raw_next, U, t / TPC);
                    raw_next = ids_load(U, t / TPC + 1);
                }
                if (grouped) {   // before the slot wait below; all three by the suffix tile
                    if (t == prep0) prep_lengths();
                    if (t == min(prep0 + 1, U.n_pre)) prep_tokens();
                    if (t == min(prep0 + 2, U.n_pre)) prep_store();
                }
                const int tb = (t % TPC) * NBT;   // the tile's first block in the loaded ids
                const bool tail = grouped && t == U.n_pre;   // the members' suffix tile
                const int id = tail ? tail_id : __shfl_sync(0xffffffffu, ids_cur, (tb + lane) & 31);
                if (T >= kKV) {   // the slot's previous tile has been consumed by its MMAs
                    // (Q.K for a K slot, P.V for a V slot, each committing to the slot's
                    // own barrier; its next completion needs the copy issued below, so
                    // its phase cannot be lapped)
                    const int tp = T - kKV;
                    const uint32_t free_bar = (is_k ? barKfree : barVfree) + 8 * (tp % kKV);
                    ok = __all_sync(0xffffffffu, mbar_wait(free_bar, (uint32_t)((tp / kKV) & 1), p.err));
                    if (!ok) {
                        *abort_flag = 1;
                        break;
                    }
                }
                if (lane == 0) mbar_expect(bar0 + 8 * st, kTile);
                __syncwarp();
                const uint32_t dst = slot0 + st * kTile;
                if (is_k) {
                    const int blk = tail ? __shfl_sync(0xffffffffu, tail_id, lane >> 1)
                                         : __shfl_sync(0xffffffffu, ids_cur, (tb + (lane >> 1)) & 31);
                    if (lane < 2 * NBT)
                        tma_load_5d(dst + (lane & 1) * kHalf + (lane >> 1) * (BS * 128), &tmap_k, (lane & 1) * 64, 0,
                                    U.g, 0, blk, bar0 + 8 * st);
                } else if (lane < NBT) {
                    tma_load_5d(dst + lane * kVBlock, &tmap_v, 0, 0, 0, U.g, id, bar0 + 8 * st);
                }
                ++T;
            }
            if (!ok) break;
            if (grouped && !is_k) {
                // suffix tile (this unit's last, T - 1): zero each member's V slots
                // past its length (p is 0 there, but the slots may hold non-finite
                // junk), then hand the tile to its P.V.  The wait is exact: this warp
                // issued the copy only after the slot's previous tile (its previous
                // phase) had been consumed.
                const int Ts = T - 1, sv = Ts % kKV;
                mbar_wait(barV + 8 * sv, (uint32_t)((Ts / kKV) & 1), p.err);
                for (int m = 0; m < U.members; ++m) {
                    const int r0 = m * p.sfx_nb * BS + __shfl_sync(0xffffffffu, L, m & 31);
                    const int r1 = (m + 1) * p.sfx_nb * BS;
                    for (int idx = lane; idx < (r1 - r0) * 2 * 8; idx += 32) {
                        const int rr = r0 + idx / 16, h = (idx / 8) & 1, c16 = idx & 7;
                        const uint32_t addr = sV + sv * kTile + (uint32_t)(rr / BS) * kVBlock + h * (kVBlock / 2) +
                                              (uint32_t)(rr % BS) * 128u + (uint32_t)c16 * 16u;
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                    }
                }
                // the zeros (generic proxy) before the P.V that reads them (async proxy).
                // Units alternate between two barriers: with one, a run of one-tile
                // units let this warp release two units' tiles before the P.V lane
                // waited for the first, and that wait then saw the phase after
                // (released, unit k + 2's tile needs V slot reuse, which waits for
                // unit k's P.V, so neither barrier is lapped).
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive_u32(barVsfx + 8 * (k & 1));
            }
            U = N;
            raw_cur = nraw_cur;
            raw_next = nraw_next;
        }
        if (!ok || *abort_flag) {
            // wait (bounded) for this warp's copies still in flight before the memory is released
            for (int t = max(0, T - kKV); t < T; ++t)
                mbar_wait(bar0 + 8 * (t % kKV), (uint32_t)((t / kKV) & 1), p.err);
            if (grouped && !is_k && lane == 0) {   // a waiting P.V lane gives up sooner
                mbar_arrive_u32(barVsfx);
                mbar_arrive_u32(barVsfx + 8);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp || warp == kQkWarp) {
        // Two issuing lanes in two warps keep the tensor pipe's queue fed: one
        // issues Q.K(T) as soon as K(T) has landed and S buffer T % 2 is free
        // (P.V(T - 2), which read P(T - 2) from it, has completed; a barrier per
        // S buffer tracks that), the other P.V(T) as soon as P(T) and V(T) are in
        // place.  Each commits and drains only its own MMAs.
        if (lane == 0) {
            const bool is_qk = warp == kQkWarp;
            bool ok = true;
            auto wait = [&](uint32_t bar, uint32_t parity) {
                if (ok && !mbar_wait(bar, parity, p.err)) {
                    ok = false;
                    *abort_flag = 1;
                }
                return ok;
            };
            int T = 0;
            for (int k = 0; k < my_units && ok && !*abort_flag; ++k) {
                const Unit U = unit(k);
                if (is_qk) {
                    // unit k's Q (the phase before, unit k - 2's, was waited for here)
                    const int qb = k & 1;
                    if (!wait(barQ + 8 * qb, (uint32_t)((k >> 1) & 1))) break;
                    const uint32_t sQb = sQ + qb * kTile;
                    for (int t = 0; t < U.n_tiles; ++t, ++T) {
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        const int st = T % kKV, sb = T % kSBufs;
                        if (!wait(barK + 8 * st, (uint32_t)((T / kKV) & 1))) break;
                        // S buffer sb held P(T - 2): its P.V must have completed (P.V(T)
                        // cannot complete before this Q.K, so the phase cannot be lapped)
                        if (T >= kSBufs && !wait(barSdone + 8 * sb, (uint32_t)(((T - kSBufs) / kSBufs) & 1))) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                            umma(tmem + sb * 128, smem_desc(sQb + off, 16, 1024),
                                 smem_desc(sK + st * kTile + off, 16, 1024), idesc_qk, kk > 0);
                        }
                        umma_commit(barS + 8 * sb);
                        umma_commit(barKfree + 8 * st);   // K slot st is free again
                    }
                    if (!ok) break;
                    umma_commit(barQfree + 8 * qb);        // Q buffer qb is free again
                } else {
                    // O is overwritten by this unit's first P.V: the previous unit's
                    // epilogue must have read it (its phase before, unit k - 2's, was
                    // waited for here)
                    if (k > 0 && !wait(barOfree, (uint32_t)((k - 1) & 1))) break;
                    for (int t = 0; t < U.n_tiles; ++t, ++T) {
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        const int st = T % kKV;
                        if (!wait(barP + 8 * (T & 1), (uint32_t)((T >> 1) & 1))) break;
                        // the suffix tile's V once the V warp has zeroed its unused
                        // slots (one such tile per unit, units alternating barriers)
                        const bool vsfx = grouped && t == U.n_pre;
                        if (!wait(vsfx ? barVsfx + 8 * (k & 1) : barV + 8 * st,
                                  vsfx ? (uint32_t)((k >> 1) & 1) : (uint32_t)((T / kKV) & 1)))
                            break;
                        tc_fence_after();
#pragma unroll
                        for (int term = 0; term < (U.precise ? 2 : 1); ++term) {   // hi, then lo (precise rows)
#pragma unroll
                            for (int kk = 0; kk < kKeys / 16; ++kk) {
                                // 16 keys of the V tile: within one block for b >= 16 (8-key groups
                                // 1024 B apart), or two whole blocks for b = 8 (groups one block apart)
                                const uint32_t v_off =
                                    (uint32_t)(kk * 16 / BS) * kVBlock + (uint32_t)((kk * 16) % BS) * 128u;
                                // keys of the first half accumulate into O0, of the second into O1
                                umma_ts(tO + (uint32_t)(kk / (kKeys / 32)) * 128u,
                                        tmem + p_col(T % kSBufs, kk) + (uint32_t)(term * (kPK / 2)),
                                        smem_desc(sV + st * kTile + v_off, BS * 128, BS >= 16 ? 1024 : kVBlock),
                                        idesc_pv, (t > 0 || term > 0 || kk % (kKeys / 32) > 0) ? 1u : 0u);
                            }
                        }
                        umma_commit(barOP + 8 * (T & 1));
                        umma_commit(barSdone + 8 * (T % kSBufs));
                        umma_commit(barVfree + 8 * st);   // V slot st is free again
                    }
                    if (!ok) break;
                    umma_commit(barUnit);   // every P.V of the unit has completed
                }
            }
            // One more commit, on a barrier used once, tracks every MMA this lane
            // issued; its phase-0 wait is exact.  (Waiting on the last P.V's own
            // barrier is not: the two P.V barriers alternate, and when P.V(T - 2)
            // has not completed either, a parity wait for P.V(T) cannot tell the
            // two apart and returns early.)
            if (!ok || *abort_flag) *abort_flag = 1;   // give up: drain what was issued
            const uint32_t end = is_qk ? barEndQk : barEnd;
            umma_commit(end);
            mbar_wait(end, 0, p.err);
        }
        __syncwarp();
    } else {
        // ---- softmax warps: row r, key part pt (scale_log2 > 0: maxima of raw scores)
        const int r = (warp & 3) * 32 + lane, pt = warp >> 2;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const float c = p.scale_log2;
        float *mx = reinterpret_cast<float *>(gbase + kOffX);   // the halves' (m, l, ok) of each row
        float *lx = mx + kParts * 128;
        int *okx = reinterpret_cast<int *>(lx + kParts * 128);
        // thread 0: the Q buffer whose release it owes once the tensor store of
        // the output tile staged there has read it (-1: none)
        int q_owed = -1;
        auto release = [&]() {
            bulk_wait_read();
            mbar_arrive_u32(barQfree + 8 * q_owed);
            q_owed = -1;
        };
        // grouped: the row's member's suffix length, read a unit ahead
        auto sfx_load = [&](int k) -> int {
            const Unit N = unit(k);
            const int j = N.j0 + r / G;
            return j < p.chunk ? __ldg(p.sfx_lens + N.s * p.chunk + j) : 0;
        };
        int sfx_next = grouped && my_units > 0 ? sfx_load(0) : 0;
        int T = 0;
        for (int k = 0; k < my_units; ++k) {
            const Unit U = unit(k);
            const int jr = U.j0 + r / G;
            const int pos = p.causal ? min(U.ctx + jr, U.seq_end - 1) : U.seq_end - 1;   // last key this row may attend
            // grouped: this row's keys in the suffix tile, [sfx_lo, sfx_hi) (a bad
            // length is clipped here and reported by the copy warps)
            const int sfx_lo = (r / G) * p.sfx_nb * BS;
            int sfx_hi = sfx_lo;
            if (grouped) {
                const int cap = min(p.max_sfx_len, min(p.sfx_max_blocks, p.sfx_nb) * BS);
                sfx_hi = jr < p.chunk ? sfx_lo + min(max(sfx_next, 0), cap) : sfx_lo;
                if (k + 1 < my_units) sfx_next = sfx_load(k + 1);
            }
            float m_ref = -INFINITY;                       // reference maximum, log2 domain
            float2 l2 = make_float2(0.f, 0.f);
            int done = 0;
            for (int t = 0; t < U.n_tiles; ++t, ++T) {
                const int st = T & 1, sb = T % kSBufs;   // st: P barrier of this tile
                bool ok = mbar_wait(barS + 8 * sb, (uint32_t)((T / kSBufs) & 1), p.err);
                if (t == 1 && tid == 0 && q_owed >= 0) release();   // the previous unit's store was issued a tile ago
                uint32_t sr[kPC][32];
                if (__all_sync(0xffffffffu, ok)) {
                    tc_fence_after();
#pragma unroll
                    for (int cc = 0; cc < kPC; ++cc) tmem_ld32(tmem + sb * 128 + lane_off + pt * kPK + cc * 32, sr[cc]);
                    tmem_ld_wait();
                } else {
                    ok = false;
                }
                const int key0 = t * kKeys + pt * kPK;
                if (grouped && t == U.n_pre) {   // suffix tile: the row's own member's keys only
#pragma unroll
                    for (int cc = 0; cc < kPC; ++cc)
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int kx = pt * kPK + cc * 32 + i;
                            if (kx < sfx_lo || kx >= sfx_hi) sr[cc][i] = __float_as_uint(-INFINITY);
                        }
                } else if (!__all_sync(0xffffffffu, key0 + kPK - 1 <= pos)) {   // tile crosses some row's causal edge
#pragma unroll
                    for (int cc = 0; cc < kPC; ++cc)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (key0 + cc * 32 + i > pos) sr[cc][i] = __float_as_uint(-INFINITY);
                }
                float mh;
                if constexpr (kPC == 2) mh = max_tree64(sr[0], sr[1]);
                else mh = max_tree32(sr[0]);
                if (__any_sync(0xffffffffu, !ok || *abort_flag)) {   // give up
                    *abort_flag = 1;
                    mbar_arrive_u32(barP + 8 * st);   // keep the arrival count balanced
                    break;
                }
                // this half's own reference: it moves only when the tile maximum
                // exceeds it by more than kRescaleThreshold; the halves' sums meet in
                // the epilogue, so the halves never wait for each other here
                const float mt_ = mh * c;
                float alpha = 1.f;
                if (mt_ > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mt_ != -INFINITY)) {
                    alpha = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - mt_);
                    m_ref = mt_;
                }
                const float2 c2 = make_float2(c, c);
                const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
                const float2 nm2 = make_float2(nm, nm);
                // P goes back into this part's S columns (read above), two bf16 per
                // column; Q.K(T + 2) overwrites them only after P.V(T) has read them
                float2 ps2 = make_float2(0.f, 0.f);
                float2 ps2b = make_float2(0.f, 0.f);   // a second chain: the sums are 16 adds deep, not 32
                uint32_t pw[32];
                if (!U.precise) {
#pragma unroll
                    for (int cc = 0; cc < kPC; ++cc) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[cc][2 * e]),
                                                                    __uint_as_float(sr[cc][2 * e + 1])),
                                                        c2, nm2);
                            const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                            if (e & 1) ps2b = __fadd2_rn(ps2b, pe);
                            else ps2 = __fadd2_rn(ps2, pe);
                            pw[cc * 16 + e] = pack_bf16x2(pe.x, pe.y);
                        }
                    }
                    if constexpr (kPC == 2) tmem_st32(tmem + sb * 128 + lane_off + pt * kPK, pw);
                    else tmem_st16(tmem + sb * 128 + lane_off + pt * kPK, pw);
                } else {
                    // hi = bf16(p) into the first half of this part's S columns, lo =
                    // bf16(p - hi) into the second, 32 scores at a time: a whole part's
                    // hi and lo words at once spilled registers
#pragma unroll
                    for (int cc = 0; cc < kPC; ++cc) {
                        uint32_t ph[16], pl[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[cc][2 * e]),
                                                                    __uint_as_float(sr[cc][2 * e + 1])),
                                                        c2, nm2);
                            const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                            ps2 = __fadd2_rn(ps2, pe);
                            ph[e] = pack_bf16x2(pe.x, pe.y);
                            const float2 hi = bf16x2_to_float2(ph[e]);
                            pl[e] = pack_bf16x2(pe.x - hi.x, pe.y - hi.y);
                        }
                        tmem_st16(tmem + sb * 128 + lane_off + pt * kPK + cc * 16, ph);
                        tmem_st16(tmem + sb * 128 + lane_off + pt * kPK + kPK / 2 + cc * 16, pl);
                    }
                }
                tmem_st_wait();
                ps2 = __fadd2_rn(ps2, ps2b);
                l2.x = l2.x * alpha + (ps2.x + ps2.y);
                // rescale this half's accumulator (all of d) once P.V(T - 1) has
                // completed (the barrier's previous phase, P.V(T - 3), completed before
                // Q.K(T - 1) was issued, which S(T - 1), read before this tile, needed)
                if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    const int tp = T - 1;
                    mbar_wait(barOP + 8 * (tp & 1), (uint32_t)((tp >> 1) & 1), p.err);
                    tc_fence_after();
#pragma unroll
                    for (int cc = 0; cc < kD / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + pt * 128 + lane_off + cc * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + pt * 128 + lane_off + cc * 32, o);
                    }
                    tmem_st_wait();
                }
                // keys past the sequence end inside its last block: zero their V rows
                // (their p is 0, but the slots may hold non-finite junk).  The wait is
                // exact: S(T) needed Q.K(T), issued after P.V(T - 2), which needed
                // V(T - 2), had completed.
                const int tile0 = t * kKeys;
                const int tail_lo = U.seq_end - tile0, blk_end = ((U.seq_end + BS - 1) / BS) * BS - tile0;
                const bool zero_tail = tail_lo > 0 && tail_lo < kKeys && (U.seq_end % BS) != 0;
                if (zero_tail) {
                    const int sv = T % kKV;   // V ring slot of this tile
                    mbar_wait(barV + 8 * sv, (uint32_t)((T / kKV) & 1), p.err);
                    const int nrows = min(blk_end, kKeys) - tail_lo;
                    for (int idx = tid; idx < nrows * 2 * 8; idx += kSoftWarps * 32) {
                        const int rr = tail_lo + idx / 16, h = (idx / 8) & 1, c16 = idx & 7;
                        const uint32_t addr = sV + sv * kTile + (uint32_t)(rr / BS) * kVBlock + h * (kVBlock / 2) +
                                              (uint32_t)(rr % BS) * 128u + (uint32_t)c16 * 16u;
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                    }
                    // the zeroed V rows (generic proxy) before the P.V that reads them (async proxy)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tc_fence_before();
                mbar_arrive_u32(barP + 8 * st);
                done = t + 1;
            }
            // ---- epilogue: the row's two halves merged by their references (O0 f0 +
            // O1 f1) / (l0 f0 + l1 f1), f_h = 2^(m_h - max(m0, m1)); this thread
            // writes half of d: bf16, or fp32 with the row's log-sum-exp.  The
            // unit's P.V have all completed once the P.V lane's unit commit has
            // arrived (the phase before, the previous unit's, was waited for here).
            const bool empty = U.n_tiles == 0;   // no keys: O = 0, lse = -inf, tensor memory never written
            if (tid == 0 && q_owed >= 0) release();   // (units of fewer than two tiles)
            // A full M-tile of bf16 rows is staged in the unit's Q buffer (every Q.K
            // of the unit has completed) in the Q tile's layout and written by two
            // tensor stores: rows written straight from registers leave each warp
            // store 32 lines apart, and those stores held the epilogue ~1 us.
            // (with fewer queries than an M-tile holds, every tile has all `chunk` of
            // them and the output map's box is that high)
            const bool tma_out = p.o_part == nullptr && !empty && U.j0 + min(QPT, p.chunk) <= p.chunk;
            const uint32_t sOut = sQ + (uint32_t)(k & 1) * kTile;
            const bool fin = done == U.n_tiles && !*abort_flag && mbar_wait(barUnit, (uint32_t)(k & 1), p.err);
            mx[pt * 128 + r] = m_ref;
            lx[pt * 128 + r] = l2.x;
            okx[pt * 128 + r] = fin ? 1 : 0;
            part_sync(warp);
            float mh2[kParts], lh2[kParts];
            bool row_fin = true;
#pragma unroll
            for (int q = 0; q < kParts; ++q) {
                mh2[q] = mx[q * 128 + r];
                lh2[q] = lx[q * 128 + r];
                row_fin = row_fin && okx[q * 128 + r] != 0;
            }
            part_sync(warp);   // the next unit's epilogue writes these again
            // one decision for the warp and its partner (both hold the same rows)
            const bool all_fin = __all_sync(0xffffffffu, row_fin);
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < kParts; ++q) M = fmaxf(M, mh2[q]);
            float f[kParts], lt = 0.f;
#pragma unroll
            for (int q = 0; q < kParts; ++q) {
                f[q] = mh2[q] == -INFINITY ? 0.f : fast_exp2(mh2[q] - M);
                lt += lh2[q] * f[q];
            }
            tc_fence_after();
            if (all_fin) {
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                const bool row_ok = jr < p.chunk;
                const size_t row = ((size_t)U.s * p.chunk + jr) * p.num_q_heads + (size_t)U.g * G + (r % G);
#pragma unroll
                for (int cc = 0; cc < kD / kParts / 32; ++cc) {
                    const int d0 = pt * (kD / kParts) + cc * 32;   // this chunk's first dim
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.f;
                    if (!empty) {
#pragma unroll
                        for (int q = 0; q < kParts; ++q) {
                            uint32_t oq[32];
                            tmem_ld32(tO + q * 128 + lane_off + d0, oq);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] += __uint_as_float(oq[i]) * f[q];
                        }
                    }
                    if (row_ok && p.o_part != nullptr) {
                        float4 *dst = reinterpret_cast<float4 *>(p.o_part + row * kD + d0);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(o[q4 * 4 + 0] * inv, o[q4 * 4 + 1] * inv, o[q4 * 4 + 2] * inv,
                                                  o[q4 * 4 + 3] * inv);
                    } else if (row_ok) {
                        __nv_bfloat16 *dst = p.out + row * kD + d0;
                        // 16-byte chunk c of the row's half goes to chunk c ^ (r % 8) of its
                        // 128-byte line: the Q tile's swizzle, which the tensor store undoes
                        const uint32_t line = sOut + (uint32_t)pt * kHalf + (uint32_t)r * 128u;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 v;
                            v.x = pack_bf16x2(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
                            v.y = pack_bf16x2(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
                            v.z = pack_bf16x2(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
                            v.w = pack_bf16x2(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
                            if (tma_out) {
                                const uint32_t c16 = (uint32_t)(cc * 4 + q4);
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                                 line + ((c16 ^ ((uint32_t)r & 7u)) << 4)),
                                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                                             : "memory");
                            } else {
                                *reinterpret_cast<uint4 *>(dst + q4 * 8) = v;
                            }
                        }
                    }
                }
                // sum of exp2(s * scale * log2 e) over the row's keys is lt * 2^M
                if (row_ok && p.o_part != nullptr && pt == 0)
                    p.lse[row] = lt > 0.f ? (M + log2f(lt)) * kLn2 : -INFINITY;
            }
            if (tma_out) {
                // both halves by one tensor store each, once every softmax thread has
                // written its rows (generic writes, then reads by the async proxy)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                soft_sync();
                if (tid == 0) {
                    if (all_fin) {
                        tma_store_4d(&tmap_o, 0, 0, U.g, U.s * p.chunk + U.j0, sOut);
                        tma_store_4d(&tmap_o, 64, 0, U.g, U.s * p.chunk + U.j0, sOut + kHalf);
                        bulk_commit();
                    }
                    q_owed = k & 1;   // released once the stores have read it
                }
            } else if (tid == 0) {
                mbar_arrive_u32(barQfree + 8 * (k & 1));   // nothing staged in the unit's Q buffer
            }
            // O has been read: the next unit's first P.V may overwrite it
            tc_fence_before();
            mbar_arrive_u32(barOfree);
            if (!all_fin) break;   // gave up (the partner warp decides alike)
        }
        if (tid == 0) {   // no store may still read shared memory, or be in flight, when the CTA ends
            if (q_owed >= 0) release();
            bulk_wait_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---- host side --------------------------------------------------------------

// pa_set_prefill_ctas: a fixed persistent grid size (0: one CTA per SM).
std::atomic<int32_t> g_prefill_ctas{0};

template <int G, int BS, bool kGrouped>
cudaError_t launch_kernel(const PrefillArgs &a, const CUtensorMap &mq, const CUtensorMap &mkv, const CUtensorMap &mv,
                         const CUtensorMap &mo, const Params &prm, cudaStream_t stream) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<G, BS, kGrouped>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    // persistent grid: one CTA per SM (or the set count), and enough CTAs that
    // none holds more than kMaxUnits units
    const int64_t n_units = (int64_t)prm.num_mt * prm.num_kv * prm.num_seqs;
    if (n_units == 0) return cudaSuccess;
    int64_t ctas = g_prefill_ctas.load(std::memory_order_relaxed);
    if (ctas <= 0) ctas = device_sm_count();
    if (ctas <= 0) return cudaErrorUnknown;
    ctas = std::max<int64_t>(std::min<int64_t>(ctas, n_units), (n_units + kMaxUnits - 1) / kMaxUnits);
    if (ctas > INT32_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<G, BS, kGrouped>, mq, mkv, mv, mo, prm);
}

template <int G, int BS>
cudaError_t launch_group(const PrefillArgs &a, const CUtensorMap &mq, const CUtensorMap &mkv, const CUtensorMap &mv,
                         const CUtensorMap &mo, const Params &prm, cudaStream_t stream) {
    return a.sfx_tables != nullptr ? launch_kernel<G, BS, true>(a, mq, mkv, mv, mo, prm, stream)
                                   : launch_kernel<G, BS, false>(a, mq, mkv, mv, mo, prm, stream);
}

}  // namespace prefill

void set_prefill_ctas(int32_t ctas) { prefill::g_prefill_ctas.store(ctas, std::memory_order_relaxed); }

bool prefill_supported(int head_dim, int group, int block_size) {
    return head_dim == prefill::kD &&
           (block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    using namespace prefill;
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorUnknown;
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const int G = a.num_q_heads / a.pool.num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return cudaErrorInvalidValue;
    const int Hkv = a.pool.num_kv_heads;

    // q viewed as (d, head in group, kv-head, row = s * C + j); box 64 x G x 1 x (128 / G).
    // The bf16 output, of q's shape, the same way (tensor stores of full M-tiles).
    CUtensorMap mq, mo, mkv;
    for (int which = 0; which < 2; ++which) {
        cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)G, (cuuint64_t)Hkv,
                              (cuuint64_t)a.num_seqs * (cuuint64_t)a.chunk_len};
        cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)G * kD * 2, (cuuint64_t)a.num_q_heads * kD * 2};
        // the output's box: a whole M-tile of queries, or all of them when fewer
        const int qrows = which == 0 ? kRows / G : std::max(1, std::min(kRows / G, a.chunk_len));
        cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)qrows};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        void *base = which == 0 || a.out == nullptr ? const_cast<void *>(a.q) : a.out;   // no bf16 output: unused
        if (encode(which == 0 ? &mq : &mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // pool viewed as (d, slot, kv-head, K|V, block); box 64 x 16 x 1 x 1 x 1
    {
        const int BS = a.pool.block_size;
        cuuint64_t dims[5] = {(cuuint64_t)kD, (cuuint64_t)BS, (cuuint64_t)Hkv, 2, (cuuint64_t)a.pool.num_blocks};
        cuuint64_t strides[4] = {(cuuint64_t)kD * 2, (cuuint64_t)BS * kD * 2, (cuuint64_t)a.pool.kv_stride * 2,
                                 (cuuint64_t)a.pool.block_stride * 2};
        cuuint32_t box[5] = {64, (cuuint32_t)BS, 1, 1, 1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        if (encode(&mkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(a.pool.base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    CUtensorMap mv;   // V: one box per block (both halves of d)
    if (encode_pool_block_map(&mv, a.pool, 1, a.pool.block_size) != cudaSuccess) return cudaErrorInvalidValue;
    Params prm;
    prm.out = static_cast<__nv_bfloat16 *>(a.out);
    prm.tables = a.tables;
    prm.max_blocks = a.max_blocks;
    prm.ctx_lens = a.ctx_lens;
    prm.max_ctx_len = a.max_ctx_len;
    prm.chunk = a.chunk_len;
    prm.num_q_heads = a.num_q_heads;
    prm.num_blocks = a.pool.num_blocks;
    prm.scale_log2 = a.scale * kLog2e;
    prm.err = err;
    prm.causal = a.causal ? 1 : 0;
    prm.o_part = a.o_part;
    prm.lse = a.lse;
    prm.order = a.order;
    prm.num_mt = (a.chunk_len + kRows / G - 1) / (kRows / G);
    prm.num_kv = Hkv;
    prm.num_seqs = a.num_seqs;
    prm.early_meta = a.early_meta ? 1 : 0;
    prm.sfx_tables = a.sfx_tables;
    prm.sfx_max_blocks = a.sfx_max_blocks;
    prm.sfx_lens = a.sfx_lens;
    prm.sfx_nb = a.sfx_nb;
    prm.max_sfx_len = a.max_sfx_len;
    prm.new_k = static_cast<const __nv_bfloat16 *>(a.new_k);
    prm.new_v = static_cast<const __nv_bfloat16 *>(a.new_v);
    prm.pool = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.pool.base));
    prm.block_stride = a.pool.block_stride;
    prm.kv_stride = a.pool.kv_stride;
    auto by_block = [&](auto gtag) -> cudaError_t {
        constexpr int GG = decltype(gtag)::value;
        switch (a.pool.block_size) {
            case 8: return launch_group<GG, 8>(a, mq, mkv, mv, mo, prm, stream);
            case 16: return launch_group<GG, 16>(a, mq, mkv, mv, mo, prm, stream);
            case 32: return launch_group<GG, 32>(a, mq, mkv, mv, mo, prm, stream);
            case 64: return launch_group<GG, 64>(a, mq, mkv, mv, mo, prm, stream);
            default: return cudaErrorInvalidValue;
        }
    };
    switch (G) {
        case 1: return by_block(std::integral_constant<int, 1>());
        case 2: return by_block(std::integral_constant<int, 2>());
        case 4: return by_block(std::integral_constant<int, 4>());
        case 8: return by_block(std::integral_constant<int, 8>());
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
