// pa_block_manager.cpp -- host block manager behind the pa_bm_* C ABI.
//
// how-pagedattention-works (aiinfrainterviews.com):
//  * "A strong answer": equal-size blocks are taken on demand as a sequence
//    grows; each sequence has its own table; only its last block can be
//    partly filled, and equal sizes leave no external fragmentation.
//  * feature table: sequences that share a prompt point at one set of blocks
//    with a reference count per block; a beam fork shares blocks and copies
//    only the block it diverges in (copy-on-write).
//  * "What interviewers probe next": a request is admitted when
//    ceil(prompt / b) blocks plus one to grow into are free, above a small
//    reserved watermark; when the pool runs dry mid-decode a preempted
//    sequence's blocks are swapped to pinned host memory (feature table,
//    preemption row: swap at block granularity).
// auto-20261007-1900-en (lihaoran.work), "How many tail slots remain unused?":
// a sequence of T tokens holds ceil(T / b) blocks.
//
// Free blocks sit on a stack that hands out the lowest ids first and reuses
// the most recently released block next.  The manager never touches the GPU;
// the copy it plans is executed by pa_copy_blocks.
#include <cstdint>
#include <new>
#include <vector>

#include "pa.h"

struct pa_bm {
    struct Seq {
        std::vector<int32_t> blocks;   // device blocks, or host slots while swapped out
        int64_t tokens = 0;
        bool live = false;
        bool swapped = false;
    };
    int64_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> refcount;
    std::vector<int32_t> free_stack;
    std::vector<Seq> seqs;
    std::vector<int32_t> free_seq_ids;
    int64_t host_blocks = 0;
    std::vector<int32_t> host_free;   // free host slots, lowest first

    bool valid_seq(int32_t s) const { return s >= 0 && (size_t)s < seqs.size() && seqs[s].live; }
    int32_t pop_block() {
        const int32_t b = free_stack.back();
        free_stack.pop_back();
        refcount[b] = 1;
        return b;
    }
    void release_block(int32_t b) {
        if (--refcount[b] == 0) free_stack.push_back(b);
    }
    int32_t pop_host() {
        const int32_t h = host_free.back();
        host_free.pop_back();
        return h;
    }
};

namespace {
int64_t blocks_for(int64_t tokens, int32_t b) { return (tokens + b - 1) / b; }
}  // namespace

extern "C" {

pa_status pa_bm_create(pa_bm **out, int64_t num_blocks, int32_t block_size) {
    if (!out || num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return PA_ERR_INVALID_ARG;
    pa_bm *bm = new (std::nothrow) pa_bm();
    if (!bm) return PA_ERR_NO_BLOCKS;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refcount.assign((size_t)num_blocks, 0);
    bm->free_stack.reserve((size_t)num_blocks);
    for (int64_t b = num_blocks - 1; b >= 0; --b) bm->free_stack.push_back((int32_t)b);
    *out = bm;
    return PA_OK;
}

void pa_bm_destroy(pa_bm *bm) { delete bm; }

pa_status pa_bm_add_seq(pa_bm *bm, int32_t *seq_out) {
    if (!bm || !seq_out) return PA_ERR_INVALID_ARG;
    int32_t id;
    if (!bm->free_seq_ids.empty()) {
        id = bm->free_seq_ids.back();
        bm->free_seq_ids.pop_back();
    } else {
        if (bm->seqs.size() >= (size_t)INT32_MAX) return PA_ERR_INVALID_ARG;
        id = (int32_t)bm->seqs.size();
        bm->seqs.emplace_back();
    }
    pa_bm::Seq &s = bm->seqs[id];
    s.blocks.clear();
    s.tokens = 0;
    s.live = true;
    *seq_out = id;
    return PA_OK;
}

pa_status pa_bm_append_tokens(pa_bm *bm, int32_t seq, int64_t n, int64_t *slots_out, int32_t *cow_pair_out,
                              int32_t *n_cow_out) {
    if (!bm || n < 0) return PA_ERR_INVALID_ARG;
    if (!bm->valid_seq(seq)) return PA_ERR_NOT_FOUND;
    pa_bm::Seq &s = bm->seqs[seq];
    if (s.swapped) return PA_ERR_SWAPPED;
    const int32_t b = bm->block_size;
    if (n_cow_out) *n_cow_out = 0;
    if (n == 0) return PA_OK;
    const int64_t new_tokens = s.tokens + n;
    const int64_t fresh = blocks_for(new_tokens, b) - (int64_t)s.blocks.size();
    // Writing into a partly filled last block that another table also holds
    // needs a private copy of it first.
    const bool cow = (s.tokens % b) != 0 && bm->refcount[s.blocks.back()] > 1;
    if ((int64_t)bm->free_stack.size() < fresh + (cow ? 1 : 0)) return PA_ERR_NO_BLOCKS;
    if (cow) {
        const int32_t src = s.blocks.back();
        const int32_t dst = bm->pop_block();
        bm->release_block(src);
        s.blocks.back() = dst;
        if (cow_pair_out) {
            cow_pair_out[0] = src;
            cow_pair_out[1] = dst;
        }
        if (n_cow_out) *n_cow_out = 1;
    }
    for (int64_t i = 0; i < fresh; ++i) s.blocks.push_back(bm->pop_block());
    if (slots_out)
        for (int64_t t = s.tokens; t < new_tokens; ++t)
            slots_out[t - s.tokens] = (int64_t)s.blocks[(size_t)(t / b)] * b + t % b;
    s.tokens = new_tokens;
    return PA_OK;
}

pa_status pa_bm_fork(pa_bm *bm, int32_t parent, int32_t *child_out) {
    if (!bm || !child_out) return PA_ERR_INVALID_ARG;
    if (!bm->valid_seq(parent)) return PA_ERR_NOT_FOUND;
    if (bm->seqs[parent].swapped) return PA_ERR_SWAPPED;
    int32_t child;
    pa_status st = pa_bm_add_seq(bm, &child);
    if (st != PA_OK) return st;
    pa_bm::Seq &p = bm->seqs[parent];  // add_seq may have grown seqs: take references after it
    pa_bm::Seq &c = bm->seqs[child];
    c.blocks = p.blocks;
    c.tokens = p.tokens;
    for (int32_t blk : c.blocks) ++bm->refcount[blk];
    *child_out = child;
    return PA_OK;
}

pa_status pa_bm_free_seq(pa_bm *bm, int32_t seq) {
    if (!bm) return PA_ERR_INVALID_ARG;
    if (!bm->valid_seq(seq)) return PA_ERR_NOT_FOUND;
    pa_bm::Seq &s = bm->seqs[seq];
    if (s.swapped)
        for (int32_t h : s.blocks) bm->host_free.push_back(h);
    else
        for (int32_t blk : s.blocks) bm->release_block(blk);
    s.blocks.clear();
    s.tokens = 0;
    s.live = false;
    s.swapped = false;
    bm->free_seq_ids.push_back(seq);
    return PA_OK;
}

pa_status pa_bm_get_table(const pa_bm *bm, int32_t seq, int32_t *table_out, int32_t cap, int32_t *num_blocks_out,
                          int64_t *num_tokens_out) {
    if (!bm || cap < 0 || (cap > 0 && !table_out)) return PA_ERR_INVALID_ARG;
    if (!bm->valid_seq(seq)) return PA_ERR_NOT_FOUND;
    const pa_bm::Seq &s = bm->seqs[seq];
    if (s.swapped) return PA_ERR_SWAPPED;
    if ((int64_t)s.blocks.size() > cap && table_out) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < cap; ++i) table_out[i] = (size_t)i < s.blocks.size() ? s.blocks[i] : -1;
    if (num_blocks_out) *num_blocks_out = (int32_t)s.blocks.size();
    if (num_tokens_out) *num_tokens_out = s.tokens;
    return PA_OK;
}

int64_t pa_bm_num_free(const pa_bm *bm) { return bm ? (int64_t)bm->free_stack.size() : -1; }

int32_t pa_bm_refcount(const pa_bm *bm, int64_t block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->refcount[(size_t)block];
}

pa_status pa_bm_can_admit(const pa_bm *bm, int64_t prompt_tokens, int64_t watermark_blocks, int32_t *admit) {
    if (!bm || !admit || prompt_tokens < 0 || watermark_blocks < 0) return PA_ERR_INVALID_ARG;
    const int64_t need = blocks_for(prompt_tokens, bm->block_size) + 1 + watermark_blocks;
    *admit = (int64_t)bm->free_stack.size() >= need ? 1 : 0;
    return PA_OK;
}

pa_status pa_bm_set_host_pool(pa_bm *bm, int64_t host_blocks) {
    if (!bm || host_blocks < 0 || host_blocks > INT32_MAX) return PA_ERR_INVALID_ARG;
    if ((int64_t)bm->host_free.size() != bm->host_blocks) return PA_ERR_INVALID_ARG;   // slots in use
    bm->host_blocks = host_blocks;
    bm->host_free.clear();
    bm->host_free.reserve((size_t)host_blocks);
    for (int64_t h = host_blocks - 1; h >= 0; --h) bm->host_free.push_back((int32_t)h);
    return PA_OK;
}

pa_status pa_bm_swap_out(pa_bm *bm, int32_t seq, int32_t *pairs_out, int32_t cap, int32_t *n_pairs_out) {
    if (!bm || !n_pairs_out || cap < 0) return PA_ERR_INVALID_ARG;
    if (!bm->valid_seq(seq)) return PA_ERR_NOT_FOUND;
    pa_bm::Seq &s = bm->seqs[seq];
    if (s.swapped) return PA_ERR_SWAPPED;
    const size_t n = s.blocks.size();
    if ((int64_t)n > cap || (n > 0 && !pairs_out)) return PA_ERR_INVALID_ARG;
    if (bm->host_free.size() < n) return PA_ERR_NO_BLOCKS;
    for (size_t i = 0; i < n; ++i) {
        const int32_t dev = s.blocks[i], h = bm->pop_host();
        pairs_out[2 * i] = dev;
        pairs_out[2 * i + 1] = h;
        bm->release_block(dev);
        s.blocks[i] = h;
    }
    s.swapped = true;
    *n_pairs_out = (int32_t)n;
    return PA_OK;
}

pa_status pa_bm_swap_in(pa_bm *bm, int32_t seq, int32_t *pairs_out, int32_t cap, int32_t *n_pairs_out) {
    if (!bm || !n_pairs_out || cap < 0) return PA_ERR_INVALID_ARG;
    if (!bm->valid_seq(seq)) return PA_ERR_NOT_FOUND;
    pa_bm::Seq &s = bm->seqs[seq];
    if (!s.swapped) return PA_ERR_SWAPPED;
    const size_t n = s.blocks.size();
    if ((int64_t)n > cap || (n > 0 && !pairs_out)) return PA_ERR_INVALID_ARG;
    if (bm->free_stack.size() < n) return PA_ERR_NO_BLOCKS;
    for (size_t i = 0; i < n; ++i) {
        const int32_t h = s.blocks[i], dev = bm->pop_block();
        pairs_out[2 * i] = dev;
        pairs_out[2 * i + 1] = h;
        bm->host_free.push_back(h);
        s.blocks[i] = dev;
    }
    s.swapped = false;
    *n_pairs_out = (int32_t)n;
    return PA_OK;
}

int64_t pa_bm_num_free_host(const pa_bm *bm) { return bm ? (int64_t)bm->host_free.size() : -1; }

int32_t pa_bm_is_swapped(const pa_bm *bm, int32_t seq) {
    if (!bm || !bm->valid_seq(seq)) return -1;
    return bm->seqs[seq].swapped ? 1 : 0;
}

}  // extern "C"
