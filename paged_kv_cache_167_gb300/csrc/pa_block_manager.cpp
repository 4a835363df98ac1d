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
// Prefix cache.  how-pagedattention-works, the shared-system-prompt paragraph:
// a prompt prefix many requests share is kept once, every table pointing at
// its blocks, and a request that finds its prefix cached skips recomputing it.
// auto-20261007-1900-en, "Shared prefixes need matching computation": a
// block's keys and values depend on the whole preceding context and on the
// conditions of the computation, so a block is reused only when everything
// before it and a caller-given condition key (model, adapter, ...) match.
// The index therefore keys a full block by (its parent entry, the condition,
// its b token ids), compared exactly; the bucket hash chains a 64-bit FNV-1a
// hash (Fowler, Noll and Vo) of the token ids onto the parent's hash.  The
// index holds one reference on each cached block, so a cached prefix outlives
// the sequences that computed it.  A cached block that no sequence holds is
// evictable: when the free list runs dry, or on request, the least recently
// used such entry is dropped together with every entry below it (they could
// no longer be reached), and blocks left with no reference return to the free
// list.
//
// Free blocks sit on a stack that hands out the lowest ids first and reuses
// the most recently released block next.  The manager never touches the GPU;
// the copy it plans is executed by pa_copy_blocks.
#include <cstdint>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pa.h"

namespace {

struct PrefixKey {
    uint64_t hash = 0;       // chained content hash, the bucket hash only
    int32_t parent = -1;     // parent entry, -1 for a sequence's first block
    uint64_t condition = 0;
    std::vector<int32_t> tokens;
};
struct PrefixKeyHash {
    size_t operator()(const PrefixKey &k) const { return (size_t)k.hash; }
};
struct PrefixKeyEq {
    bool operator()(const PrefixKey &a, const PrefixKey &b) const {
        return a.parent == b.parent && a.condition == b.condition && a.tokens == b.tokens;
    }
};

constexpr uint64_t kFnvOffset = 14695981039346656037ull, kFnvPrime = 1099511628211ull;
uint64_t fnv_bytes(uint64_t h, uint64_t v, int nbytes) {
    for (int i = 0; i < nbytes; ++i) {
        h ^= (v >> (8 * i)) & 0xff;
        h *= kFnvPrime;
    }
    return h;
}

}  // namespace

struct pa_bm {
    struct Node {
        PrefixKey key;
        int32_t block = -1;
        uint64_t tick = 0;
        std::vector<int32_t> children;
    };
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

    // prefix cache
    std::vector<Node> nodes;
    std::vector<int32_t> free_nodes;
    std::unordered_map<PrefixKey, int32_t, PrefixKeyHash, PrefixKeyEq> index;
    std::vector<int32_t> node_of_block;             // entry caching the block, -1 if none
    std::set<std::pair<uint64_t, int32_t>> lru;     // (tick, entry) of entries no sequence holds
    uint64_t clock = 0;
    int64_t hit_tokens = 0, query_tokens = 0;

    bool valid_seq(int32_t s) const { return s >= 0 && (size_t)s < seqs.size() && seqs[s].live; }
    bool evictable(int32_t b) const { return node_of_block[b] >= 0 && refcount[b] == 1; }
    // Blocks an allocation can get: free ones plus cached ones no sequence holds.
    int64_t available() const { return (int64_t)free_stack.size() + (int64_t)lru.size(); }
    int32_t pop_block() {
        if (free_stack.empty()) evict_lru();
        const int32_t b = free_stack.back();
        free_stack.pop_back();
        refcount[b] = 1;
        return b;
    }
    void ref_inc(int32_t b) {
        if (evictable(b)) lru.erase({nodes[node_of_block[b]].tick, node_of_block[b]});
        ++refcount[b];
    }
    void release_block(int32_t b) {
        if (--refcount[b] == 0)
            free_stack.push_back(b);
        else if (evictable(b))
            lru.insert({nodes[node_of_block[b]].tick, node_of_block[b]});
    }
    void set_tick(int32_t n) {
        const int32_t b = nodes[n].block;
        if (evictable(b)) lru.erase({nodes[n].tick, n});
        nodes[n].tick = ++clock;
        if (evictable(b)) lru.insert({nodes[n].tick, n});
    }
    // The chain of entries matching tokens[0 .. n) block by block.
    void match(const int32_t *tokens, int64_t n, uint64_t condition, std::vector<int32_t> &chain) const {
        chain.clear();
        PrefixKey key;
        key.condition = condition;
        uint64_t h = fnv_bytes(kFnvOffset, condition, 8);
        for (int64_t i = 0; i + block_size <= n; i += block_size) {
            key.tokens.assign(tokens + i, tokens + i + block_size);
            key.hash = h = chain_hash(h, tokens + i);
            auto it = index.find(key);
            if (it == index.end()) break;
            chain.push_back(it->second);
            key.parent = it->second;
        }
    }
    uint64_t chain_hash(uint64_t parent_hash, const int32_t *tok) const {
        uint64_t h = fnv_bytes(kFnvOffset, parent_hash, 8);
        for (int32_t j = 0; j < block_size; ++j) h = fnv_bytes(h, (uint32_t)tok[j], 4);
        return h;
    }
    // Drops entry n and every entry below it, with the index's references.
    int64_t evict_subtree(int32_t n) {
        int64_t freed = 0;
        const int32_t parent = nodes[n].key.parent;
        if (parent >= 0) {
            std::vector<int32_t> &sib = nodes[parent].children;
            for (size_t i = 0; i < sib.size(); ++i)
                if (sib[i] == n) {
                    sib[i] = sib.back();
                    sib.pop_back();
                    break;
                }
        }
        std::vector<int32_t> stack{n};
        while (!stack.empty()) {
            const int32_t m = stack.back();
            stack.pop_back();
            Node &node = nodes[m];
            for (int32_t c : node.children) stack.push_back(c);
            const int32_t b = node.block;
            if (evictable(b)) lru.erase({node.tick, m});
            node_of_block[b] = -1;
            if (--refcount[b] == 0) {
                free_stack.push_back(b);
                ++freed;
            }
            index.erase(node.key);
            node = Node();
            free_nodes.push_back(m);
        }
        return freed;
    }
    int64_t evict_lru() {
        if (lru.empty()) return 0;
        return evict_subtree(lru.begin()->second);
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
    bm->node_of_block.assign((size_t)num_blocks, -1);
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
    if (bm->available() < fresh + (cow ? 1 : 0)) return PA_ERR_NO_BLOCKS;
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
    for (int32_t blk : c.blocks) bm->ref_inc(blk);
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
    *admit = bm->available() >= need ? 1 : 0;
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
    if (bm->available() < (int64_t)n) return PA_ERR_NO_BLOCKS;
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

pa_status pa_bm_prefix_match(const pa_bm *bm, const int32_t *tokens, int64_t n_tokens, uint64_t condition,
                             int64_t *matched_tokens_out) {
    if (!bm || !matched_tokens_out || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    std::vector<int32_t> chain;
    bm->match(tokens, n_tokens, condition, chain);
    *matched_tokens_out = (int64_t)chain.size() * bm->block_size;
    return PA_OK;
}

pa_status pa_bm_add_seq_cached(pa_bm *bm, const int32_t *tokens, int64_t n_tokens, uint64_t condition,
                               int32_t *seq_out, int64_t *matched_tokens_out) {
    if (!bm || !seq_out || !matched_tokens_out || n_tokens < 0 || (n_tokens > 0 && !tokens))
        return PA_ERR_INVALID_ARG;
    std::vector<int32_t> chain;
    bm->match(tokens, n_tokens, condition, chain);
    int32_t id;
    const pa_status st = pa_bm_add_seq(bm, &id);
    if (st != PA_OK) return st;
    pa_bm::Seq &s = bm->seqs[id];
    for (int32_t n : chain) {
        bm->ref_inc(bm->nodes[n].block);
        s.blocks.push_back(bm->nodes[n].block);
    }
    for (size_t i = chain.size(); i-- > 0;) bm->set_tick(chain[i]);   // deepest first: ancestors stay newer
    s.tokens = (int64_t)chain.size() * bm->block_size;
    bm->hit_tokens += s.tokens;
    bm->query_tokens += n_tokens;
    *seq_out = id;
    *matched_tokens_out = s.tokens;
    return PA_OK;
}

pa_status pa_bm_cache_seq(pa_bm *bm, int32_t seq, const int32_t *tokens, int64_t n_tokens, uint64_t condition,
                          int64_t *inserted_out) {
    if (!bm || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    if (!bm->valid_seq(seq)) return PA_ERR_NOT_FOUND;
    pa_bm::Seq &s = bm->seqs[seq];
    if (s.swapped) return PA_ERR_SWAPPED;
    if (n_tokens > s.tokens) return PA_ERR_INVALID_ARG;
    const int32_t b = bm->block_size;
    std::vector<int32_t> chain;
    PrefixKey key;
    key.condition = condition;
    uint64_t h = fnv_bytes(kFnvOffset, condition, 8);
    int64_t inserted = 0;
    for (int64_t i = 0; (i + 1) * b <= n_tokens; ++i) {
        key.tokens.assign(tokens + i * b, tokens + (i + 1) * b);
        key.hash = h = bm->chain_hash(h, tokens + i * b);
        auto it = bm->index.find(key);
        int32_t n;
        if (it != bm->index.end()) {
            n = it->second;                               // already cached (maybe in another block)
        } else {
            const int32_t blk = s.blocks[(size_t)i];
            if (bm->node_of_block[blk] >= 0) break;       // held under other content: stop here
            if (!bm->free_nodes.empty()) {
                n = bm->free_nodes.back();
                bm->free_nodes.pop_back();
            } else {
                n = (int32_t)bm->nodes.size();
                bm->nodes.emplace_back();
            }
            pa_bm::Node &node = bm->nodes[n];
            node.key = key;
            node.block = blk;
            node.children.clear();
            if (key.parent >= 0) bm->nodes[key.parent].children.push_back(n);
            bm->ref_inc(blk);                             // the index's reference
            bm->node_of_block[blk] = n;
            bm->index.emplace(key, n);
            ++inserted;
        }
        chain.push_back(n);
        key.parent = n;
    }
    for (size_t i = chain.size(); i-- > 0;) bm->set_tick(chain[i]);
    if (inserted_out) *inserted_out = inserted;
    return PA_OK;
}

pa_status pa_bm_prefix_evict(pa_bm *bm, int64_t n_blocks, int64_t *freed_out) {
    if (!bm || n_blocks < 0) return PA_ERR_INVALID_ARG;
    int64_t freed = 0;
    while (freed < n_blocks && !bm->lru.empty()) freed += bm->evict_lru();
    if (freed_out) *freed_out = freed;
    return PA_OK;
}

int64_t pa_bm_num_cached(const pa_bm *bm) { return bm ? (int64_t)bm->index.size() : -1; }

int64_t pa_bm_num_evictable(const pa_bm *bm) { return bm ? (int64_t)bm->lru.size() : -1; }

pa_status pa_bm_prefix_stats(const pa_bm *bm, int64_t *hit_tokens_out, int64_t *query_tokens_out) {
    if (!bm || !hit_tokens_out || !query_tokens_out) return PA_ERR_INVALID_ARG;
    *hit_tokens_out = bm->hit_tokens;
    *query_tokens_out = bm->query_tokens;
    return PA_OK;
}

}  // extern "C"
