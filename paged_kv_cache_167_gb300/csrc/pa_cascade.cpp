// pa_cascade.cpp -- host planning of a cascade decode (pa_cascade_plan).
//
// A group of sequences whose tables begin with the same physical blocks holds
// that prefix once (how-pagedattention-works (aiinfrainterviews.com), the
// shared-system-prompt paragraph; auto-20261007-1900-en (lihaoran.work),
// "Shared prefixes need matching computation").  The plan splits each table
// at the end of the run its group shares, so that the prefix can be attended
// once for the whole group (pa_prefix_attention) and each sequence's own
// blocks on their own (pa_decode_cascade).
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "pa.h"

pa_status pa_cascade_plan(const int32_t *tables, int32_t max_blocks, const int32_t *seq_lens, int32_t num_seqs,
                          int32_t group_size, int32_t block_size, int32_t *prefix_tables, int32_t *prefix_lens,
                          int32_t *group_order, int32_t *suffix_tables, int32_t *suffix_lens) {
    if (num_seqs < 0 || group_size <= 0 || block_size <= 0 || max_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (num_seqs % group_size != 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!tables || !seq_lens || !prefix_tables || !prefix_lens || !suffix_tables || !suffix_lens)
        return PA_ERR_INVALID_ARG;
    const int64_t cap = (int64_t)max_blocks * block_size;
    for (int32_t s = 0; s < num_seqs; ++s)
        if (seq_lens[s] < 0 || seq_lens[s] > cap) return PA_ERR_INVALID_ARG;
    const int32_t num_groups = num_seqs / group_size;
    for (int32_t gi = 0; gi < num_groups; ++gi) {
        const int32_t first = gi * group_size;
        int32_t min_len = seq_lens[first];
        for (int32_t k = 1; k < group_size; ++k)
            if (seq_lens[first + k] < min_len) min_len = seq_lens[first + k];
        // whole blocks only, and every member keeps at least one token of its own
        const int32_t limit = min_len > 0 ? (min_len - 1) / block_size : 0;
        int32_t shared = 0;
        while (shared < limit) {
            const int32_t id = tables[(int64_t)first * max_blocks + shared];
            bool same = id >= 0;
            for (int32_t k = 1; k < group_size && same; ++k)
                same = tables[(int64_t)(first + k) * max_blocks + shared] == id;
            if (!same) break;
            ++shared;
        }
        int32_t *prow = prefix_tables + (int64_t)gi * max_blocks;
        for (int32_t i = 0; i < max_blocks; ++i) prow[i] = i < shared ? tables[(int64_t)first * max_blocks + i] : -1;
        prefix_lens[gi] = shared * block_size;
        for (int32_t k = 0; k < group_size; ++k) {
            const int32_t s = first + k;
            const int32_t *row = tables + (int64_t)s * max_blocks;
            int32_t *srow = suffix_tables + (int64_t)s * max_blocks;
            for (int32_t i = 0; i < max_blocks; ++i) srow[i] = i + shared < max_blocks ? row[i + shared] : -1;
            suffix_lens[s] = seq_lens[s] - shared * block_size;
        }
    }
    if (group_order) {   // longest prefix first, ties in index order
        std::vector<int32_t> order(num_groups);
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t a, int32_t b) { return prefix_lens[a] > prefix_lens[b]; });
        std::copy(order.begin(), order.end(), group_order);
    }
    return PA_OK;
}
