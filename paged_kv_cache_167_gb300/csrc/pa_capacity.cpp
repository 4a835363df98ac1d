// pa_capacity.cpp -- how many requests of a given length mix fit a KV budget
// when each reserves max_seq_len tokens contiguously, against when each holds
// only ceil(L / b) blocks with a shared prompt prefix stored once, and how much
// of the reserved or held memory stays unused.
//
// how-pagedattention-works (aiinfrainterviews.com), "A strong answer": the
// worked Llama 3.1 70B example (a contiguous allocator reserves max_seq_len
// tokens per request; paged requests hold whole blocks, so only the last
// block of each is partly empty) and the shared-system-prompt paragraph (one
// set of prefix blocks, referenced by every conversation's table).
// auto-20261007-1900-en (lihaoran.work), "How many tail slots remain unused?":
// ceil(T / b) blocks and ceil(T / b) * b - T idle slots per sequence.
//
// Closed-form host arithmetic: O(n) over the length list however large the
// budget, so a scheduler can call it per admission decision.
#include <cstdint>
#include <limits>

#include "pa.h"

namespace {

int64_t blocks_for(int64_t tokens, int64_t b) { return (tokens + b - 1) / b; }

}  // namespace

extern "C" pa_status pa_capacity_estimate(const int64_t *lens, int64_t n_lens, int64_t shared_prefix_tokens,
                                          int32_t block_size, int64_t max_seq_len, int64_t bytes_per_token,
                                          int64_t budget_bytes, pa_capacity *out) {
    if (!lens || !out || n_lens <= 0 || block_size <= 0 || max_seq_len <= 0 || bytes_per_token <= 0 ||
        budget_bytes < 0 || shared_prefix_tokens < 0)
        return PA_ERR_INVALID_ARG;
    const int64_t b = block_size;
    const int64_t kMax = std::numeric_limits<int64_t>::max();
    if (max_seq_len > kMax / bytes_per_token || b > kMax / bytes_per_token) return PA_ERR_INVALID_ARG;
    const int64_t shared_blocks = shared_prefix_tokens / b;   // whole prefix blocks, stored once

    int64_t private_blocks = 0;   // one pass over the list, shared blocks excluded
    double used = 0.0, held = 0.0;
    for (int64_t i = 0; i < n_lens; ++i) {
        if (lens[i] < shared_prefix_tokens || lens[i] > max_seq_len) return PA_ERR_INVALID_ARG;
        private_blocks += blocks_for(lens[i], b) - shared_blocks;
        used += (double)lens[i];
        held += (double)(blocks_for(lens[i], b) * b);
    }
    if (private_blocks == 0) return PA_ERR_INVALID_ARG;   // the list would admit without end

    out->contiguous_requests = budget_bytes / (max_seq_len * bytes_per_token);
    out->contiguous_waste = 1.0 - used / ((double)n_lens * (double)max_seq_len);
    out->paged_waste = 1.0 - used / held;
    out->mean_tail_slots = (held - used) / (double)n_lens;
    out->prefix_bytes_contiguous = (double)n_lens * (double)shared_prefix_tokens * (double)bytes_per_token;
    out->prefix_bytes_paged = ((double)(shared_blocks * b) +
                               (double)n_lens * (double)(shared_prefix_tokens - shared_blocks * b)) *
                              (double)bytes_per_token;

    // Paged admission takes requests from the list in turn until one does not
    // fit: whole passes first, then the prefix of one more pass.
    int64_t left = budget_bytes / (b * bytes_per_token);
    int64_t count = 0;
    if (left >= shared_blocks) {
        left -= shared_blocks;
        const int64_t passes = left / private_blocks;
        count = passes * n_lens;
        left -= passes * private_blocks;
        for (int64_t i = 0; i < n_lens; ++i) {
            const int64_t need = blocks_for(lens[i], b) - shared_blocks;
            if (need > left) break;
            left -= need;
            ++count;
        }
    }
    out->paged_requests = count;
    return PA_OK;
}
