// pkv_usage.cu -- memory accounting of a paged KV cache (host).
//
// PagedAttention takes blocks on demand, so a sequence of L tokens holds
// ceil(L / bs) blocks and wastes only the unused tail of its last block, and
// sequences that share a prefix hold its blocks once (PagedAttention:
// Efficient LLM Serving with vLLM, "Memory Efficiency" and "Advanced
// Features").  This counts, from the block tables themselves, the distinct
// blocks in use and the token slots they hold, so that a caller can set the
// paged cache's waste against reserving a fixed length per sequence.
#include <algorithm>
#include <cstdint>
#include <new>
#include <vector>

#include "../../include/pkv.h"

extern "C" int pkv_kv_cache_usage(const int32_t *block_tables, const int32_t *context_lens,
                                  int num_seqs, int max_blocks_per_seq, int block_size,
                                  int64_t num_blocks, int64_t *tokens, int64_t *blocks,
                                  int64_t *occupied_slots)
{
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0 ||
        (num_seqs > 0 && (!block_tables || !context_lens)) || !tokens || !blocks || !occupied_slots)
        return PKV_EINVAL;
    // lengths and block ids first, and the largest id in use, which sizes
    // the per-block array below (whatever num_blocks says)
    int32_t max_id = -1;
    for (int s = 0; s < num_seqs; ++s) {
        const int L = context_lens[s];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks_per_seq * block_size)
            return PKV_EINVAL;
        const int32_t *bt = block_tables + (int64_t)s * max_blocks_per_seq;
        const int64_t nbl = ((int64_t)L + block_size - 1) / block_size;
        for (int64_t j = 0; j < nbl; ++j) {
            if (bt[j] < 0 || (int64_t)bt[j] >= num_blocks)
                return PKV_EINVAL;
            max_id = std::max(max_id, bt[j]);
        }
    }
    // rows of each physical block that some sequence reads: a shared block
    // counts the longest prefix any of its sharers covers
    int64_t t = 0, nb = 0, slots = 0;
    try {
        std::vector<int32_t> rows((size_t)max_id + 1, 0);
        for (int s = 0; s < num_seqs; ++s) {
            const int L = context_lens[s];
            t += L;
            const int32_t *bt = block_tables + (int64_t)s * max_blocks_per_seq;
            const int64_t nbl = ((int64_t)L + block_size - 1) / block_size;
            for (int64_t j = 0; j < nbl; ++j) {
                int32_t &r = rows[(size_t)bt[j]];
                r = std::max(r, (int32_t)std::min<int64_t>(block_size, L - j * block_size));
            }
        }
        for (int32_t r : rows)
            if (r > 0) {
                ++nb;
                slots += r;
            }
    } catch (const std::bad_alloc &) {
        return PKV_EHOSTMEM;
    }
    *tokens = t;
    *blocks = nb;
    *occupied_slots = slots;
    return PKV_OK;
}
