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
    // rows of each physical block that some sequence reads: a shared block
    // counts the longest prefix any of its sharers covers
    std::vector<int32_t> rows((size_t)num_blocks, 0);
    int64_t t = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int L = context_lens[s];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks_per_seq * block_size)
            return PKV_EINVAL;
        t += L;
        const int32_t *bt = block_tables + (int64_t)s * max_blocks_per_seq;
        const int nb = (L + block_size - 1) / block_size;
        for (int j = 0; j < nb; ++j) {
            const int32_t b = bt[j];
            if (b < 0 || (int64_t)b >= num_blocks)
                return PKV_EINVAL;
            rows[b] = std::max(rows[b], std::min(block_size, L - j * block_size));
        }
    }
    int64_t nb = 0, slots = 0;
    for (int32_t r : rows)
        if (r > 0) {
            ++nb;
            slots += r;
        }
    *tokens = t;
    *blocks = nb;
    *occupied_slots = slots;
    return PKV_OK;
}
