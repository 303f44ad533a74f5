// pkv_block_pool.cu -- host allocator of the physical blocks of a paged KV
// cache, with prefix caching.
//
// Blocks are taken on demand, one more whenever a sequence's last block is
// full ("The PagedAttention Algorithm", Steps 1-3); sharers hold a block
// through a reference count and a write into a shared block copies it first
// ("Advanced Features", KV-Cache Sharing (Copy-on-Write)); and the blocks of
// a common prompt prefix stay cached so that later requests starting with
// the same tokens reuse them instead of recomputing them ("Advanced
// Features", Prefix Caching) -- all on the page "PagedAttention: Efficient
// LLM Serving with vLLM".
//
// A full block of a prompt is cached under a key that chains the keys of the
// blocks before it with its own tokens, so a hit means the same tokens at the
// same positions after the same prefix; the tokens and the parent key are
// kept with the entry and compared on every hit, so a key collision can only
// cost a miss.  Cached blocks no sequence holds stay reusable until the pool
// runs out of free blocks, then the least recently released goes first.
#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

namespace {

// The SplitMix64 output function (Steele, Lea, Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014), used here to mix a chain key.
uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

constexpr uint64_t kRootKey = 0x243f6a8885a308d3ull;   // key "before" the first block

uint64_t chain_key(uint64_t parent, const int32_t *tokens, int n)
{
    uint64_t h = mix64(parent ^ 0x9e3779b97f4a7c15ull);
    for (int i = 0; i < n; ++i)
        h = mix64(h ^ (uint64_t)(uint32_t)tokens[i]);
    return h;
}

}  // namespace

struct pkv_block_pool {
    int64_t num_blocks;
    int block_size;
    std::vector<int32_t> refs;              // holders per block
    std::vector<int32_t> free_list;         // blocks nobody holds and nothing caches
    std::vector<char> cached;               // block is a prefix-cache entry
    std::vector<uint64_t> key, parent;      // chain key of a cached block and of its parent
    std::vector<int32_t> tokens;            // [num_blocks * block_size] tokens of cached blocks
    std::unordered_map<uint64_t, int32_t> by_key;
    std::list<int32_t> lru;                 // cached blocks nobody holds, least recent first
    std::vector<std::list<int32_t>::iterator> lru_pos;
    uint64_t hits = 0, lookups = 0;

    int64_t available() const { return (int64_t)free_list.size() + (int64_t)lru.size(); }

    // a block for a new holder: a free one, else the least recently released
    // cached one (its cache entry goes)
    int32_t take()
    {
        int32_t b;
        if (!free_list.empty()) {
            b = free_list.back();
            free_list.pop_back();
        } else if (!lru.empty()) {
            b = lru.front();
            lru.pop_front();
            by_key.erase(key[b]);
            cached[b] = 0;
        } else {
            return -1;
        }
        refs[b] = 1;
        return b;
    }

    void hold(int32_t b)
    {
        if (refs[b]++ == 0 && cached[b])
            lru.erase(lru_pos[b]);
    }

    void drop(int32_t b)
    {
        if (--refs[b] > 0)
            return;
        if (cached[b])
            lru_pos[b] = lru.insert(lru.end(), b);
        else
            free_list.push_back(b);
    }

    // the cached block that holds `toks` after the prefix keyed `par`, or -1
    int32_t find(uint64_t k, uint64_t par, const int32_t *toks) const
    {
        auto it = by_key.find(k);
        if (it == by_key.end())
            return -1;
        const int32_t b = it->second;
        if (parent[b] != par ||
            std::memcmp(&tokens[(size_t)b * block_size], toks, sizeof(int32_t) * block_size) != 0)
            return -1;
        return b;
    }
};

namespace {

bool valid_table(const pkv_block_pool *p, const int32_t *table, int n)
{
    if (n < 0 || (n > 0 && !table))
        return false;
    for (int i = 0; i < n; ++i)
        if (table[i] < 0 || table[i] >= p->num_blocks || p->refs[table[i]] <= 0)
            return false;
    return true;
}

// Runs the body of a pool call that may allocate (a cache entry, an
// eviction-order node): a failed host allocation becomes a status instead of
// an exception through the C ABI (the pool may then be left part way
// through the call).
template <typename F>
int guarded(F &&body)
{
    try {
        return body();
    } catch (const std::bad_alloc &) {
        return PKV_EHOSTMEM;
    }
}

}  // namespace

extern "C" {

pkv_block_pool *pkv_block_pool_create(int64_t num_blocks, int block_size)
{
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0 || block_size > 65536)
        return nullptr;
    pkv_block_pool *p = new (std::nothrow) pkv_block_pool;
    if (!p)
        return nullptr;
    try {
        p->num_blocks = num_blocks;
        p->block_size = block_size;
        p->refs.assign((size_t)num_blocks, 0);
        p->cached.assign((size_t)num_blocks, 0);
        p->key.assign((size_t)num_blocks, 0);
        p->parent.assign((size_t)num_blocks, 0);
        p->tokens.assign((size_t)num_blocks * block_size, 0);
        p->lru_pos.resize((size_t)num_blocks);
        p->free_list.resize((size_t)num_blocks);
        for (int64_t i = 0; i < num_blocks; ++i)   // block 0 is handed out first
            p->free_list[(size_t)i] = (int32_t)(num_blocks - 1 - i);
    } catch (...) {
        delete p;
        return nullptr;
    }
    return p;
}

void pkv_block_pool_destroy(pkv_block_pool *pool) { delete pool; }

int64_t pkv_block_pool_available(const pkv_block_pool *pool)
{
    return pool ? pool->available() : -1;
}

int pkv_block_pool_refcount(const pkv_block_pool *pool, int32_t block)
{
    if (!pool || block < 0 || block >= pool->num_blocks)
        return -1;
    return pool->refs[block];
}

int pkv_block_pool_is_cached(const pkv_block_pool *pool, int32_t block)
{
    if (!pool || block < 0 || block >= pool->num_blocks)
        return -1;
    return pool->cached[block];
}

int pkv_block_pool_allocate(pkv_block_pool *pool, int n, int32_t *out)
{
    if (!pool || n < 0 || (n > 0 && !out))
        return PKV_EINVAL;
    if (pool->available() < n)
        return PKV_EWORKSPACE;
    for (int i = 0; i < n; ++i)
        out[i] = pool->take();
    return PKV_OK;
}

int pkv_block_pool_allocate_prompt(pkv_block_pool *pool, const int32_t *tokens, int num_tokens,
                                   int32_t *table, int table_capacity, int *cached_tokens)
{
    if (!pool || num_tokens < 0 || (num_tokens > 0 && (!tokens || !table)) || !cached_tokens)
        return PKV_EINVAL;
    const int bs = pool->block_size;
    const int64_t nb64 = ((int64_t)num_tokens + bs - 1) / bs;
    if (nb64 > table_capacity)
        return PKV_EINVAL;
    const int nb = (int)nb64, full = num_tokens / bs;
    return guarded([&] {
        // the longest run of leading full blocks the cache holds
        int reused = 0;
        uint64_t k = kRootKey;
        for (; reused < full; ++reused) {
            const int32_t *toks = tokens + (size_t)reused * bs;
            const uint64_t kn = chain_key(k, toks, bs);
            ++pool->lookups;
            const int32_t b = pool->find(kn, k, toks);
            if (b < 0)
                break;
            ++pool->hits;
            table[reused] = b;
            k = kn;
        }
        // reused blocks nobody holds sit in the eviction order but cannot
        // serve as this request's fresh blocks; a request that cannot be
        // served is refused before anything changes (the eviction order
        // included)
        int64_t idle = 0;
        for (int i = 0; i < reused; ++i)
            idle += pool->refs[table[i]] == 0;
        if (pool->available() - idle < nb - reused)
            return (int)PKV_EWORKSPACE;
        // holding the reused blocks first keeps them out of the eviction order
        for (int i = 0; i < reused; ++i)
            pool->hold(table[i]);
        for (int i = reused; i < nb; ++i)
            table[i] = pool->take();
        *cached_tokens = reused * bs;
        return (int)PKV_OK;
    });
}

int pkv_block_pool_commit_prompt(pkv_block_pool *pool, const int32_t *tokens, int num_tokens,
                                 const int32_t *table)
{
    if (!pool || num_tokens < 0 || (num_tokens > 0 && !tokens))
        return PKV_EINVAL;
    const int bs = pool->block_size, full = num_tokens / bs;
    if (!valid_table(pool, table, full))
        return PKV_EINVAL;
    return guarded([&] {
        uint64_t k = kRootKey;
        for (int i = 0; i < full; ++i) {
            const int32_t *toks = tokens + (size_t)i * bs;
            const uint64_t kn = chain_key(k, toks, bs);
            const int32_t b = table[i];
            if (!pool->cached[b] && pool->by_key.find(kn) == pool->by_key.end()) {
                pool->cached[b] = 1;
                pool->key[b] = kn;
                pool->parent[b] = k;
                std::memcpy(&pool->tokens[(size_t)b * bs], toks, sizeof(int32_t) * bs);
                pool->by_key.emplace(kn, b);
            }
            k = kn;
        }
        return (int)PKV_OK;
    });
}

int pkv_block_pool_fork(pkv_block_pool *pool, const int32_t *table, int num_blocks)
{
    if (!pool || !valid_table(pool, table, num_blocks))
        return PKV_EINVAL;
    for (int i = 0; i < num_blocks; ++i)
        pool->hold(table[i]);
    return PKV_OK;
}

int pkv_block_pool_release(pkv_block_pool *pool, const int32_t *table, int num_blocks)
{
    if (!pool || !valid_table(pool, table, num_blocks))
        return PKV_EINVAL;
    return guarded([&] {
        for (int i = 0; i < num_blocks; ++i)
            pool->drop(table[i]);
        return (int)PKV_OK;
    });
}

int pkv_block_pool_prepare_write(pkv_block_pool *pool, int32_t *table, int logical_block,
                                 int64_t *copy_pair)
{
    if (!pool || !table || logical_block < 0 || !copy_pair ||
        !valid_table(pool, table + logical_block, 1))
        return PKV_EINVAL;
    const int32_t b = table[logical_block];
    if (pool->refs[b] == 1 && !pool->cached[b])
        return 0;                      // the writer is its only holder
    if (pool->available() < 1)
        return PKV_EWORKSPACE;
    return guarded([&] {
        const int32_t nb = pool->take();
        pool->drop(b);
        table[logical_block] = nb;
        copy_pair[0] = b;
        copy_pair[1] = nb;
        return 1;
    });
}

int pkv_block_pool_append_slots(pkv_block_pool *pool, int32_t *tables, int table_stride,
                                const int32_t *lens, int n, int64_t *slots, int64_t *copy_pairs,
                                int *num_pairs, int *num_done)
{
    if (!pool || n < 0 || table_stride <= 0 || !num_pairs || !num_done ||
        (n > 0 && (!tables || !lens || !slots || !copy_pairs)))
        return PKV_EINVAL;
    *num_pairs = 0;
    *num_done = 0;
    const int bs = pool->block_size;
    // every row checked before any changes: lengths, room for the new block
    // index, and the blocks holding the tokens so far held by someone
    for (int s = 0; s < n; ++s) {
        const int L = lens[s];
        if (L < 0 || L / bs >= table_stride ||
            !valid_table(pool, tables + (int64_t)s * table_stride, (int)(((int64_t)L + bs - 1) / bs)))
            return PKV_EINVAL;
    }
    // in batch order, as one call per sequence would: a sibling that shares
    // the block a copy left behind may then write it in place
    return guarded([&] {
        for (int s = 0; s < n; ++s) {
            int32_t *t = tables + (int64_t)s * table_stride;
            const int j = lens[s] / bs, off = lens[s] % bs;
            if (off == 0) {                       // the token starts a block
                if (pool->available() < 1)
                    return (int)PKV_EWORKSPACE;
                t[j] = pool->take();
            } else if (pool->refs[t[j]] > 1 || pool->cached[t[j]]) {   // shared: copy first
                if (pool->available() < 1)
                    return (int)PKV_EWORKSPACE;
                const int32_t b = t[j], nb = pool->take();
                pool->drop(b);
                t[j] = nb;
                copy_pairs[2 * (int64_t)*num_pairs] = b;
                copy_pairs[2 * (int64_t)*num_pairs + 1] = nb;
                ++*num_pairs;
            }
            slots[s] = (int64_t)t[j] * bs + off;
            ++*num_done;
        }
        return (int)PKV_OK;
    });
}

int pkv_block_pool_stats(const pkv_block_pool *pool, int64_t *free_blocks, int64_t *cached_blocks,
                         int64_t *evictable_blocks, uint64_t *lookups, uint64_t *hits)
{
    if (!pool)
        return PKV_EINVAL;
    if (free_blocks)
        *free_blocks = (int64_t)pool->free_list.size();
    if (cached_blocks)
        *cached_blocks = (int64_t)pool->by_key.size();
    if (evictable_blocks)
        *evictable_blocks = (int64_t)pool->lru.size();
    if (lookups)
        *lookups = pool->lookups;
    if (hits)
        *hits = pool->hits;
    return PKV_OK;
}

}  // extern "C"
