// Host code under AddressSanitizer and UndefinedBehaviorSanitizer: the
// shared-prefix planner, the block pool and the cache-usage accounting,
// called through their C ABI on random inputs, including the awkward ones
// (empty, negative and over-the-bound lengths, tables that are prefixes of
// others, out-of-range block ids, a pool that runs dry, scalar arguments at
// and past their limits).  The checks of what
// the calls compute live in the Python tests; this program only has to run
// to the end without a sanitizer report.  Built and run by
// tests/test_host_sanitizers.py.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <numeric>
#include <random>
#include <vector>

#include "../../include/pkv.h"

namespace {

std::mt19937_64 rng(12345);
int uni(int lo, int hi) { return std::uniform_int_distribution<int>(lo, hi)(rng); }   // inclusive
double unit() { return std::uniform_real_distribution<double>(0.0, 1.0)(rng); }
template <typename T> T pick(std::initializer_list<T> v) { return v.begin()[uni(0, (int)v.size() - 1)]; }

[[noreturn]] void fail(const char *what, long a, long b)
{
    std::printf("FAIL %s: %ld %ld\n", what, a, b);
    std::exit(2);
}

// One random batch: prompts shared by several members (some members ending
// inside the prompt), singletons, empty and invalid contexts, in random
// order; planned with a size query first and then for real.
void planner_case(long &planned, long &refused)
{
    const int bs = pick({8, 16, 32}), G = pick({1, 2, 4, 8}), Hk = uni(1, 4);
    std::vector<std::vector<int32_t>> rows;
    std::vector<int32_t> lens;
    int32_t next_block = 0;
    const int want = pick({1, 3, 20, 200, 900});
    while ((int)rows.size() < want) {
        if (unit() < 0.5) {
            const int prompt = uni(1, 3000), full = prompt / bs;
            std::vector<int32_t> shared(full);
            std::iota(shared.begin(), shared.end(), next_block);
            next_block += full;
            for (int m = uni(1, 40); m > 0; --m) {
                const int L = unit() < 0.15 ? uni(1, prompt) : prompt + uni(0, 500);
                const int nb = (L + bs - 1) / bs;
                std::vector<int32_t> r(shared.begin(), shared.begin() + std::min(nb, full));
                while ((int)r.size() < nb)
                    r.push_back(next_block++);
                rows.push_back(r);
                lens.push_back(L);
            }
        } else {
            const int L = unit() < 0.1 ? 0 : uni(0, 5000), nb = (L + bs - 1) / bs;
            std::vector<int32_t> r(nb);
            std::iota(r.begin(), r.end(), next_block);
            next_block += nb;
            rows.push_back(r);
            lens.push_back(L > 0 || unit() < 0.5 ? L : -uni(1, 5));
        }
    }
    const int B = (int)rows.size();
    std::vector<int> order(B);
    std::iota(order.begin(), order.end(), 0);
    std::shuffle(order.begin(), order.end(), rng);
    int MB = 1, mcl = 1;
    for (const auto &r : rows)
        MB = std::max(MB, (int)r.size());
    std::vector<int32_t> bt((size_t)B * MB, -1), cl(B);
    for (int s = 0; s < B; ++s) {
        const auto &r = rows[(size_t)order[s]];
        std::copy(r.begin(), r.end(), bt.begin() + (size_t)s * MB);
        cl[s] = lens[(size_t)order[s]];
        mcl = std::max(mcl, (int)cl[s]);
    }
    if (unit() < 0.1)
        mcl = std::max(1, mcl - uni(1, 100));   // some lengths above the bound: invalid
    mcl = std::min(mcl, MB * bs);
    const int target = unit() < 0.6 ? 0 : std::max(bs, 32) * uni(1, 8);
    const size_t cap = pkv_shared_plan_max_ints(B, G * Hk, Hk, mcl, target);
    size_t need = 0, ws = 0;
    int rc = pkv_plan_shared_prefix(bt.data(), cl.data(), B, MB, bs, G * Hk, Hk, 128, mcl, target,
                                    nullptr, 0, &need, &ws);
    if (rc == PKV_EUNSUPPORTED) {
        ++refused;
        return;
    }
    if (rc != PKV_EWORKSPACE)
        fail("size query status", rc, 0);
    if (need > cap)
        fail("plan size above its bound", (long)need, (long)cap);
    std::vector<int32_t> plan(need);
    rc = pkv_plan_shared_prefix(bt.data(), cl.data(), B, MB, bs, G * Hk, Hk, 128, mcl, target,
                                plan.data(), plan.size(), &need, &ws);
    if (rc != PKV_OK)
        fail("plan status", rc, 0);
    ++planned;
}

// Random tables with a few out-of-range block ids and lengths.
void usage_case()
{
    const int bs = pick({8, 16, 32}), B = uni(1, 50), MB = uni(1, 40), NB = uni(1, 500);
    std::vector<int32_t> bt((size_t)B * MB), cl(B);
    for (auto &x : bt)
        x = unit() < 0.02 ? uni(-3, NB + 3) : uni(0, NB - 1);
    for (auto &x : cl)
        x = unit() < 0.05 ? uni(-5, MB * bs + 5) : uni(0, MB * bs);
    int64_t tokens = 0, blocks = 0, slots = 0;
    (void)pkv_kv_cache_usage(bt.data(), cl.data(), B, MB, bs, NB, &tokens, &blocks, &slots);
}

// A pool driven by random requests: prompts that reuse a few cached
// prefixes, forks, releases, writes into shared blocks, growth.
void pool_case()
{
    const int bs = pick({8, 16}), NB = uni(8, 200);
    pkv_block_pool *pool = pkv_block_pool_create(NB, bs);
    if (!pool)
        fail("pool create", NB, bs);
    std::vector<std::vector<int32_t>> prefixes(4), live;
    for (auto &p : prefixes) {
        p.resize((size_t)uni(1, 60));
        for (auto &x : p)
            x = uni(0, 30);
    }
    for (int step = 0; step < 400; ++step) {
        const double op = unit();
        if (op < 0.35 || live.empty()) {
            std::vector<int32_t> toks(prefixes[(size_t)uni(0, 3)]);
            toks.resize((size_t)uni(0, (int)toks.size()));
            for (int n = uni(0, 30); n > 0; --n)
                toks.push_back(uni(0, 30));
            if (toks.empty())
                continue;
            const int nb = ((int)toks.size() + bs - 1) / bs;
            std::vector<int32_t> table((size_t)nb + 1, -7);
            int cached = 0;
            if (pkv_block_pool_allocate_prompt(pool, toks.data(), (int)toks.size(), table.data(),
                                               (int)table.size(), &cached) != PKV_OK)
                continue;
            table.resize((size_t)nb);
            if (unit() < 0.8)
                pkv_block_pool_commit_prompt(pool, toks.data(), (int)toks.size(), table.data());
            live.push_back(table);
        } else if (op < 0.5) {
            const size_t k = (size_t)uni(0, (int)live.size() - 1);
            pkv_block_pool_release(pool, live[k].data(), (int)live[k].size());
            live.erase(live.begin() + (long)k);
        } else if (op < 0.6) {
            const size_t k = (size_t)uni(0, (int)live.size() - 1);
            pkv_block_pool_fork(pool, live[k].data(), (int)live[k].size());
            live.push_back(live[k]);
        } else if (op < 0.8) {
            const size_t k = (size_t)uni(0, (int)live.size() - 1);
            if (live[k].empty())
                continue;
            int64_t pair[2] = {-1, -1};
            pkv_block_pool_prepare_write(pool, live[k].data(), uni(0, (int)live[k].size() - 1), pair);
        } else if (op < 0.9) {
            const size_t k = (size_t)uni(0, (int)live.size() - 1);
            int32_t fresh = -1;
            if (pkv_block_pool_allocate(pool, 1, &fresh) == PKV_OK)
                live[k].push_back(fresh);
        } else {
            // one token more for every live sequence, in one call: rows padded
            // to a common stride, a random position inside each last block or
            // at the start of the next
            const int n = (int)live.size(), stride = 72;
            std::vector<int32_t> rows((size_t)n * stride, -1), lens(n);
            for (int i = 0; i < n; ++i) {
                const auto &t = live[(size_t)i];
                std::copy(t.begin(), t.begin() + std::min<size_t>(t.size(), stride), rows.begin() + (size_t)i * stride);
                lens[i] = t.empty() ? 0 : ((int)t.size() - 1) * bs + uni(1, bs);
            }
            std::vector<int64_t> slots((size_t)std::max(n, 1)), pairs((size_t)std::max(n, 1) * 2);
            int np = 0, done = 0;
            const int rc = pkv_block_pool_append_slots(pool, rows.data(), stride, lens.data(), n,
                                                       slots.data(), pairs.data(), &np, &done);
            if (rc == PKV_OK || rc == PKV_EWORKSPACE)
                for (int i = 0; i < done; ++i) {
                    const int held = (lens[i] + bs - 1) / bs, now = lens[i] / bs + 1;
                    live[(size_t)i].assign(rows.begin() + (size_t)i * stride,
                                           rows.begin() + (size_t)i * stride + std::max(held, now));
                }
        }
        int64_t free_blocks, cached_blocks, evictable;
        uint64_t lookups, hits;
        pkv_block_pool_stats(pool, &free_blocks, &cached_blocks, &evictable, &lookups, &hits);
        if (pkv_block_pool_available(pool) < 0)
            fail("available", (long)pkv_block_pool_available(pool), step);
    }
    for (auto &t : live)
        pkv_block_pool_release(pool, t.data(), (int)t.size());
    pkv_block_pool_destroy(pool);
}

// Scalar arguments at and past their limits (sizes near INT_MAX, negative
// ones, a pool of huge blocks) with small valid arrays: every call must come
// back with a status, with no overflow and no exception through the C ABI.
long extreme_arguments()
{
    const int ext[] = {INT32_MIN, -1, 0, 1, 7, 16, 24, 65535, 1 << 20, INT32_MAX - 15, INT32_MAX};
    long calls = 0;
    for (int a : ext)
        for (int b : ext)
            for (int c : ext)
                for (int d : ext)
                    for (int e : ext) {
                        (void)pkv_shared_plan_max_ints(a, b, c, d, e);
                        ++calls;
                    }
    std::vector<int32_t> bt(4 * 8), cl(4, 5), plan(1 << 16);
    std::iota(bt.begin(), bt.end(), 0);
    size_t need = 0, ws = 0;
    for (int bs : ext)
        for (int H : ext)
            for (int Hk : ext)
                for (int D : ext)
                    for (int mcl : ext)
                        for (int P : ext) {
                            (void)pkv_plan_shared_prefix(bt.data(), cl.data(), 4, 8, bs, H, Hk, D, mcl, P,
                                                         plan.data(), plan.size(), &need, &ws);
                            ++calls;
                        }
    int64_t tokens = 0, blocks = 0, slots = 0;
    for (int bs : ext)
        for (int mb = 1; mb <= 8; ++mb)
            for (int64_t nb : {INT64_MIN, (int64_t)-1, (int64_t)0, (int64_t)1, (int64_t)64, INT64_MAX}) {
                (void)pkv_kv_cache_usage(bt.data(), cl.data(), 4, mb, bs, nb, &tokens, &blocks, &slots);
                ++calls;
            }
    for (int64_t nb : {INT64_MIN, (int64_t)-1, (int64_t)0, (int64_t)1, (int64_t)64})
        for (int bs : ext) {
            pkv_block_pool *pool = pkv_block_pool_create(nb, bs);
            if (pool) {
                int32_t out[4];
                for (int k : ext)
                    if (k <= 4)
                        (void)pkv_block_pool_allocate(pool, k, out);
                std::vector<int32_t> toks(64, 3), table(80);
                int cached = 0;
                for (int n : ext)
                    if (n <= 64)
                        (void)pkv_block_pool_allocate_prompt(pool, toks.data(), n, table.data(), 80, &cached);
                pkv_block_pool_destroy(pool);
            }
            ++calls;
        }
    return calls;
}

}  // namespace

int main()
{
    long planned = 0, refused = 0;
    for (int i = 0; i < 1500; ++i)
        planner_case(planned, refused);
    for (int i = 0; i < 3000; ++i)
        usage_case();
    for (int i = 0; i < 300; ++i)
        pool_case();
    const long extreme = extreme_arguments();
    std::printf("planned %ld refused %ld extreme-argument calls %ld\n", planned, refused, extreme);
    return 0;
}
