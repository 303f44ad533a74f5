/*
 * pkv.h -- C ABI of the paged KV-cache decode library (libpkv.so), sm_103a.
 *
 * The operations follow the PagedAttention pages:
 *   - "PagedAttention: Efficient LLM Serving with vLLM", section "The
 *     PagedAttention Algorithm", Steps 1-5: the KV cache is cut into blocks
 *     of a fixed number of tokens that may sit anywhere in GPU memory; a
 *     per-sequence page table maps logical block j to its physical block;
 *     attention gathers K/V from the scattered blocks through that table.
 *   - same page, "Advanced Features", KV-Cache Sharing (Copy-on-Write):
 *     sequences share blocks until one of them writes.
 *   - "Efficient Memory Management for Large Language Model Serving with
 *     PagedAttention" (card), "Key ideas": blocks addressed through a
 *     per-sequence block table; prefix blocks shared across sequences.
 *
 * Conventions shared by every call
 *   - Layouts are dense and row-major.  One KV cache (K or V) of one layer is
 *     [num_blocks, num_kv_heads, block_size, head_dim]: the block_size x
 *     head_dim rows of one (block, kv head) are contiguous.  A token at
 *     logical position i of sequence s sits in physical block
 *     block_tables[s * max_blocks_per_seq + i / block_size] at row
 *     i % block_size; its slot number is block * block_size + i % block_size.
 *   - Pointers are DEVICE pointers unless stated otherwise.  The caller owns
 *     every buffer, including the workspace; the library allocates no device
 *     memory; the one device buffer it has is the static 32 MiB array
 *     compiled into it for pkv_paged_attention_decode_static.  Its
 *     only state between calls is the engine choice (process-wide) and the
 *     last decode call's engine and launch count (per host thread).  Every
 *     call is asynchronous on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream) and returns
 *     after enqueueing its kernels.
 *   - Host-side argument errors return a negative pkv_status and enqueue
 *     nothing.  Data-dependent errors found on the GPU (a block id or slot
 *     out of range, an inconsistent context length, a bounded wait that ran
 *     out) are OR-ed into *device_status (may be NULL: not reported) with the
 *     PKV_DEV_* bits; the kernels skip the offending element and never trap.
 *     Read *device_status after synchronising the stream.
 *   - Element types: q, k_cache, v_cache share kv_dtype; arithmetic is fp32
 *     (fp32 accumulation for fp16/bf16 inputs).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2 } pkv_dtype;

typedef enum {
    PKV_OK = 0,
    PKV_EINVAL = -1,        /* bad pointer, size, shape or alignment */
    PKV_EUNSUPPORTED = -2,  /* valid request outside the built kernel set */
    PKV_ECUDA = -3,         /* a CUDA runtime/driver call failed */
    PKV_EWORKSPACE = -4,    /* workspace missing or too small */
    PKV_EHOSTMEM = -5       /* a host-side allocation failed (the planner, the usage
                               accounting or the block pool; a pool that returns it
                               may be left part way through the call) */
} pkv_status;

/* Bits OR-ed into *device_status by the kernels. */
#define PKV_DEV_BAD_BLOCK 1u        /* block id outside [0, num_blocks) */
#define PKV_DEV_BAD_SLOT 2u         /* slot outside [0, num_blocks * block_size) */
#define PKV_DEV_TIMEOUT 4u          /* a bounded wait on a TMA or tensor-core barrier gave up
                                       (2 s): the rows it served are zero */
#define PKV_DEV_BAD_CONTEXT_LEN 8u  /* context_lens[s] < 0 or beyond the table / max */
#define PKV_DEV_DRAIN_TIMEOUT 16u   /* after a timeout, the wait for the copies or products
                                       already issued gave up too: a CTA may have exited with
                                       them still writing its shared memory; treat the
                                       context as unreliable */

/* Supported shapes of the decode kernel. */
#define PKV_DEFAULT_PARTITION 512    /* tokens per split-context partition */

/*
 * Bytes of workspace pkv_paged_attention_decode needs for these sizes.
 * partition_size: as passed to the decode call (0 = automatic; the size
 * returned then covers whichever path the automatic choice takes).
 * Returns 0 if no workspace is needed or on invalid sizes.
 */
size_t pkv_paged_attention_workspace_bytes(int num_seqs, int num_heads, int max_context_len,
                                           int head_dim, int partition_size);

/*
 * paged_attention_decode -- single-query attention of every running sequence
 * over its paged K/V ("The PagedAttention Algorithm", Step 5).
 *
 * For query head h of sequence s, with G = num_heads / num_kv_heads and
 * kv head h / G, over the L = context_lens[s] tokens at logical positions
 * 0..L-1:
 *     out[s,h,:] = sum_i softmax_i(scale * q[s,h,:] . k_i) * v_i
 * L = 0 gives a zero row.
 *
 *   out        [num_seqs, num_heads, head_dim] of out_dtype (written)
 *   q          [num_seqs, num_heads, head_dim] of kv_dtype
 *   k_cache, v_cache  [num_blocks, num_kv_heads, block_size, head_dim] of
 *              kv_dtype, 16-byte aligned
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]; entries past
 *              ceil(L / block_size) are never read
 *   context_lens  int32 [num_seqs], each in [0, max_context_len]
 *   max_context_len  host-side upper bound of context_lens (sizes the grid);
 *              must be <= max_blocks_per_seq * block_size
 *   scale      softmax scale (e.g. 1/sqrt(head_dim))
 *   partition_size  0 = automatic; otherwise tokens per split-context
 *              partition (multiple of 32 and of block_size): each partition
 *              is reduced separately and the partials are merged by a
 *              log-sum-exp reduce kernel.  A value >= max_context_len forces
 *              the single-pass kernel.
 *   workspace  device buffer of at least
 *              pkv_paged_attention_workspace_bytes(...) bytes when the split
 *              path runs (may be NULL otherwise)
 * Supported: head_dim in {64, 128}; block_size in {8, 16, 32};
 * num_heads / num_kv_heads in {1, 2, 4, 8}; num_seqs and num_kv_heads up to
 * 65,535 (grid extents); dtypes as pkv_dtype.  PKV_EUNSUPPORTED otherwise.
 * Device errors: PKV_DEV_BAD_BLOCK / PKV_DEV_BAD_CONTEXT_LEN -> that
 * sequence's output rows (for the kv head group touched) are zero.
 */
int pkv_paged_attention_decode(void *out, int out_dtype, const void *q, const void *k_cache,
                               const void *v_cache, int kv_dtype, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, int max_context_len, float scale,
                               int partition_size, void *workspace, size_t workspace_bytes,
                               uint32_t *device_status, void *stream);

/*
 * plan_shared_prefix -- HOST planner of the shared-prefix (cascade) decode:
 * sequences forked from one prompt (parallel sampling, beam search, a common
 * system prompt; "Advanced Features", KV-Cache Sharing and Prefix Caching)
 * point their tables at the same physical blocks for the shared part.  The
 * planner orders the sequences by their block tables (lexicographically by
 * block id, valid contexts first, batch order among equal tables), so that
 * sequences whose tables start with the same block ids become neighbours
 * wherever they sit in the batch; it groups runs of such neighbours (at most
 * 24 / G sequences per group, G = num_heads / num_kv_heads) and cuts the
 * attention into work items: each partition of a group's shared prefix once
 * for all members' query heads, and every member's own tail.
 *
 *   block_tables, context_lens  HOST copies of the arrays the decode call
 *              will get on the device (same layout as for decode)
 *   partition_size  target tokens per work list (one CTA per kv head and
 *              list): a multiple of 32 and of block_size, at most 64 *
 *              block_size (PKV_EINVAL otherwise); 0 = automatic: one list per
 *              resident CTA slot of the current GPU (three per SM) over all kv
 *              heads, at least 64 tokens each.  A cut into more than 65,535
 *              lists (the grid's y extent: a partition_size far too small for
 *              the batch) returns PKV_EUNSUPPORTED.
 *              Per kv head the work is one stream of 16-token tiles: each
 *              group's shared prefix (once for all members' query heads), then
 *              each member's own tail, then the next group or ungrouped
 *              sequence.  The stream is cut into lists of nearly equal cost
 *              (tiles, plus ten tiles for every item after a list's first:
 *              what a CTA's switch between items costs); a list holds the
 *              pieces of the groups and sequences its range covers (work
 *              items), and each piece writes one partial per row.
 *   plan       HOST int32 buffer of plan_capacity_ints entries; receives the
 *              plan (opaque apart from plan[0] = number of lists, plan[1] =
 *              partial slots per (sequence, head) and plan[7] = number of
 *              items); copy it to the device and pass it to
 *              pkv_paged_attention_decode_shared
 *   plan_ints  out: entries the plan needs
 *   workspace_bytes  out: workspace the decode call needs for this plan
 * Returns PKV_EWORKSPACE (after filling both outputs) when plan is NULL or
 * too small; pkv_shared_plan_max_ints bounds the size in advance.  Takes
 * what the decode kernels take: block_size 8, 16 or 32, head_dim 64 or 128,
 * num_heads / num_kv_heads 1, 2, 4 or 8, max_context_len up to 2^30
 * (PKV_EUNSUPPORTED otherwise); PKV_EHOSTMEM if its host memory runs out.
 */
int pkv_plan_shared_prefix(const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                           int max_blocks_per_seq, int block_size, int num_heads,
                           int num_kv_heads, int head_dim, int max_context_len,
                           int partition_size, int32_t *plan, size_t plan_capacity_ints,
                           size_t *plan_ints, size_t *workspace_bytes);

/* Upper bound of plan_ints for these sizes. */
size_t pkv_shared_plan_max_ints(int num_seqs, int num_heads, int num_kv_heads, int max_context_len,
                                int partition_size);

/*
 * paged_attention_decode_shared -- the same attention as
 * pkv_paged_attention_decode, following a plan from pkv_plan_shared_prefix:
 * one CTA per (kv head, work list) takes the list's items in turn, reads each
 * shared block once for all the query heads of its group and writes the
 * output of a sequence an item holds entirely, or else one partial per row; a
 * second kernel, queued as a programmatic dependent of the first, merges the
 * partials (log-sum-exp).
 * Results equal the per-sequence path up to fp32 rounding order.
 *
 * Arguments as for pkv_paged_attention_decode, plus:
 *   plan       DEVICE copy of the plan (4-byte aligned; read only, so the
 *              same device plan serves any number of calls with the same
 *              tables and lengths, e.g. every layer of a step)
 *   num_lists, num_items, slots  plan[0], plan[7] and plan[1]
 *   workspace  at least the planner's workspace_bytes
 * The device checks the plan against the device arrays: every table the
 * plan reads must hold the block ids the plan was made with (PKV_DEV_BAD_BLOCK
 * and zero rows for the rows they serve otherwise), and every sequence's
 * context length must be the one it was made for (PKV_DEV_BAD_CONTEXT_LEN and
 * zero rows otherwise).
 * kv_dtype must be PKV_F16 or PKV_BF16 (fp32 caches: PKV_EUNSUPPORTED).
 * Enqueues two kernels.
 */
int pkv_paged_attention_decode_shared(void *out, int out_dtype, const void *q, const void *k_cache,
                                      const void *v_cache, int kv_dtype,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, int num_seqs, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, int max_context_len, float scale,
                                      const int32_t *plan, int num_lists, int num_items, int slots,
                                      void *workspace, size_t workspace_bytes,
                                      uint32_t *device_status, void *stream);

/*
 * kv_cache_usage -- HOST accounting of the paged cache ("Memory Efficiency":
 * blocks are taken on demand, so only the tail of a sequence's last block is
 * unused; "Advanced Features": sharers of a prefix hold its blocks once).
 *
 *   block_tables, context_lens  HOST arrays, layout as for decode
 *   num_blocks      size of the physical pool (block ids must lie in it)
 *   tokens          out: sum of the context lengths (tokens cached)
 *   blocks          out: distinct physical blocks the tables reference for
 *                   those tokens
 *   occupied_slots  out: token slots of those blocks that hold a token (a
 *                   shared block counts its longest sharer's rows)
 * The paged waste is 1 - occupied_slots / (blocks * block_size); reserving
 * R tokens per sequence instead wastes 1 - tokens / (num_seqs * R).  Returns
 * PKV_EINVAL for a negative length, a length beyond the table or a block id
 * outside [0, num_blocks).
 */
int pkv_kv_cache_usage(const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                       int max_blocks_per_seq, int block_size, int64_t num_blocks, int64_t *tokens,
                       int64_t *blocks, int64_t *occupied_slots);

/*
 * block pool -- HOST allocator of the physical blocks of one paged cache,
 * with prefix caching (page "PagedAttention: Efficient LLM Serving with
 * vLLM": blocks are taken on demand, "The PagedAttention Algorithm" Steps
 * 1-3; sharers hold a block by reference count and a write into a shared
 * block copies it first, "Advanced Features", KV-Cache Sharing; the blocks of
 * a common prompt prefix stay cached for later requests, "Advanced
 * Features", Prefix Caching).  A full prompt block is cached under a key
 * chained over its own tokens and every token before it; entries keep their
 * tokens, so a hit is exact.  A cached block nobody holds stays reusable
 * until the pool needs a block and has no free one: then the least recently
 * released goes.  Not thread-safe: one caller at a time per pool.
 */
typedef struct pkv_block_pool pkv_block_pool;

/* A pool of num_blocks (1 .. 2^31 - 1) blocks of block_size (1 .. 65536)
 * tokens; NULL on other sizes or when memory for it cannot be had.  Block 0
 * is handed out first. */
pkv_block_pool *pkv_block_pool_create(int64_t num_blocks, int block_size);
void pkv_block_pool_destroy(pkv_block_pool *pool);

/* Blocks for a new request's prompt: table[0 .. ceil(num_tokens /
 * block_size)) receives the longest run of leading full blocks the cache
 * holds for exactly these tokens (each now held once more), then fresh
 * blocks.  *cached_tokens = the tokens whose K/V those reused blocks already
 * hold (a multiple of block_size).  PKV_EWORKSPACE, with nothing taken, if
 * the pool cannot supply the rest; PKV_EINVAL if table_capacity is short. */
int pkv_block_pool_allocate_prompt(pkv_block_pool *pool, const int32_t *tokens, int num_tokens,
                                   int32_t *table, int table_capacity, int *cached_tokens);

/* Once the K/V of a prompt's tokens is in its blocks: caches its full
 * blocks that no entry holds yet, so later prompts with the same prefix
 * reuse them.  table must hold blocks the caller holds. */
int pkv_block_pool_commit_prompt(pkv_block_pool *pool, const int32_t *tokens, int num_tokens,
                                 const int32_t *table);

/* n fresh blocks (a growing sequence's next block): PKV_EWORKSPACE, with
 * nothing taken, if the pool has fewer. */
int pkv_block_pool_allocate(pkv_block_pool *pool, int n, int32_t *out);

/* A forked sequence holds every block of table once more. */
int pkv_block_pool_fork(pkv_block_pool *pool, const int32_t *table, int num_blocks);

/* The sequence lets go of its blocks: one holder fewer each; a block nobody
 * holds returns to the free list, or stays cached (reusable, evictable). */
int pkv_block_pool_release(pkv_block_pool *pool, const int32_t *table, int num_blocks);

/* Before writing into table[logical_block]: if another sequence holds that
 * block too, or it is a prefix-cache entry, the sequence gets a fresh block
 * in its place (table updated, one holder fewer on the old one) and
 * copy_pair = {old, new} for pkv_copy_blocks; returns 1 then, 0 when the
 * block can be written in place, PKV_EWORKSPACE when no block is left. */
int pkv_block_pool_prepare_write(pkv_block_pool *pool, int32_t *table, int logical_block,
                                 int64_t *copy_pair);

/* Room for one more token in each of n sequences, in one call (a decode
 * step's bookkeeping; "The PagedAttention Algorithm", Steps 1-3, and
 * "Advanced Features", KV-Cache Sharing).  Sequence s holds lens[s] tokens
 * in row s of tables (int32 [n, table_stride], host); its new token goes to
 * position lens[s]: a fresh block when that position starts a block (written
 * at index lens[s] / block_size), else the row's last block, copied first
 * (as prepare_write does) if another sequence or the prefix cache holds it.
 * Sequences are served in batch order, as one call each would be.
 *   slots       out, int64 [n]: block * block_size + offset of each new token
 *               (the slot mapping pkv_reshape_and_cache takes)
 *   copy_pairs  out, int64 [n, 2]: (source, copy) of each block copied, in
 *               order (what pkv_copy_blocks takes); *num_pairs of them
 *   num_done    out: sequences served
 * Every row is checked before anything changes (PKV_EINVAL: a negative
 * length, no room for the new block index, or a block nobody holds).
 * PKV_EWORKSPACE when the pool runs out: the first *num_done sequences are
 * served, the rest untouched.  PKV_EHOSTMEM as for the other pool calls. */
int pkv_block_pool_append_slots(pkv_block_pool *pool, int32_t *tables, int table_stride,
                                const int32_t *lens, int n, int64_t *slots, int64_t *copy_pairs,
                                int *num_pairs, int *num_done);

/* Blocks a new holder can get (free + cached ones nobody holds), -1 for a
 * NULL pool; holders of a block; whether it is a cache entry (-1 if out of
 * range); and counters (any pointer may be NULL). */
int64_t pkv_block_pool_available(const pkv_block_pool *pool);
int pkv_block_pool_refcount(const pkv_block_pool *pool, int32_t block);
int pkv_block_pool_is_cached(const pkv_block_pool *pool, int32_t block);
int pkv_block_pool_stats(const pkv_block_pool *pool, int64_t *free_blocks, int64_t *cached_blocks,
                         int64_t *evictable_blocks, uint64_t *lookups, uint64_t *hits);

/*
 * reshape_and_cache -- write each new token's key/value rows into its slot
 * ("The PagedAttention Algorithm", Step 2: generated tokens fill the block).
 *
 *   key, value   [num_tokens, num_kv_heads, head_dim] of dtype, 16-byte aligned
 *   k_cache, v_cache  [num_blocks, num_kv_heads, block_size, head_dim]
 *   slot_mapping int64 [num_tokens]; slot = block * block_size + row.
 *                A negative slot marks a padding token: skipped, no error.
 *                A slot >= num_blocks * block_size: skipped, PKV_DEV_BAD_SLOT.
 * Bit-exact copy.  Two tokens with the same slot in one call: undefined.
 */
int pkv_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                          int dtype, const int64_t *slot_mapping, int num_tokens,
                          int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                          uint32_t *device_status, void *stream);

/*
 * copy_blocks -- copy-on-write block copies ("Advanced Features", KV-Cache
 * Sharing (Copy-on-Write): sharers keep one copy of a block until one of
 * them writes to it, the way a forked process shares memory pages).
 *
 *   k_caches, v_caches  HOST arrays of num_layers DEVICE pointers, one K and
 *                one V cache per layer, each 16-byte aligned
 *   src_dst_pairs  int64 [num_pairs, 2] (device): block dst of every layer's
 *                K and V cache becomes a copy of block src
 *   block_bytes  bytes of one block of one cache (num_kv_heads * block_size *
 *                head_dim * element size), a multiple of 16
 * Pairs with an id outside [0, num_blocks): skipped, PKV_DEV_BAD_BLOCK.
 * Caller contract: destinations are distinct and no destination is also a
 * source in the same call.
 */
int pkv_copy_blocks(void *const *k_caches, void *const *v_caches, int num_layers,
                    const int64_t *src_dst_pairs, int num_pairs, size_t block_bytes,
                    int64_t num_blocks, uint32_t *device_status, void *stream);

/*
 * swap_blocks -- move whole blocks between the GPU pool and a host pool (a
 * preempted request's KV cache goes to CPU memory when the GPU is full and
 * comes back when it resumes: "vLLM: The Serving Engine", smart scheduling;
 * the paper's section 7.3 compares swapping with recomputation).  One
 * kernel moves all pairs of all layers, reading and writing the host pool
 * over the host link.
 *
 *   gpu_k, gpu_v    HOST arrays of num_layers DEVICE pointers to the caches
 *                   [gpu_blocks, Hk, bs, D], 16-byte aligned
 *   host_k, host_v  HOST arrays of num_layers pointers to HOST pools of
 *                   host_blocks blocks of the same size, pinned and mapped for
 *                   the device (cudaHostAlloc, or torch's pin_memory);
 *                   PKV_EINVAL otherwise
 *   pairs           int64 [num_pairs, 2] (device): (gpu block, host block)
 *   block_bytes     bytes of one block of one cache, a multiple of 16
 *   direction       PKV_SWAP_OUT (gpu block -> host block) or PKV_SWAP_IN
 *                   (host block -> gpu block)
 * Pairs with an id outside its pool: skipped, PKV_DEV_BAD_BLOCK.  Bit-exact
 * copy.  Caller contract: the destination blocks are distinct; the host
 * pools stay allocated until the stream has passed the call.
 */
enum { PKV_SWAP_OUT = 0, PKV_SWAP_IN = 1 };
int pkv_swap_blocks(void *const *gpu_k, void *const *gpu_v, void *const *host_k,
                    void *const *host_v, int num_layers, const int64_t *pairs, int num_pairs,
                    size_t block_bytes, int64_t gpu_blocks, int64_t host_blocks, int direction,
                    uint32_t *device_status, void *stream);

/*
 * paged_attention_decode_static -- the same attention as
 * pkv_paged_attention_decode, for callers that cannot allocate device
 * memory.  (The pages have no counterpart; this is a convenience of this
 * library.)  Callers of this kind include plugins whose host engine owns all
 * device memory and gives them none, code running under an allocator that
 * is full or must not grow, and latency-critical loops that must not call
 * cudaMalloc because it may synchronise the device.
 *
 * A context longer than one partition takes the split-context path, whose
 * partials live in a buffer inside libpkv.so: pkv_static_workspace_capacity()
 * bytes (32 MiB) on every GPU that uses it, held until the process exits.  A
 * batch whose contexts all fit one partition (max_context_len <=
 * partition_size) takes the single pass and uses no buffer.  It calls no
 * allocator.  The first call on a device looks up the buffer's address for
 * that device (cudaGetSymbolAddress, with the device current) and keeps it;
 * make that first call before any stream capture begins, and do not use the
 * library across a cudaDeviceReset (the kept address would be stale).
 *
 * Arguments as for pkv_paged_attention_decode, without the workspace;
 * partition_size 0 means PKV_DEFAULT_PARTITION tokens.  Returns
 * PKV_EWORKSPACE when the split path's num_seqs * num_heads *
 * ceil(max_context_len / partition_size) * (2 + head_dim) * 4 bytes (plus
 * alignment) exceed the capacity.  All calls on one device share the
 * buffer: calls whose kernels may overlap on the GPU (different streams
 * without ordering) race and give wrong results; calls ordered on one stream
 * are safe.  The buffer keeps the last call's partials; nothing in it needs
 * to start at zero (the partition pass writes every partial the reduce
 * reads).
 */
int pkv_paged_attention_decode_static(void *out, int out_dtype, const void *q,
                                      const void *k_cache, const void *v_cache, int kv_dtype,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, int num_seqs, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, int max_context_len, float scale,
                                      int partition_size, uint32_t *device_status, void *stream);

/* Bytes of the library-owned buffer pkv_paged_attention_decode_static uses. */
size_t pkv_static_workspace_capacity(void);

/*
 * Engine of the decode kernels, process-wide (tests and benchmarks compare
 * them): 0 = automatic (warp-level tensor-core MMA for 16-bit caches, CUDA
 * cores for fp32 caches), 1 = CUDA cores, 2 = warp-level tensor-core MMA
 * (16-bit caches only; fp32 caches then return PKV_EUNSUPPORTED), 3 =
 * tcgen05: the shared-prefix decode on tcgen05 MMAs with accumulators in
 * tensor memory (head_dim 128; other head dims return PKV_EUNSUPPORTED), the
 * per-sequence decode as for 2.  Returns PKV_EINVAL for other values.
 */
int pkv_decode_set_engine(int engine);

/* Engine (1, 2 or 3) of the last successful decode call on this host thread. */
int pkv_last_decode_engine(void);

/* Static, NUL-terminated description of a pkv_status value. */
const char *pkv_status_string(int status);

/*
 * Test hook of the kernels' bounded waits (no counterpart on the pages: it
 * exists so that the error path of a wait that gives up can run on a GPU
 * without faulting or hanging it).  Enqueues one CTA that waits, with the
 * bounded wait every decode kernel uses, on an mbarrier phase that nothing
 * completes (no arrival, no copy), then runs the drain wait that follows a
 * timeout in those kernels on the same phase.  Both give up after limit_ns
 * nanoseconds (1 .. 2e9) or max_polls polls (0: limit_ns / 4 polls, more than
 * the time limit lets through),
 * whichever comes first, and the CTA returns; *device_status (required)
 * then holds PKV_DEV_TIMEOUT | PKV_DEV_DRAIN_TIMEOUT.  The context stays
 * usable.  PKV_EINVAL for a NULL status or a limit outside the range.
 */
int pkv_test_bounded_wait(uint64_t limit_ns, uint64_t max_polls, uint32_t *device_status,
                          void *stream);

/* Number of kernels the last successful pkv_paged_attention_decode call on
 * this host thread enqueued (1 = single pass, 2 = partition pass + reduce). */
int pkv_last_decode_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
