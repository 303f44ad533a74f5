/*
 * pkv_oracle.c -- plain CPU reference ("oracle") for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline / reference legs of the benchmark load this library.  The
 * CUDA library never links, includes or calls it, and it shares no code,
 * header, table or helper with the CUDA library.
 *
 * Everything is computed in fp64 with the most direct loops available; speed
 * is not a goal.  Sources (the PagedAttention summary pages):
 *
 *   [P4-alg]  PagedAttention: Efficient LLM Serving with vLLM,
 *             "The PagedAttention Algorithm", Steps 1-5 (blocks of a fixed
 *             number of tokens, a page table from logical block to physical
 *             block, attention gathers K/V from the scattered blocks).
 *   [P4-mem]  same page, "Memory Efficiency" (100 tokens -> 7 blocks of 16).
 *   [P4-cow]  same page, "Advanced Features", KV-Cache Sharing
 *             (Copy-on-Write): shared blocks until the first write.
 *   [P2-key]  Efficient Memory Management for Large Language Model Serving
 *             with PagedAttention (card), "Key ideas": KV split into
 *             fixed-size blocks addressed through a per-sequence block table.
 *
 * The pages never write the attention formula down; they present paging as
 * memory management that leaves attention itself unchanged.  The oracle
 * therefore gathers each sequence's logical tokens into contiguous arrays and
 * applies textbook single-query softmax attention to them:
 *     z_i   = scale * sum_d q[d] * k_i[d]
 *     out   = sum_i exp(z_i - max z) * v_i / sum_i exp(z_i - max z)
 * Query head h reads kv head h / G with G = H / Hk (consecutive query heads
 * share one kv head; reduces to multi-head attention for G = 1).
 *
 * Cache layout: k_cache and v_cache are [num_blocks, Hk, block_size, D],
 * row-major.  A token at logical position i of sequence s lives in physical
 * block block_tables[s][i / bs] at offset i % bs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* Status bits reported by the oracle (same meaning as the library's device
 * status word, defined here on their own). */
enum { ORC_BAD_BLOCK = 1, ORC_BAD_SLOT = 2, ORC_BAD_LEN = 8 };

/* ------------------------------------------------------------------ decode */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double pkv_oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25);  /* (1024 + m) * 2^(e - 15 - 10) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double pkv_oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int elem_bytes(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

static double load_elem(const void *base, int dtype, int64_t i)
{
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * i, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char *)base + 2 * i, 2);
    return dtype == ORC_F16 ? pkv_oracle_f16_to_f64(h) : pkv_oracle_bf16_to_f64(h);
}

/* --------------------------------------------------------------- blocks */

/* Blocks a sequence of n tokens occupies: ceil(n / bs) [P4-mem]. */
int64_t pkv_oracle_blocks_for_tokens(int64_t n_tokens, int64_t block_size)
{
    return (n_tokens + block_size - 1) / block_size;
}

/* Copy the K and V rows of kv head `kvh` for logical positions 0..L-1 of one
 * sequence into contiguous fp64 arrays K[L][D], V[L][D] [P4-alg Step 4-5].
 * Returns a nonzero status if a referenced block id is out of range. */
static int gather_head(double *K, double *V, const void *k_cache, const void *v_cache,
                       int dtype, const int32_t *table, int L, int kvh, int Hk, int D,
                       int bs, int64_t num_blocks)
{
    for (int i = 0; i < L; ++i) {
        int64_t phys = table[i / bs];
        int off = i % bs;
        if (phys < 0 || phys >= num_blocks)
            return ORC_BAD_BLOCK;
        int64_t row = ((phys * Hk + kvh) * bs + off) * (int64_t)D;
        for (int d = 0; d < D; ++d) {
            K[(int64_t)i * D + d] = load_elem(k_cache, dtype, row + d);
            V[(int64_t)i * D + d] = load_elem(v_cache, dtype, row + d);
        }
    }
    return 0;
}

/* ------------------------------------------------------------ attention */

typedef struct {
    double *out;                 /* [B, H, D] */
    const void *q;               /* [B, H, D] in `dtype` */
    const void *k_cache, *v_cache;
    int dtype;
    const int32_t *block_tables; /* [B, max_blocks_per_seq] */
    int max_blocks_per_seq;
    const int32_t *context_lens; /* [B] */
    int B, H, Hk, D, bs;
    int64_t num_blocks;
    double scale;
    int partition_size;          /* 0: one pass; else partials merged by log-sum-exp */
    uint32_t *seq_status;        /* [B] */
    int tid, nthreads;
} attn_job;

/* Textbook softmax attention of one query vector over L contiguous rows. */
static void attend(double *o, const double *q, const double *K, const double *V,
                   int L, int D, double scale, double *z)
{
    double m = -INFINITY, l = 0.0;
    for (int i = 0; i < L; ++i) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q[d] * K[(int64_t)i * D + d];
        z[i] = scale * dot;
        if (z[i] > m)
            m = z[i];
    }
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    for (int i = 0; i < L; ++i) {
        double p = exp(z[i] - m);
        l += p;
        for (int d = 0; d < D; ++d)
            o[d] += p * V[(int64_t)i * D + d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= l;
}

/* The same result reached in partitions of P tokens: each partition keeps its
 * own maximum m_p, normaliser l_p and normalised output o_p; the partitions
 * are merged with weights l_p * exp(m_p - M), M = max_p m_p.  This is an exact
 * algebraic regrouping of `attend` (the split-context form of the kernel). */
static void attend_partitioned(double *o, const double *q, const double *K, const double *V,
                               int L, int D, double scale, int P, double *z, double *op)
{
    int np = (L + P - 1) / P;
    double M = -INFINITY;
    double *mp = (double *)malloc(sizeof(double) * (size_t)np);
    double *lp = (double *)malloc(sizeof(double) * (size_t)np);
    double *opart = (double *)malloc(sizeof(double) * (size_t)np * (size_t)D);
    for (int p = 0; p < np; ++p) {
        int i0 = p * P, i1 = i0 + P < L ? i0 + P : L;
        attend(op, q, K + (int64_t)i0 * D, V + (int64_t)i0 * D, i1 - i0, D, scale, z);
        double m = -INFINITY, l = 0.0;
        for (int i = 0; i < i1 - i0; ++i)
            if (z[i] > m)
                m = z[i];
        for (int i = 0; i < i1 - i0; ++i)
            l += exp(z[i] - m);
        mp[p] = m;
        lp[p] = l;
        memcpy(opart + (int64_t)p * D, op, sizeof(double) * (size_t)D);
        if (m > M)
            M = m;
    }
    double wsum = 0.0;
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    for (int p = 0; p < np; ++p) {
        double w = lp[p] * exp(mp[p] - M);
        wsum += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * opart[(int64_t)p * D + d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= wsum;
    free(mp);
    free(lp);
    free(opart);
}

static void *attn_worker(void *arg)
{
    attn_job *j = (attn_job *)arg;
    int G = j->H / j->Hk;
    int maxL = 0;
    for (int s = 0; s < j->B; ++s)
        if (j->context_lens[s] > maxL)
            maxL = j->context_lens[s];
    size_t rows = (size_t)(maxL > 0 ? maxL : 1);
    double *K = (double *)malloc(sizeof(double) * rows * (size_t)j->D);
    double *V = (double *)malloc(sizeof(double) * rows * (size_t)j->D);
    double *z = (double *)malloc(sizeof(double) * rows);
    double *qd = (double *)malloc(sizeof(double) * (size_t)j->D);
    double *op = (double *)malloc(sizeof(double) * (size_t)j->D);

    for (int s = j->tid; s < j->B; s += j->nthreads) {
        int L = j->context_lens[s];
        double *out_s = j->out + (int64_t)s * j->H * j->D;
        memset(out_s, 0, sizeof(double) * (size_t)j->H * (size_t)j->D);
        j->seq_status[s] = 0;
        if (L < 0 || (int64_t)L > (int64_t)j->max_blocks_per_seq * j->bs) {
            j->seq_status[s] = ORC_BAD_LEN;
            continue;
        }
        if (L == 0)
            continue;                      /* nothing to attend: output stays 0 */
        const int32_t *table = j->block_tables + (int64_t)s * j->max_blocks_per_seq;
        for (int kvh = 0; kvh < j->Hk; ++kvh) {
            int st = gather_head(K, V, j->k_cache, j->v_cache, j->dtype, table, L, kvh,
                                 j->Hk, j->D, j->bs, j->num_blocks);
            if (st) {
                j->seq_status[s] |= (uint32_t)st;
                memset(out_s, 0, sizeof(double) * (size_t)j->H * (size_t)j->D);
                break;
            }
            for (int g = 0; g < G; ++g) {
                int h = kvh * G + g;
                for (int d = 0; d < j->D; ++d)
                    qd[d] = load_elem(j->q, j->dtype, ((int64_t)s * j->H + h) * j->D + d);
                if (j->partition_size > 0)
                    attend_partitioned(out_s + (int64_t)h * j->D, qd, K, V, L, j->D, j->scale,
                                       j->partition_size, z, op);
                else
                    attend(out_s + (int64_t)h * j->D, qd, K, V, L, j->D, j->scale, z);
            }
        }
    }
    free(K);
    free(V);
    free(z);
    free(qd);
    free(op);
    return NULL;
}

/* Single-query attention of every sequence over its paged K/V.
 * Returns the OR of the per-sequence status bits; a sequence with a bad
 * context length or block id gets an all-zero output row. */
uint32_t pkv_oracle_paged_attention(double *out, const void *q, const void *k_cache,
                                    const void *v_cache, int dtype,
                                    const int32_t *block_tables, int max_blocks_per_seq,
                                    const int32_t *context_lens, int num_seqs, int num_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int64_t num_blocks, double scale, int partition_size,
                                    int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    uint32_t *seq_status = (uint32_t *)calloc((size_t)(num_seqs > 0 ? num_seqs : 1), sizeof(uint32_t));
    attn_job *jobs = (attn_job *)malloc(sizeof(attn_job) * (size_t)nthreads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        attn_job j = {out, q, k_cache, v_cache, dtype, block_tables, max_blocks_per_seq,
                      context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, scale, partition_size, seq_status, t, nthreads};
        jobs[t] = j;
    }
    if (nthreads == 1) {
        attn_worker(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t)
            pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
        for (int t = 0; t < nthreads; ++t)
            pthread_join(th[t], NULL);
    }
    uint32_t st = 0;
    for (int s = 0; s < num_seqs; ++s)
        st |= seq_status[s];
    free(seq_status);
    free(jobs);
    free(th);
    return st;
}

/* Contiguous single-query attention: q [H, D], K and V [L, Hk, D] already in
 * token order, fp64 in and out.  Used by the tests to compare the paged
 * oracle against ordinary attention over the same logical tokens. */
void pkv_oracle_contiguous_attention(double *out, const double *q, const double *K,
                                     const double *V, int L, int H, int Hk, int D,
                                     double scale)
{
    int G = H / Hk;
    double *Kh = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)D);
    double *Vh = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)D);
    double *z = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    for (int h = 0; h < H; ++h) {
        int kvh = h / G;
        if (L == 0) {
            memset(out + (int64_t)h * D, 0, sizeof(double) * (size_t)D);
            continue;
        }
        for (int i = 0; i < L; ++i)
            for (int d = 0; d < D; ++d) {
                Kh[(int64_t)i * D + d] = K[((int64_t)i * Hk + kvh) * D + d];
                Vh[(int64_t)i * D + d] = V[((int64_t)i * Hk + kvh) * D + d];
            }
        attend(out + (int64_t)h * D, q + (int64_t)h * D, Kh, Vh, L, D, scale, z);
    }
    free(Kh);
    free(Vh);
    free(z);
}

/* ------------------------------------------------------ cache scatter */

/* Write each new token's K and V rows into its slot [P4-alg Step 2]:
 * slot = physical_block * bs + offset; k_cache[block, h, offset, :] = key[t, h, :].
 * A negative slot is padding and is skipped; a slot past the pool is skipped
 * and reported. */
uint32_t pkv_oracle_reshape_and_cache(const void *key, const void *value, void *k_cache,
                                      void *v_cache, int dtype, const int64_t *slot_mapping,
                                      int num_tokens, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks)
{
    uint32_t st = 0;
    size_t row = (size_t)head_dim * (size_t)elem_bytes(dtype);
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size) {
            st |= ORC_BAD_SLOT;
            continue;
        }
        int64_t b = slot / block_size, o = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (size_t)(((b * num_kv_heads + h) * block_size + o)) * row;
            size_t src = ((size_t)t * (size_t)num_kv_heads + (size_t)h) * row;
            memcpy((char *)k_cache + dst, (const char *)key + src, row);
            memcpy((char *)v_cache + dst, (const char *)value + src, row);
        }
    }
    return st;
}

/* ------------------------------------------------------- block copy */

/* Copy-on-write copies [P4-cow]: for each (src, dst) pair and each layer,
 * physical block dst of both caches becomes a copy of block src. */
uint32_t pkv_oracle_copy_blocks(void *const *k_caches, void *const *v_caches, int num_layers,
                                const int64_t *src_dst_pairs, int num_pairs, size_t block_bytes,
                                int64_t num_blocks)
{
    uint32_t st = 0;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t src = src_dst_pairs[2 * p], dst = src_dst_pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            st |= ORC_BAD_BLOCK;
            continue;
        }
        for (int l = 0; l < num_layers; ++l) {
            memcpy((char *)k_caches[l] + (size_t)dst * block_bytes,
                   (const char *)k_caches[l] + (size_t)src * block_bytes, block_bytes);
            memcpy((char *)v_caches[l] + (size_t)dst * block_bytes,
                   (const char *)v_caches[l] + (size_t)src * block_bytes, block_bytes);
        }
    }
    return st;
}

/* Swapping blocks out to host memory and back in (PagedAttention: Efficient
 * LLM Serving with vLLM, "vLLM: The Serving Engine": a preempted request's
 * KV cache goes to CPU memory when the GPU is full and comes back when it
 * resumes; the paper's section 7.3 compares this with recomputation). */
/* Pair p = (gpu block, host block); direction 0 copies every layer's K and V
 * gpu block -> host block, direction 1 host block -> gpu block.  A pair with
 * an id outside its pool is skipped and flags ORC_BAD_BLOCK. */
uint32_t pkv_oracle_swap_blocks(void *const *gpu_k, void *const *gpu_v, void *const *host_k,
                                void *const *host_v, int num_layers, const int64_t *pairs,
                                int num_pairs, size_t block_bytes, int64_t gpu_blocks,
                                int64_t host_blocks, int direction)
{
    uint32_t st = 0;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t g = pairs[2 * p], h = pairs[2 * p + 1];
        if (g < 0 || g >= gpu_blocks || h < 0 || h >= host_blocks) {
            st |= ORC_BAD_BLOCK;
            continue;
        }
        for (int l = 0; l < num_layers; ++l) {
            char *gk = (char *)gpu_k[l] + (size_t)g * block_bytes;
            char *gv = (char *)gpu_v[l] + (size_t)g * block_bytes;
            char *hk = (char *)host_k[l] + (size_t)h * block_bytes;
            char *hv = (char *)host_v[l] + (size_t)h * block_bytes;
            if (direction == 0) {
                memcpy(hk, gk, block_bytes);
                memcpy(hv, gv, block_bytes);
            } else {
                memcpy(gk, hk, block_bytes);
                memcpy(gv, hv, block_bytes);
            }
        }
    }
    return st;
}
