/*
 * oracle.c -- plain, slow, fp64 CPU reference for paged KV-cache attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this code. The GPU library never
 * links, includes or calls it, and it shares no code with the GPU library.
 *
 * Sources (the web pages this method is taken from):
 *   [page 1] "从 token 调度到采样输出，追踪每一步张量维度的变化，搞懂 LLM 推理到底在算什么"
 *            (zizhi168.cn/news/2384056): §02 Paged Attention, §03 Embedding
 *            (flattened [num_sched_tokens]), §04 Attention (six steps, GQA
 *            index map, cu_seqlens, prefill/decode table), §07 (log-sum-exp
 *            renormalisation of split attention).
 *   [page 2] "别只当API调用侠了！一文带你深入大模型“体内”，看懂推理全流程"
 *            (su666666.com/news/35626): PagedAttention deep-dive (physical
 *            block pool, block table, copy-on-write), step 4 (scaled
 *            dot-product attention with a causal mask), step 6 (KV cache).
 *   [page 3] adg.csdn.net survey of LLM inference optimisation
 *            (adg.csdn.net/695256bb5b9f5f31781b99f3): §1.5 KV-cache sizing,
 *            §3.3 GQA, §3.4 FlashAttention (exact attention), §3.5 PagedAttention.
 *
 * Everything is the plain definition written out: no tiling, no online
 * softmax, no reordering. Inputs are bf16 bit patterns (uint16); they are
 * widened exactly to double and all arithmetic is fp64.
 *
 * Layouts (all row-major, element strides implied):
 *   pool         [2][num_blocks][block_size][num_kv_heads][head_dim]  bf16
 *                index 0 = K, index 1 = V (one layer; [page 1] §02)
 *   q            [num_tokens][num_heads][head_dim]                    bf16
 *   k_new, v_new [num_tokens][num_kv_heads][head_dim]                 bf16
 *   slot_mapping [num_tokens]                                          int32
 *   block_table  [num_seqs][max_blocks]                                int32
 *   cu_seqlens   [num_seqs + 1]                                        int32
 *   seq_lens     [num_seqs]  (context length INCLUDING this step's tokens)
 *
 * Return codes: 0 = ok, otherwise a positive code naming the bad input
 * (the oracle refuses inputs the method does not define).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_SHAPE 1
#define ORACLE_BAD_SLOT 2
#define ORACLE_BAD_BLOCK 3
#define ORACLE_BAD_LENGTHS 4
#define ORACLE_NO_MEMORY 5

/* bf16 -> fp64, exact: a bf16 value is the top half of an IEEE fp32. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Flat element offset of pool[kv][block][offset][head][0]. */
static size_t pool_index(int kv, int64_t block, int64_t offset, int64_t head,
                         int64_t num_blocks, int64_t block_size,
                         int64_t num_kv_heads, int64_t head_dim)
{
    return ((((size_t)kv * num_blocks + block) * block_size + offset) * num_kv_heads + head)
           * head_dim;
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * KV write ([page 1] §02: slot_mapping tells the kernel where each newly
 * produced K/V goes; a slot is a physical block id times block_size plus the
 * offset inside the block).
 *
 * For every token t with slot s = slot_mapping[t] >= 0:
 *   pool[0][s / block_size][s % block_size][h][:] = k_new[t][h][:]
 *   pool[1][s / block_size][s % block_size][h][:] = v_new[t][h][:]
 * A slot of -1 means "no write" (padding). Everything else in the pool is
 * left untouched. The copy is of bits: bf16 in, bf16 out.
 */
int oracle_kv_cache_write(uint16_t *pool, const uint16_t *k_new, const uint16_t *v_new,
                          const int32_t *slot_mapping, int32_t num_tokens,
                          int32_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim)
{
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0)
        return ORACLE_BAD_SHAPE;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int32_t t = 0; t < num_tokens; ++t) {
        const int64_t s = slot_mapping[t];
        if (s == -1) continue;
        if (s < 0 || s >= num_slots) return ORACLE_BAD_SLOT;
        const int64_t block = s / block_size;
        const int64_t offset = s % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            const uint16_t *src_k = k_new + ((size_t)t * num_kv_heads + h) * head_dim;
            const uint16_t *src_v = v_new + ((size_t)t * num_kv_heads + h) * head_dim;
            uint16_t *dst_k = pool + pool_index(0, block, offset, h, num_blocks, block_size,
                                                num_kv_heads, head_dim);
            uint16_t *dst_v = pool + pool_index(1, block, offset, h, num_blocks, block_size,
                                                num_kv_heads, head_dim);
            for (int32_t d = 0; d < head_dim; ++d) {
                dst_k[d] = src_k[d];
                dst_v[d] = src_v[d];
            }
        }
    }
    return ORACLE_OK;
}

/* Which request owns flattened token t ([page 1] §04: cu_seqlens separates
 * requests inside the flattened token axis). Linear scan: obviously right. */
static int find_request(const int32_t *cu_seqlens, int32_t num_seqs, int32_t t)
{
    for (int32_t i = 0; i < num_seqs; ++i)
        if (cu_seqlens[i] <= t && t < cu_seqlens[i + 1]) return i;
    return -1;
}

/* Shared argument bundle for the attention routines below. */
typedef struct {
    const uint16_t *q;
    const uint16_t *pool;
    const int32_t *block_table;
    int32_t max_blocks;
    const int32_t *cu_seqlens;
    const int32_t *seq_lens;
    int32_t num_seqs, num_tokens, num_heads, num_kv_heads, head_dim, block_size, num_blocks;
    double scale;
} attn_args;

static int check_args(const attn_args *a)
{
    if (a->num_seqs < 0 || a->num_tokens < 0 || a->num_heads <= 0 || a->num_kv_heads <= 0 ||
        a->head_dim <= 0 || a->block_size <= 0 || a->num_blocks <= 0 || a->max_blocks < 0)
        return ORACLE_BAD_SHAPE;
    if (a->num_heads % a->num_kv_heads != 0) return ORACLE_BAD_SHAPE;
    if (a->cu_seqlens[0] != 0 || a->cu_seqlens[a->num_seqs] != a->num_tokens)
        return ORACLE_BAD_LENGTHS;
    for (int32_t i = 0; i < a->num_seqs; ++i) {
        const int32_t ql = a->cu_seqlens[i + 1] - a->cu_seqlens[i];
        if (ql < 0 || a->seq_lens[i] < ql) return ORACLE_BAD_LENGTHS;
        if (a->seq_lens[i] > (int64_t)a->max_blocks * a->block_size) return ORACLE_BAD_LENGTHS;
        const int32_t nblk = (a->seq_lens[i] + a->block_size - 1) / a->block_size;
        for (int32_t b = 0; b < nblk; ++b) {
            const int32_t id = a->block_table[(size_t)i * a->max_blocks + b];
            if (id < 0 || id >= a->num_blocks) return ORACLE_BAD_BLOCK;
        }
    }
    return ORACLE_OK;
}

/*
 * Attention of one query row (token t, head h) over the logical keys
 * [key_begin, key_end) intersected with the causal range [0, pos].
 *
 *   GQA ([page 1] §04): kv = h / (num_heads / num_kv_heads)
 *   position of query j of request i: pos = seq_len_i - query_len_i + j
 *     (the new tokens are the last query_len_i tokens of the context;
 *      causal mask of [page 2] step 4: a position sees itself and earlier
 *      positions only)
 *   logical key p lives at pool[.][block_table[i][p / bs]][p % bs][kv]
 *     ([page 1] §02 block_table read; [page 2] block table = logical ->
 *      physical map)
 *   scores s_p = scale * sum_d q[t][h][d] * k_p[d]   (scaled dot product)
 *   softmax, two passes: m = max_p s_p, P_p = exp(s_p - m) / sum exp(s - m)
 *   o = sum_p P_p v_p, lse = m + ln sum_p exp(s_p - m)
 *
 * An empty key range gives o = 0 and lse = -inf. When probs is not NULL it
 * receives P over the keys in range (for the sums-to-one check).
 * Returns the number of keys used.
 */
static int64_t attend_row(const attn_args *a, int32_t t, int32_t h, int64_t key_begin,
                          int64_t key_end, double *out, double *lse, double *scores,
                          double *probs)
{
    const int32_t i = find_request(a->cu_seqlens, a->num_seqs, t);
    const int32_t query_len = a->cu_seqlens[i + 1] - a->cu_seqlens[i];
    const int32_t j = t - a->cu_seqlens[i];
    const int64_t pos = (int64_t)a->seq_lens[i] - query_len + j;
    const int32_t group = a->num_heads / a->num_kv_heads;
    const int32_t kv = h / group;
    const int32_t D = a->head_dim;

    int64_t lo = key_begin < 0 ? 0 : key_begin;
    int64_t hi = pos + 1;
    if (key_end >= 0 && key_end < hi) hi = key_end;

    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    if (hi <= lo) {
        *lse = -INFINITY;
        return 0;
    }

    const uint16_t *qrow = a->q + ((size_t)t * a->num_heads + h) * D;
    const int32_t *table = a->block_table + (size_t)i * a->max_blocks;

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t p = lo; p < hi; ++p) {
        const int32_t block = table[p / a->block_size];
        const int64_t offset = p % a->block_size;
        const uint16_t *krow = a->pool + pool_index(0, block, offset, kv, a->num_blocks,
                                                    a->block_size, a->num_kv_heads, D);
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += bf16_value(qrow[d]) * bf16_value(krow[d]);
        const double s = a->scale * dot;
        scores[p - lo] = s;
        if (s > m) m = s;
    }
    /* pass 2: normaliser */
    double sum = 0.0;
    for (int64_t p = lo; p < hi; ++p) sum += exp(scores[p - lo] - m);
    /* pass 3: probabilities times V */
    for (int64_t p = lo; p < hi; ++p) {
        const double prob = exp(scores[p - lo] - m) / sum;
        if (probs) probs[p - lo] = prob;
        const int32_t block = table[p / a->block_size];
        const int64_t offset = p % a->block_size;
        const uint16_t *vrow = a->pool + pool_index(1, block, offset, kv, a->num_blocks,
                                                    a->block_size, a->num_kv_heads, D);
        for (int32_t d = 0; d < D; ++d) out[d] += prob * bf16_value(vrow[d]);
    }
    *lse = m + log(sum);
    return hi - lo;
}

/*
 * Paged attention for a list of flattened query tokens (every head of each).
 *   out [num_rows][num_heads][head_dim] fp64, lse [num_rows][num_heads] fp64.
 * key_begin/key_end restrict the logical key range (key_end < 0: no upper
 * limit); the full method uses key_begin = 0, key_end = -1. A restricted
 * range gives the partial result of one split-KV partition ([page 1] §07).
 * Rows are independent, so they are spread over OpenMP threads; this changes
 * no arithmetic.
 */
int oracle_paged_attention_rows(double *out, double *lse, const int32_t *rows, int32_t num_rows,
                                const uint16_t *q, const uint16_t *pool,
                                const int32_t *block_table, int32_t max_blocks,
                                const int32_t *cu_seqlens, const int32_t *seq_lens,
                                int32_t num_seqs, int32_t num_tokens, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                int32_t num_blocks, double scale, int64_t key_begin,
                                int64_t key_end)
{
    const attn_args a = {q, pool, block_table, max_blocks, cu_seqlens, seq_lens, num_seqs,
                         num_tokens, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         scale};
    const int rc = check_args(&a);
    if (rc != ORACLE_OK) return rc;
    for (int32_t r = 0; r < num_rows; ++r)
        if (rows[r] < 0 || rows[r] >= num_tokens) return ORACLE_BAD_SHAPE;

    int64_t max_len = 1;
    for (int32_t i = 0; i < num_seqs; ++i)
        if (seq_lens[i] > max_len) max_len = seq_lens[i];

    int failed = 0;
    const int64_t work = (int64_t)num_rows * num_heads;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_len);
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t w = 0; w < work; ++w) {
            if (!scores) continue;
            const int32_t r = (int32_t)(w / num_heads);
            const int32_t h = (int32_t)(w % num_heads);
            attend_row(&a, rows[r], h, key_begin, key_end,
                       out + ((size_t)r * num_heads + h) * head_dim,
                       lse + (size_t)r * num_heads + h, scores, NULL);
        }
        free(scores);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Full attention output for every flattened token: rows = 0 .. num_tokens-1. */
int oracle_paged_attention(double *out, double *lse, const uint16_t *q, const uint16_t *pool,
                           const int32_t *block_table, int32_t max_blocks,
                           const int32_t *cu_seqlens, const int32_t *seq_lens, int32_t num_seqs,
                           int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int32_t num_blocks,
                           double scale)
{
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_tokens > 0 ? num_tokens : 1));
    if (!rows) return ORACLE_NO_MEMORY;
    for (int32_t t = 0; t < num_tokens; ++t) rows[t] = t;
    const int rc = oracle_paged_attention_rows(out, lse, rows, num_tokens, q, pool, block_table,
                                               max_blocks, cu_seqlens, seq_lens, num_seqs,
                                               num_tokens, num_heads, num_kv_heads, head_dim,
                                               block_size, num_blocks, scale, 0, -1);
    free(rows);
    return rc;
}

/*
 * The softmax row P of one (token t, head h) over its causal key range
 * [0, pos]; probs must hold seq_len entries. Returns the number of keys
 * written, or a negative error code.
 */
int64_t oracle_attention_probs(double *probs, int32_t t, int32_t h, const uint16_t *q,
                               const uint16_t *pool, const int32_t *block_table,
                               int32_t max_blocks, const int32_t *cu_seqlens,
                               const int32_t *seq_lens, int32_t num_seqs, int32_t num_tokens,
                               int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t num_blocks, double scale)
{
    const attn_args a = {q, pool, block_table, max_blocks, cu_seqlens, seq_lens, num_seqs,
                         num_tokens, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         scale};
    const int rc = check_args(&a);
    if (rc != ORACLE_OK) return -rc;
    if (t < 0 || t >= num_tokens || h < 0 || h >= num_heads) return -ORACLE_BAD_SHAPE;
    const int32_t i = find_request(cu_seqlens, num_seqs, t);
    double *scores = (double *)malloc(sizeof(double) * (size_t)(seq_lens[i] > 0 ? seq_lens[i] : 1));
    double *out = (double *)malloc(sizeof(double) * (size_t)head_dim);
    if (!scores || !out) {
        free(scores);
        free(out);
        return -ORACLE_NO_MEMORY;
    }
    double lse;
    const int64_t n = attend_row(&a, t, h, 0, -1, out, &lse, scores, probs);
    free(scores);
    free(out);
    return n;
}

/*
 * Log-sum-exp merge of split-KV partial results ([page 1] §07: chunked
 * prefill, Flash-Decoding and sequence parallelism all renormalise the
 * pieces with log-sum-exp).
 *   part_out [num_parts][num_rows][head_dim], part_lse [num_parts][num_rows]
 *   M = max_p lse_p, w_p = exp(lse_p - M)
 *   out = sum_p w_p o_p / sum_p w_p,  lse = M + ln sum_p w_p
 * A partition with lse = -inf holds no keys and contributes nothing (its o_p
 * is not read). A row whose partitions are all empty gives out = 0 and
 * lse = -inf.
 */
void oracle_lse_merge(double *out, double *out_lse, const double *part_out,
                      const double *part_lse, int32_t num_parts, int64_t num_rows,
                      int32_t head_dim)
{
    for (int64_t r = 0; r < num_rows; ++r) {
        double M = -INFINITY;
        for (int32_t p = 0; p < num_parts; ++p) {
            const double l = part_lse[(size_t)p * num_rows + r];
            if (l > M) M = l;
        }
        double *o = out + (size_t)r * head_dim;
        for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (M == -INFINITY) {
            out_lse[r] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int32_t p = 0; p < num_parts; ++p) {
            const double l = part_lse[(size_t)p * num_rows + r];
            if (l == -INFINITY) continue;
            const double w = exp(l - M);
            wsum += w;
            const double *op = part_out + ((size_t)p * num_rows + r) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) o[d] += w * op[d];
        }
        for (int32_t d = 0; d < head_dim; ++d) o[d] /= wsum;
        out_lse[r] = M + log(wsum);
    }
}

/*
 * KV-cache sizing ([page 3] §1.5): bytes per token = 2 (K and V) * layers *
 * heads * head_dim * bytes per element, where under GQA the heads that are
 * cached are the KV heads ([page 1] §04: GQA shrinks the cache by the group
 * factor). The batch total multiplies by batch size and sequence length.
 */
int64_t oracle_kv_bytes_per_token(int64_t num_layers, int64_t num_kv_heads, int64_t head_dim,
                                  int64_t bytes_per_element)
{
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_element;
}

int64_t oracle_kv_cache_bytes(int64_t batch, int64_t seq_len, int64_t num_layers,
                              int64_t num_kv_heads, int64_t head_dim, int64_t bytes_per_element)
{
    return batch * seq_len *
           oracle_kv_bytes_per_token(num_layers, num_kv_heads, head_dim, bytes_per_element);
}
