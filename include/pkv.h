/*
 * pkv.h -- C ABI of libpkv: paged KV-cache write and variable-length paged
 * attention for NVIDIA GB300 (sm_103a).
 *
 * Sources (the web pages the method comes from):
 *   [page 1] "从 token 调度到采样输出，追踪每一步张量维度的变化，搞懂 LLM 推理到底在算什么"
 *            (zizhi168.cn/news/2384056)
 *   [page 2] "别只当API调用侠了！一文带你深入大模型“体内”，看懂推理全流程"
 *            (su666666.com/news/35626)
 *   [page 3] adg.csdn.net survey of LLM inference optimisation
 *            (adg.csdn.net/695256bb5b9f5f31781b99f3)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller. The library
 *   never allocates device memory, never frees it, never synchronises the
 *   stream and keeps no state between calls, with stated exceptions: the
 *   built-in scratch array of pkv_paged_attention_varlen_noalloc and the
 *   host-side block manager objects (pkv_bm_*), which the caller creates and
 *   destroys.
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *   void*; NULL is the legacy default stream). A call returns as soon as the
 *   kernels are queued.
 * - bf16 tensors are raw 16-bit bfloat16 values. Layouts are row-major and
 *   dense (no strides), with the shapes given beside each argument.
 * - Host-detectable errors (null pointers, unsupported sizes, bad options)
 *   return a non-zero pkv_status and enqueue nothing.
 * - Device-detectable errors (an index that the tables give but that lies
 *   outside the pool, inconsistent lengths) never trap: the offending item is
 *   skipped, its outputs are unspecified, and the matching PKV_DEV_* bit is
 *   OR-ed into *dev_status when dev_status is not NULL. The caller zeroes
 *   *dev_status before the call and reads it after synchronising.
 * - KV pool of one layer ([page 1] §02 gives the per-model pool
 *   [num_layers, 2, num_blocks, block_size, num_kv_heads, head_dim]; a
 *   multi-layer caller passes the base of one layer):
 *       kv_pool [2][num_blocks][block_size][num_kv_heads][head_dim] bf16,
 *       index 0 holds K, index 1 holds V; the pointer must be 16-byte aligned.
 *   Supported: head_dim 64 or 128; block_size a multiple of 16 (up to 256);
 *   num_heads a multiple of num_kv_heads; at most 65534 requests per call.
 *   A call with prefill work (max_query_len above 32 / G, G = num_heads /
 *   num_kv_heads), and a cascade call's prefix pass over its prefix groups,
 *   takes at most 8575 requests (groups) at head_dim 128 and 33151 at 64:
 *   the prefill kernel holds their work list in shared memory. Beyond that
 *   the call returns PKV_ERR_UNSUPPORTED and enqueues nothing.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pkv_status;

#define PKV_OK 0
#define PKV_ERR_INVALID_ARG 1       /* null pointer, negative size, inconsistent shape */
#define PKV_ERR_UNSUPPORTED 2       /* valid, but outside what the kernels implement */
#define PKV_ERR_CUDA 3              /* a CUDA runtime call failed (e.g. launch) */
#define PKV_ERR_WORKSPACE 4         /* workspace missing or smaller than required */
#define PKV_ERR_NO_BLOCKS 5         /* the block pool cannot satisfy the request */

/* Bits OR-ed into *dev_status by the kernels. */
#define PKV_DEV_BAD_SLOT 1          /* slot_mapping entry outside [-1, num_blocks*block_size) */
#define PKV_DEV_BAD_BLOCK 2         /* block_table entry outside [0, num_blocks) */
#define PKV_DEV_BAD_LENGTHS 4       /* seq_len < query_len, cu_seqlens not monotone, or a
                                       length beyond max_seq_len / max_query_len /
                                       max_blocks_per_seq * block_size */
#define PKV_DEV_TIMEOUT 8           /* an internal pipeline wait gave up; outputs of the
                                       affected tile are unspecified */
#define PKV_DEV_V_RANGE 16          /* the chunked-prefill kernel met a V value of magnitude
                                       >= 65536 (or inf / NaN), beyond the fp16 range its
                                       P.V product uses; that request's outputs are
                                       unspecified */

/*
 * pkv_kv_cache_write -- scatter the step's new K/V rows into the paged pool.
 * ([page 1] §02: slot_mapping says where each new K/V is written; a slot is
 * physical_block * block_size + offset_in_block.)
 *
 *   kv_pool      [2][num_blocks][block_size][num_kv_heads][head_dim] bf16, in/out
 *   k_new, v_new [num_tokens][num_kv_heads][head_dim] bf16 (16-byte aligned)
 *   slot_mapping [num_tokens] int32; -1 skips the token (padding)
 *
 * For each token t with s = slot_mapping[t] >= 0:
 *   kv_pool[0][s / block_size][s % block_size][:][:] = k_new[t]
 *   kv_pool[1][s / block_size][s % block_size][:][:] = v_new[t]
 * A bit copy; every other slot is left untouched. Slots must be distinct
 * (duplicates race). num_tokens == 0 is a no-op.
 * Errors: PKV_DEV_BAD_SLOT for a slot outside [-1, num_blocks*block_size).
 */
pkv_status pkv_kv_cache_write(void *kv_pool, const void *k_new, const void *v_new,
                              const int32_t *slot_mapping, int32_t num_tokens,
                              int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                              int32_t head_dim, int32_t *dev_status, void *stream);

/*
 * pkv_attention_workspace_size -- bytes of scratch that
 * pkv_paged_attention_varlen needs for these sizes and this partition_size
 * (at least 256: the prefill kernel's work tickets; split-KV partials on top:
 * [num_seqs][P][H][D] + [num_seqs][P][H] fp32 for P partitions; when
 * num_tokens > num_seqs and num_seqs <= 256, [num_seqs] int32 more: the order
 * in which a batch of several-query (verification) requests runs, longest
 * context first; 0 only for invalid sizes and for more than 65535
 * partitions a request, which pkv_paged_attention_varlen refuses as
 * PKV_ERR_UNSUPPORTED). The caller allocates it (a 256-byte aligned
 * device buffer at least this large) and ZERO-FILLS it once before its first
 * use (it holds the counter from which prefill CTAs take their work items;
 * the split-KV partials need no clearing). Every call that
 * completes without PKV_DEV_TIMEOUT leaves it zero-filled again, so one
 * workspace serves any number of calls on one stream; calls that may run
 * concurrently need separate workspaces. After a PKV_DEV_TIMEOUT, clear it
 * again before reuse.
 */
size_t pkv_attention_workspace_size(int32_t num_seqs, int32_t num_tokens, int32_t num_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    int32_t max_seq_len, int32_t partition_size);

/*
 * pkv_paged_attention_varlen -- causal GQA attention of flattened queries
 * over a paged KV cache.
 * ([page 1] §03/§04: all requests' tokens are flattened into
 * [num_sched_tokens] and separated by cu_seqlens; the six steps GQA-share,
 * QK^T, scale, mask, softmax, times V; kv_head = q_head / (num_heads /
 * num_kv_heads); block_table maps a request's logical blocks to physical
 * ones ([page 2] PagedAttention deep-dive). [page 2] step 4: causal mask.
 * [page 1] §07: long contexts are split and the pieces renormalised by
 * log-sum-exp. [page 3] §3.4: the fused kernel is exact attention.)
 *
 *   out          [num_tokens][num_heads][head_dim] fp32, written
 *   out_lse      [num_tokens][num_heads] fp32 natural-log log-sum-exp of the
 *                scaled scores, written; may be NULL
 *   q            [num_tokens][num_heads][head_dim] bf16 (16-byte aligned)
 *   kv_pool      see above; the step's new K/V must already be written
 *                (call pkv_kv_cache_write first, on the same stream)
 *   block_table  [num_seqs][max_blocks_per_seq] int32 physical block ids
 *   cu_seqlens_q [num_seqs + 1] int32, cu[0] = 0, cu[num_seqs] = num_tokens
 *   seq_lens     [num_seqs] int32 context length of each request INCLUDING
 *                its query_len = cu[i+1] - cu[i] new tokens
 *   max_query_len, max_seq_len: upper bounds of the per-request values (the
 *                host never reads device tables; the grid is sized by them)
 *   scale        score scale, normally 1/sqrt(head_dim)
 *   partition_size  split-KV partition length in tokens for query_len == 1
 *                requests: 0 = never split; -1 = automatic (1024 tokens,
 *                doubled until no request has more than 32 partitions);
 *                > 0 = that many tokens, a multiple of 16. A split request's
 *                partitions are merged by log-sum-exp in a small second grid
 *                behind the first
 *   workspace, workspace_bytes: scratch of at least
 *                pkv_attention_workspace_size(...) bytes, zero-filled before
 *                its first use (see there)
 *
 * Query j of request i sits at position pos = seq_len_i - query_len_i + j
 * and attends to keys 0..pos (bottom-right causal alignment). Keys beyond
 * seq_len_i are never read, so unwritten slots of a partial last block may
 * hold anything, NaN included.
 * Requests of 1 .. max(1, 32 / G) queries (decode, and speculative
 * verification steps; G = num_heads / num_kv_heads) run on the decode kernel
 * (HBM-bound, warp-level tensor-core products; query_len == 1 requests split
 * into partitions merged by log-sum-exp, several-query requests one
 * partition); longer requests run on the chunked-prefill kernel (tcgen05
 * tensor cores).
 * The kernels use programmatic dependent launch: each waits for the grid
 * before it in the stream to finish before touching memory, so ordinary
 * stream order holds. A batch with requests for both kernels runs them side
 * by side, all on `stream`: the prefill grid first, keeping about its share
 * of the SMs (prefill tiles against decode bytes, estimated on the device)
 * and leaving the rest, then the decode grid, which launches once every
 * prefill CTA has started and completes only after the prefill grid has.
 * When num_tokens and max_query_len show that no request can be short
 * enough for the decode kernel (num_seqs * max_query_len - num_tokens <
 * max_query_len - max(1, 32 / G)), no decode grid is launched, and a
 * request that is short anyway (cu_seqlens_q at odds with num_tokens) is
 * flagged PKV_DEV_BAD_LENGTHS.
 */
pkv_status pkv_paged_attention_varlen(float *out, float *out_lse, const void *q,
                                      const void *kv_pool, const int32_t *block_table,
                                      int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q,
                                      const int32_t *seq_lens, int32_t num_seqs,
                                      int32_t num_tokens, int32_t max_query_len,
                                      int32_t max_seq_len, int32_t num_heads,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks, float scale,
                                      int32_t partition_size, void *workspace,
                                      size_t workspace_bytes, int32_t *dev_status,
                                      void *stream);

/*
 * pkv_paged_attention_varlen_append -- one step's KV write and attention in
 * one call: pkv_kv_cache_write(kv_pool, k_new, v_new, slot_mapping, ...)
 * followed by pkv_paged_attention_varlen(...) over the same pool ([page 1]
 * §02: a step appends its tokens' K/V to the cache through slot_mapping, then
 * attends over it). Arguments: those of the two calls (k_new, v_new
 * [num_tokens][num_kv_heads][head_dim] bf16, 16-byte aligned; slot_mapping
 * [num_tokens] int32, -1 skips a token).
 *
 * The results are those of the two calls made one after the other. The
 * difference is the overlap: the library knows what the write touches, so
 * the decode grid of a batch of one-query (or at most 32/G-query) requests
 * reads its inputs and the keys before each request's first query position
 * while the write is still running, and waits for the write only before the
 * keys from that position on. It therefore REQUIRES that slot_mapping[t] be
 * the pool slot that block_table gives to token t's position
 * (seq_len - query_len + j for the request's query j): the slots the step
 * appends. A slot outside the pool sets PKV_DEV_BAD_SLOT as in
 * pkv_kv_cache_write; a slot elsewhere in the pool gives unspecified results
 * (the debug mode, PKV_DEBUG_CHECKS=1 in the Python binding, checks the
 * mapping). Batches with prefill chunks, and batches of several-query
 * requests that run longest context first, wait for the write as the
 * separate calls do.
 *
 * Errors: as the two calls; every check of both runs before anything is
 * enqueued.
 */
pkv_status pkv_paged_attention_varlen_append(
    float *out, float *out_lse, const void *q, void *kv_pool, const void *k_new,
    const void *v_new, const int32_t *slot_mapping, const int32_t *block_table,
    int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
    int32_t num_seqs, int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float scale, int32_t partition_size, void *workspace,
    size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * pkv_paged_attention_varlen_range -- the same attention over a range of
 * each request's keys, for work split along the sequence: sequence
 * parallelism, where each GPU holds part of a long context, or any caller
 * that attends to a context in pieces. ([page 1] §07: long-context chunked
 * prefill, Flash-Decoding and sequence parallelism all split the sequence
 * dimension and combine the pieces exactly by log-sum-exp renormalisation;
 * pkv_lse_merge does that combination.)
 *
 * Arguments as pkv_paged_attention_varlen, plus two device arrays:
 *   key_start_pos   [num_seqs] int32 >= 0: absolute position of the first
 *                   key of request i's block table; its seq_lens[i] >= 1
 *                   keys sit at key_start_pos[i] + p, p < seq_lens[i]
 *   query_start_pos [num_seqs] int32 >= 0: absolute position of request i's
 *                   first query; query j sits at query_start_pos[i] + j
 * Query j of request i sees key p iff
 *   key_start_pos[i] + p <= query_start_pos[i] + j     (causal, absolute)
 * and the result is attention over exactly those keys: the normalised
 * output and the natural-log lse of that key range. A query that sees no key
 * of the range gets out = 0 and lse = -inf (an empty piece, which
 * pkv_lse_merge ignores). The ordinary call is key_start_pos = 0 and
 * query_start_pos = seq_len - query_len. seq_lens may be smaller than the
 * query count here; max_seq_len only bounds seq_lens (>= 1).
 * Merging the pieces of a context cut into ranges [s_r, e_r) with
 * pkv_lse_merge gives the attention over the whole context (to rounding).
 * Errors: as pkv_paged_attention_varlen; a NULL position array with
 * num_tokens > 0 is PKV_ERR_INVALID_ARG; a negative position or a zero
 * seq_len sets PKV_DEV_BAD_LENGTHS (that request is skipped).
 */
pkv_status pkv_paged_attention_varlen_range(
    float *out, float *out_lse, const void *q, const void *kv_pool, const int32_t *block_table,
    int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
    const int32_t *key_start_pos, const int32_t *query_start_pos, int32_t num_seqs,
    int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
    int32_t partition_size, void *workspace, size_t workspace_bytes, int32_t *dev_status,
    void *stream);

/*
 * pkv_lse_merge -- combine partial attention results by log-sum-exp
 * ([page 1] §07: chunked prefill, Flash-Decoding and sequence parallelism
 * renormalise their pieces with log-sum-exp).
 *
 *   part_out [num_parts][num_tokens][num_heads][head_dim] fp32
 *   part_lse [num_parts][num_tokens][num_heads] fp32
 *   out      [num_tokens][num_heads][head_dim] fp32, written
 *   out_lse  [num_tokens][num_heads] fp32, written; may be NULL
 *
 * Per row: M = max_p lse_p, w_p = exp(lse_p - M),
 *   out = sum_p w_p * part_out_p / sum_p w_p,  lse = M + ln(sum_p w_p).
 * A partition with lse = -inf is empty: its part_out values never enter the
 * sums (they may hold anything, NaN included); a row whose partitions are
 * all empty gives out = 0 and lse = -inf.
 * head_dim must be a multiple of 4 (at most 512); pointers 16-byte aligned.
 */
pkv_status pkv_lse_merge(float *out, float *out_lse, const float *part_out,
                         const float *part_lse, int32_t num_parts, int32_t num_tokens,
                         int32_t num_heads, int32_t head_dim, void *stream);

/*
 * pkv_paged_attention_varlen_noalloc -- pkv_paged_attention_varlen for
 * callers that cannot allocate device memory.
 * (The pages have no counterpart: this is a packaging variant of the call
 * above, not a step of the method.)
 *
 * Some callers cannot provide scratch memory: an engine whose memory manager
 * already owns the whole GPU, a server that must not call cudaMalloc while
 * it is serving, or a plugin that receives only its inputs and outputs. This
 * call takes the same arguments as pkv_paged_attention_varlen without
 * workspace / workspace_bytes and runs the same kernels; its split-KV
 * scratch is a 16 MiB array built into the library, which every GPU that
 * loads the library keeps until the process exits.
 * - It allocates nothing (no cudaMalloc or cudaFree, no allocating library).
 * - When the sizes would need more than 16 MiB of scratch (the value
 *   pkv_attention_workspace_size returns), it returns PKV_ERR_WORKSPACE and
 *   enqueues nothing; a larger partition_size lowers the need.
 * - The first call on each device looks up the array's device address with
 *   that device current; make that first call before any stream capture on
 *   the device.
 * - Every call on a device shares the one array, which keeps the last call's
 *   contents: calls that may overlap on the GPU (other streams, other host
 *   threads) race on it. The work-ticket counter inside it is cleared by
 *   every call.
 */
pkv_status pkv_paged_attention_varlen_noalloc(
    float *out, float *out_lse, const void *q, const void *kv_pool, const int32_t *block_table,
    int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
    int32_t num_seqs, int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float scale, int32_t partition_size, int32_t *dev_status, void *stream);

/*
 * pkv_cascade_decode -- decode attention for requests that share a
 * copy-on-write prefix, reading each shared prefix once per group instead of
 * once per request. ([page 2] PagedAttention deep-dive: forked sequences
 * point at the same physical prompt blocks; [page 1] §07: attention over
 * parts of the keys is combined exactly by log-sum-exp renormalisation.)
 *
 *   out      [num_seqs][num_heads][head_dim] fp32, out_lse [num_seqs][num_heads]
 *            fp32 (nullable): exactly what pkv_paged_attention_varlen returns
 *            for one decode query per request over its whole context
 *   q        [num_seqs][num_heads][head_dim] bf16 (one query per request)
 *   Prefix groups (device arrays): the requests of group g are
 *            group_starts[g] .. group_starts[g+1]-1 ([num_prefix_groups + 1],
 *            non-decreasing, within [0, num_seqs]; requests outside every
 *            group have no prefix); prefix_lens [num_prefix_groups] tokens
 *            (>= 0, a multiple of block_size); prefix_tables
 *            [num_prefix_groups][max_prefix_blocks] the physical blocks of
 *            each prefix. max_group_size >= the largest group, max_prefix_len
 *            >= the largest prefix.
 *   Tails (device arrays): tail_tables [num_seqs][max_tail_blocks] the blocks
 *            of each request after its prefix, tail_lens [num_seqs] >= 1 (the
 *            tail holds at least the new token), max_tail_len >= their max.
 *   workspace: pkv_cascade_workspace_size(...) bytes, 256-byte aligned,
 *            zero-filled before first use; left reusable (as for
 *            pkv_paged_attention_varlen); one workspace per concurrent call.
 * A request's context is its group's prefix followed by its tail. The prefix
 * pass runs every group's queries (members x heads as the rows of tensor-core
 * tiles) against the prefix blocks once, split into key segments, on about a
 * fifth of the SMs; the tails run through the decode kernel at the same
 * time on the others (launched right behind the prefix pass on `stream`);
 * the partial results merge by log-sum-exp.
 * Errors: as pkv_paged_attention_varlen; PKV_DEV_BAD_LENGTHS for inconsistent
 * group_starts or lengths.
 */
size_t pkv_cascade_workspace_size(int32_t num_seqs, int32_t num_prefix_groups,
                                  int32_t max_group_size, int32_t max_prefix_len,
                                  int32_t max_tail_len, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim);
pkv_status pkv_cascade_decode(float *out, float *out_lse, const void *q, const void *kv_pool,
                              int32_t num_prefix_groups, const int32_t *group_starts,
                              const int32_t *prefix_lens, const int32_t *prefix_tables,
                              int32_t max_prefix_blocks, int32_t max_group_size,
                              int32_t max_prefix_len, const int32_t *tail_tables,
                              int32_t max_tail_blocks, const int32_t *tail_lens,
                              int32_t max_tail_len, int32_t num_seqs, int32_t num_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int32_t num_blocks, float scale, void *workspace,
                              size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * ---------------------------------------------------------------------------
 * Host block manager and block copies -- the allocator side of the paged
 * cache ([page 2] PagedAttention deep-dive: the physical block pool carved up
 * at start-up; a block table per sequence mapping logical to physical blocks;
 * a free block appended to a sequence's table when its last block is full;
 * forking copies only the table, so the blocks are shared; a shared block
 * gets its own copy when a sequence writes into it; the tables live on the
 * CPU and are copied to the GPU for every step).
 *
 * Readings where the page is silent: the free pool is first-in first-out
 * (the order given to pkv_bm_create, ascending ids by default; a block whose
 * last reference goes away joins the back); a shared block is copied only
 * when the writer's next token falls inside it (it is partially filled) -- a
 * full shared block is never written again, so the next token goes to a
 * fresh block without a copy; a copy covers the whole block, K and V.
 *
 * The manager is plain host memory and host code (no CUDA call); it is not
 * thread-safe. Sequence ids are caller-chosen int64 values.
 * ---------------------------------------------------------------------------
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager of num_blocks blocks of block_size token slots. free_order
 * (host, [num_blocks], nullable) is the initial order of the free pool and
 * must be a permutation of 0..num_blocks-1. *out receives the handle.
 * Errors: PKV_ERR_INVALID_ARG (bad sizes, not a permutation). */
pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *free_order,
                         pkv_block_manager **out);
void pkv_bm_destroy(pkv_block_manager *bm);

/* A new, empty sequence. PKV_ERR_INVALID_ARG if the id exists. */
pkv_status pkv_bm_add_seq(pkv_block_manager *bm, int64_t seq_id);

/* child becomes a copy of parent's block table and length; every block it
 * names gains a reference. PKV_ERR_INVALID_ARG for an unknown parent or an
 * existing child. */
pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child);

/* Drop the sequence; blocks left without references return to the pool. */
pkv_status pkv_bm_free_seq(pkv_block_manager *bm, int64_t seq_id);

/* Room for num_tokens more tokens of one sequence (host arrays):
 *   slots      [num_tokens] int32, out: the slot of each new token, in order
 *   copy_src, copy_dst [max_copies] int32, out: block copies to run (with
 *              pkv_copy_blocks) before the tokens are written; an append makes
 *              at most one; *num_copies receives the count
 * All or nothing: PKV_ERR_NO_BLOCKS (the pool is short; nothing changes),
 * PKV_ERR_INVALID_ARG (unknown sequence, missing output). */
pkv_status pkv_bm_append(pkv_block_manager *bm, int64_t seq_id, int32_t num_tokens,
                         int32_t *slots, int32_t *copy_src, int32_t *copy_dst, int32_t max_copies,
                         int32_t *num_copies);

/* One step for a batch (host arrays; the outputs are exactly the inputs of
 * pkv_copy_blocks, pkv_kv_cache_write and pkv_paged_attention_varlen once
 * copied to the device):
 *   seq_ids     [num_seqs] int64, distinct existing sequences, in batch order
 *   num_new     [num_seqs] int32, tokens each sequence adds this step (>= 0)
 *   block_table [num_seqs][max_blocks] int32, out: tables, padded with -1
 *   seq_lens    [num_seqs] int32, out: lengths including the new tokens
 *   cu_seqlens  [num_seqs + 1] int32, out: prefix sums of num_new
 *   slot_mapping [sum num_new] int32, out: slots of the new tokens
 *   copy_src, copy_dst [max_copies] int32, out; *num_copies the count
 * Appends happen in batch order (a copy taken by one sequence can leave a
 * later sibling the sole owner of the shared block). All or nothing:
 * PKV_ERR_NO_BLOCKS if the pool cannot hold the whole batch,
 * PKV_ERR_INVALID_ARG for an unknown or repeated sequence, a table row too
 * short for a sequence, or more copies than max_copies. */
pkv_status pkv_bm_build_step(pkv_block_manager *bm, const int64_t *seq_ids, const int32_t *num_new,
                             int32_t num_seqs, int32_t max_blocks, int32_t *block_table,
                             int32_t *seq_lens, int32_t *cu_seqlens, int32_t *slot_mapping,
                             int32_t *copy_src, int32_t *copy_dst, int32_t max_copies,
                             int32_t *num_copies);

/* Views: free blocks; a sequence's length (-1 if unknown); a block's
 * reference count (-1 if out of range); a sequence's block table into
 * table[capacity] (*num_blocks receives its length; PKV_ERR_WORKSPACE if
 * capacity is too small). */
int32_t pkv_bm_num_free(const pkv_block_manager *bm);
int64_t pkv_bm_seq_len(const pkv_block_manager *bm, int64_t seq_id);
int32_t pkv_bm_refcount(const pkv_block_manager *bm, int32_t block);
pkv_status pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *table,
                              int32_t capacity, int32_t *num_blocks);

/*
 * pkv_copy_blocks -- copy whole blocks inside the pool (the device half of
 * copy-on-write):
 *   kv_pool            [2][num_blocks][block_size][num_kv_heads][head_dim] bf16
 *   copy_src, copy_dst [num_copies] int32 (device)
 * For each c: kv_pool[h][copy_dst[c]] = kv_pool[h][copy_src[c]] for h = K, V.
 * Copies of one call must be independent (no block both a source and a
 * destination); pkv_bm_build_step's copies are. num_copies == 0 is a no-op.
 * Errors: PKV_DEV_BAD_BLOCK for an id outside [0, num_blocks) (that copy is
 * skipped).
 */
pkv_status pkv_copy_blocks(void *kv_pool, const int32_t *copy_src, const int32_t *copy_dst,
                           int32_t num_copies, int32_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, int32_t head_dim, int32_t *dev_status,
                           void *stream);

/* Human-readable name of a pkv_status value (static storage). */
const char *pkv_status_string(pkv_status status);

/* ABI version of this header: 1. */
int32_t pkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
