// launch.h -- internal launch interface between the C-ABI layer (api.cpp)
// and the kernels. Not part of the public ABI.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; no driver-API linkage)
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace pkv {

// A kernel's dynamic shared-memory limit is a per-device attribute: raise it
// once on every device the process launches the kernel on (thread-safe; a
// process may drive several GPUs from several host threads).
class SmemLimit {
 public:
  cudaError_t ensure(const void* func, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return e;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

struct KvWriteParams {
  void* pool;                 // [2][NB][BS][Hkv][D] bf16
  const void* k_new;          // [T][Hkv][D] bf16
  const void* v_new;          // [T][Hkv][D] bf16
  const int32_t* slot_mapping;  // [T]
  int32_t num_tokens;
  int64_t num_slots;          // NB * BS
  int32_t row_vecs;           // 16-byte vectors per token row = Hkv * D / 8
  int32_t* status;
};

// Attention problem shared by the decode, merge and prefill kernels.
// Key segments of a shared prefix of L tokens in the cascade's prefix pass:
// its 128-key tiles cut into segments of prefix_tiles_per_segment tiles, of
// which prefix_segment_count are non-empty (at most `splits`).
__host__ __device__ inline int prefix_tiles_per_segment(int L, int splits) {
  const int t = (L + 127) / 128;
  return (t + splits - 1) / splits;
}
__host__ __device__ inline int prefix_segment_count(int L, int splits) {
  const int t = (L + 127) / 128;
  const int tps = prefix_tiles_per_segment(L, splits);
  return tps > 0 ? (t + tps - 1) / tps : 0;
}

struct AttnParams {
  float* out;                 // [T][H][D] fp32
  float* out_lse;             // [T][H] fp32 or null
  const uint16_t* q;          // [T][H][D] bf16
  const void* kv_pool;        // [2][NB][BS][Hkv][D] bf16
  const int32_t* block_table; // [B][max_blocks]
  const int32_t* cu_seqlens;  // [B+1]; null: one query per request (request i is query i)
  const int32_t* seq_lens;    // [B]
  int32_t max_blocks;
  int32_t num_seqs, num_tokens, max_query_len, max_seq_len;
  int32_t num_heads, num_kv_heads, head_dim, block_size, num_blocks;
  float scale_log2;           // scale * log2(e)
  // split-KV for query_len == 1 requests (merged by the decode merge grid)
  int32_t part_size;          // tokens per partition (multiple of 16)
  int32_t num_parts;          // partitions per request covering max_seq_len
  float* ws_out;              // [B][num_parts][H][D] (null when num_parts == 1)
  float* ws_lse;              // [B][num_parts][H]
  int32_t* sched;             // prefill work tickets: [0] next item, [1] CTAs done;
                              // zero between calls
  int32_t* status;
  // key-range mode (both null otherwise): the keys of request i in its block
  // table sit at absolute positions key_start[i] + p, its queries at
  // query_start[i] + j; query j sees key p iff key_start + p <= query_start + j
  const int32_t* key_start;
  const int32_t* query_start;
  // requests of 1 .. decode_max_q queries run on the decode kernel (its MMA
  // rows are (query, head) pairs, at most decode_max_rows per request in the
  // launch); longer ones on the prefill kernel
  int32_t decode_max_q, decode_max_rows;
  // shared-prefix (cascade) pass of the prefill kernel (prefix_mode 1):
  // every query of a "request" (a prefix group) sees all seq_len keys, no
  // causal mask; the keys are cut into at most kv_splits segments, segment s
  // writing its normalised partial to out + s * split_out_stride and its lse
  // to out_lse + s * split_lse_stride
  int32_t prefix_mode;        // 0: ordinary causal prefill
  int32_t kv_splits;
  int64_t split_out_stride, split_lse_stride;
  // A call with both kinds of request launches the prefill grid, then the
  // decode grid right behind it on the same stream (programmatic dependent
  // launch), the two sharing the SMs:
  //   prefill grid, shared_sms > 0: it keeps about as many of the SMs as
  //     its share of the estimated work (prefill tiles against decode
  //     bytes, out of shared_sms), its other CTAs leave at once, so that
  //     the decode grid -- launched when every prefill CTA has started or
  //     left -- has the rest;
  //   decode grid, after_prefill: its CTAs do not wait for the prefill grid;
  //     one extra CTA (z = num_seqs) waits for it and exits, so that the
  //     decode grid completes only after the prefill grid has.
  //   no_decode: the host has shown that no request is short enough for the
  //     decode kernel (no decode grid is launched); the prefill kernel flags
  //     one that is as PKV_DEV_BAD_LENGTHS.
  int32_t shared_sms;
  int32_t after_prefill;
  int32_t no_decode;
  // decode grid only: request of grid slice z is order[z] (null: z), written
  // by a one-CTA kernel launched before the decode grid (longest context
  // first)
  int32_t* order;
  // decode grid only: the kernel enqueued right before it is this call's own
  // KV write (pkv_paged_attention_varlen_append), which writes only the slots
  // of the requests' query positions: CTAs of a plain decode batch read the
  // keys before the first query's position without waiting for it
  int32_t early_pool;
};

cudaError_t launch_kv_write(const KvWriteParams& p, cudaStream_t stream);

// pkv_paged_attention_varlen with its workspace in caller-independent scratch
// of `scratch_bytes` bytes whose device address `scratch` returns (for the
// current device). Every host-side check runs first; a call whose workspace
// would exceed the scratch returns PKV_ERR_WORKSPACE; nothing is enqueued on
// an error. The work tickets are cleared on the stream before the launches.
int32_t attention_with_scratch(float* out, float* out_lse, const void* q, const void* kv_pool,
                               const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                               int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
                               int32_t max_seq_len, int32_t num_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int32_t num_blocks,
                               float scale, int32_t partition_size, int32_t* dev_status,
                               void* stream, size_t scratch_bytes,
                               cudaError_t (*scratch)(void**));

// Decode kernel (query_len == 1 requests): TMA-staged pages, QK^T and PV on
// the warp-level tensor cores (mma.sync); split-KV partitions merged by a
// second, small grid launched behind it. `kv_map` views the pool as
// [D/64][Hkv][2*NB*BS rows][64] (strides 128 B, D*2, Hkv*D*2) with a box of
// {64, 16, 1, D/64} and 128-byte swizzle. Up to 16 query heads per CTA.
cudaError_t launch_decode_mma(const AttnParams& p, const CUtensorMap& kv_map,
                              cudaStream_t stream);

// Chunked-prefill kernel (query_len > 1 requests), tcgen05 tensor cores.
// `q_map`: q as [T][H][D] with a box of {64, G, 128/G}, 128-byte swizzle.
// `kv_map`: the pool viewed as for the decode kernel but with a box of
// {64, 16, 1, 1} (one 64-column chunk of 16 keys), 128-byte swizzle.
// Launched with programmatic dependent launch: its CTAs start work after the
// preceding grid has completed, and let the next grid launch as soon as
// each has started.
cudaError_t launch_prefill(const AttnParams& p, const CUtensorMap& q_map,
                           const CUtensorMap& kv_map, cudaStream_t stream);

// Whether the prefill kernel's shared memory (its K/V/Q stages plus the work
// list of num_seqs requests) fits the 227 KB a CTA may have: up to 8575
// requests at head_dim 128, 33151 at 64. False for other head dims.
bool prefill_fits(int32_t num_seqs, int32_t head_dim);

// Shared-prefix (cascade) merge: row r of out (num_rows = B * H rows of
// head_dim) from the tail partial (slot 0) and the prefix segments (slots
// 1 .. segments of its request's group, prefix_segment_count of the group's
// prefix length; none for a request outside every group), each slot
// [num_rows][head_dim] fp32 with lse [num_rows]. Launched with programmatic
// dependent launch (waits for the grid before it).
cudaError_t launch_cascade_merge(float* out, float* out_lse, const float* part_out,
                                 const float* part_lse, int64_t num_rows, int32_t num_heads,
                                 int32_t head_dim, const int32_t* group_starts,
                                 const int32_t* prefix_lens, int32_t num_groups, int32_t splits,
                                 cudaStream_t stream);

// Whole-block copies in the pool; block_vecs = 16-byte vectors in one
// block of one half (K or V).
cudaError_t launch_copy_blocks(void* pool, const int32_t* src, const int32_t* dst,
                               int32_t num_copies, int32_t num_blocks, int64_t block_vecs,
                               int32_t* status, cudaStream_t stream);

// Public dense merge: part_out [P][T*H][D], part_lse [P][T*H].
cudaError_t launch_lse_merge(float* out, float* out_lse, const float* part_out,
                             const float* part_lse, int32_t num_parts, int64_t num_rows,
                             int32_t head_dim, cudaStream_t stream);


}  // namespace pkv
