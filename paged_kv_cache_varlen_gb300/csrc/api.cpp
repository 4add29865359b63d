// api.cpp -- the C ABI of libpkv (declared in include/pkv.h): host-side
// argument validation, TMA tensor-map encoding and kernel dispatch.
//
// Nothing here allocates device memory, synchronises a stream or keeps
// state across calls (the cached items are the driver entry point of
// cuTensorMapEncodeTiled and, per device, the kernels' shared-memory limits).
// Every host-side check and tensor-map encoding of a call happens before its
// first launch, so a rejected call enqueues nothing.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pkv.h"
#include "launch.h"

namespace {

using pkv::AttnParams;

// Automatic split-KV partitions: 1024 tokens, doubled until a request has at
// most 32 (measured on GB300: 1024 is best for contexts up to 4K, 4096 for
// 32K-128K; fewer, longer partitions amortise each CTA's prologue/epilogue).
constexpr int32_t kAutoPartition = 1024;
constexpr int32_t kMaxAutoParts = 32;
// partitions of one request at most (the decode grid's y dimension)
constexpr int32_t kMaxParts = 65535;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// A 3-D bf16 tensor [d2][d1][d0] (d0 contiguous) with byte strides s1, s2.
bool encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2,
               CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 4-D bf16 tensor [d3][d2][d1][d0] (d0 contiguous) with byte strides s1..s3.
bool encode_4d(CUtensorMap* map, const void* base, const uint64_t (&dims)[4],
               const uint64_t (&strides)[3], const uint32_t (&box)[4],
               CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t s[3] = {strides[0], strides[1], strides[2]};
  const cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), d, s, b, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Partition length and count for query_len == 1 requests.
bool resolve_partition(int32_t max_seq_len, int32_t partition_size, int32_t* ps, int32_t* np) {
  if (partition_size < -1) return false;
  if (partition_size > 0 && partition_size % 16 != 0) return false;
  const int32_t len = max_seq_len > 0 ? max_seq_len : 1;
  int32_t s = partition_size == 0 ? ((len + 15) / 16) * 16
                                  : (partition_size < 0 ? kAutoPartition : partition_size);
  // automatic: kAutoPartition tokens, doubled until at most kMaxAutoParts per
  // request (also bounds the partials the merge reads)
  while (partition_size < 0 && (len + s - 1) / s > kMaxAutoParts) s *= 2;
  int32_t n = (len + s - 1) / s;
  if (n <= 1) {
    n = 1;
    if (s < len) s = ((len + 15) / 16) * 16;
  }
  *ps = s;
  *np = n;
  return true;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: partial outputs [B][P][H][D] fp32 and partial lse [B][P][H]
// fp32 (split-KV only), then the prefill work tickets (256 bytes, always),
// which are zero between calls.
constexpr size_t kSchedBytes = 256;

// Batches of several-query (verification) requests run the decode grid in
// longest-request-first order when they have at most this many requests:
// their CTAs each stream a whole context, and in request order the longest
// ones could start last.
constexpr int32_t kOrderMaxSeqs = 256;

bool decode_ordered(int32_t num_seqs, int32_t num_tokens) {
  return num_tokens > num_seqs && num_seqs <= kOrderMaxSeqs;
}

struct WorkspaceLayout {
  size_t lse_off, sched_off, order_off, total;
};

// [split-KV partials][lse][tickets][decode order: num_seqs int32, only for
// batches decode_ordered() picks]
WorkspaceLayout workspace_layout(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                 int32_t nparts, bool ordered = false) {
  WorkspaceLayout w{0, 0, 0, 0};
  if (nparts > 1) {
    const size_t rows = (size_t)num_seqs * nparts * num_heads;
    w.lse_off = round_up(rows * head_dim * sizeof(float), 256);
    w.sched_off = w.lse_off + round_up(rows * sizeof(float), 256);
  }
  w.order_off = w.sched_off + kSchedBytes;
  w.total = w.order_off + (ordered ? round_up((size_t)num_seqs * sizeof(int32_t), 256) : 0);
  return w;
}

// Shared-prefix (cascade) decode: key segments per prefix so that the
// prefix pass spreads over about a fifth of a GPU's SMs (30 CTAs of its
// one-per-SM grid; the results do not depend on it): it runs beside the
// tail decode, which keeps the other SMs busy from the start. (Measured on
// 4 groups of 64 members sharing 2048-token prefixes: 113.8 us per call
// with one segment per group against 118.6 us with two.)
constexpr int64_t kCascadeRefSMs = 30;

int32_t cascade_splits(int32_t num_groups, int32_t max_group_size, int32_t max_prefix_len,
                       int32_t num_heads, int32_t num_kv_heads) {
  if (num_groups <= 0 || max_group_size <= 0 || max_prefix_len <= 0) return 1;
  const int32_t qp = 2 * (128 / (num_heads / num_kv_heads));  // queries per prefill work item
  const int64_t items = (int64_t)num_groups * ((max_group_size + qp - 1) / qp) * num_kv_heads;
  const int64_t tiles = (max_prefix_len + 127) / 128;
  int64_t s = (kCascadeRefSMs + items - 1) / items;
  if (s > tiles) s = tiles;
  return s < 1 ? 1 : (int32_t)s;
}

// Cascade workspace: partial outputs [S+1][B][H][D] fp32 and lse [S+1][B][H]
// (the tail, then S prefix segments), then the tail pass's own split-KV
// workspace (zero-filled once, like any attention workspace).
struct CascadeLayout {
  int32_t splits;
  size_t lse_off, ws_off, ws_bytes, ws_sched_off, total;
};

CascadeLayout cascade_layout(int32_t num_seqs, int32_t num_groups, int32_t max_group_size,
                             int32_t max_prefix_len, int32_t max_tail_len, int32_t num_heads,
                             int32_t num_kv_heads, int32_t head_dim) {
  CascadeLayout c{};
  c.splits = cascade_splits(num_groups, max_group_size, max_prefix_len, num_heads, num_kv_heads);
  const size_t rows = (size_t)(c.splits + 1) * num_seqs * num_heads;
  c.lse_off = round_up(rows * head_dim * sizeof(float), 256);
  c.ws_off = c.lse_off + round_up(rows * sizeof(float), 256);
  int32_t ps = 0, np = 1;
  resolve_partition(max_tail_len, -1, &ps, &np);
  const WorkspaceLayout wl = workspace_layout(num_seqs, num_heads, head_dim, np);
  c.ws_bytes = wl.total;
  c.ws_sched_off = wl.sched_off;
  c.total = c.ws_off + c.ws_bytes;
  return c;
}


// One attention call after every host-side check, with its tensor maps
// encoded: nothing has been enqueued yet. `empty` marks a call with no
// tokens (a no-op).
struct AttnPlan {
  AttnParams p{};
  bool ordered = false;   // decode-only batch run in longest-request-first order
  CUtensorMap kv_rows{};  // decode: 16-key boxes of whole rows of one KV head
  CUtensorMap q_map{};    // prefill: {64, G, 128/G} boxes of q
  CUtensorMap kv_box{};   // prefill: 16-key boxes of one 64-column chunk
  bool prefill = false;   // some request may have more queries than the decode kernel takes
  bool empty = false;
  WorkspaceLayout wl{};
};

pkv_status plan_attention(AttnPlan* a, float* out, float* out_lse, const void* q,
                          const void* kv_pool, const int32_t* block_table,
                          int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                          const int32_t* seq_lens, int32_t num_seqs, int32_t num_tokens,
                          int32_t max_query_len, int32_t max_seq_len, int32_t num_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, float scale, int32_t partition_size,
                          const int32_t* key_start, const int32_t* query_start,
                          int32_t* dev_status) {
  if (num_seqs < 0 || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) {
    a->empty = true;
    return PKV_OK;
  }
  if (num_seqs == 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65534) return PKV_ERR_UNSUPPORTED;  // grid z: requests + one
  if (!out || !q || !kv_pool || !block_table || !cu_seqlens_q || !seq_lens)
    return PKV_ERR_INVALID_ARG;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return PKV_ERR_INVALID_ARG;
  if (block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  // a key range may hold fewer keys than the request has queries
  if (max_query_len < 1 || max_seq_len < (key_start ? 1 : max_query_len))
    return PKV_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (block_size % 16 != 0 || block_size > 256) return PKV_ERR_UNSUPPORTED;
  if ((int64_t)2 * num_blocks * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const int32_t group = num_heads / num_kv_heads;
  if (max_query_len > 1 && (group > 128 || (128 % group) != 0)) return PKV_ERR_UNSUPPORTED;
  // requests longer than the decode kernel takes: the prefill kernel's work
  // list of num_seqs requests must fit its shared memory
  if (max_query_len > (32 / group > 1 ? 32 / group : 1) && !pkv::prefill_fits(num_seqs, head_dim))
    return PKV_ERR_UNSUPPORTED;

  int32_t ps = 0, np = 1;
  if (!resolve_partition(max_seq_len, partition_size, &ps, &np)) return PKV_ERR_INVALID_ARG;
  if (np > kMaxParts) return PKV_ERR_UNSUPPORTED;  // the decode grid's y dimension
  a->ordered = max_query_len <= (32 / group > 1 ? 32 / group : 1) &&
               decode_ordered(num_seqs, num_tokens);
  a->wl = workspace_layout(num_seqs, num_heads, head_dim, np, a->ordered);

  AttnParams& p = a->p;
  p.out = out;
  p.out_lse = out_lse;
  p.q = static_cast<const uint16_t*>(q);
  p.kv_pool = kv_pool;
  p.block_table = block_table;
  p.cu_seqlens = cu_seqlens_q;
  p.seq_lens = seq_lens;
  p.max_blocks = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_tokens = num_tokens;
  p.max_query_len = max_query_len;
  p.max_seq_len = max_seq_len;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.part_size = ps;
  p.num_parts = np;
  p.ws_out = nullptr;
  p.ws_lse = nullptr;
  p.sched = nullptr;
  p.status = dev_status;
  p.key_start = key_start;
  p.query_start = query_start;
  // the decode kernel takes requests of up to 32 (query, head) rows: two
  // subgroups of its 16-row MMA tiles
  p.decode_max_q = 32 / group > 1 ? 32 / group : 1;
  p.decode_max_rows = (max_query_len < p.decode_max_q ? max_query_len : p.decode_max_q) * group;
  p.prefix_mode = 0;
  p.kv_splits = 1;
  p.split_out_stride = 0;
  p.split_lse_stride = 0;

  a->prefill = max_query_len > p.decode_max_q;
  return PKV_OK;
}

// The pool [2][NB][BS][Hkv][D] viewed as [D/64][Hkv][2*NB*BS rows][64]
// (strides 128 B, D*2, Hkv*D*2; the V half starts at row NB*BS), 128-byte
// swizzle, with a box of 16 rows of one KV head and `chunks` 64-column
// chunks. With all D/64 chunks (decode) the box lands as the 16 keys' first
// 128-byte halves, then their second halves: 8 consecutive keys of one half
// then sit in 8 different bank groups (conflict-free ldmatrix). With one
// chunk (prefill) each copy lands 16 rows of one chunk of a 128-key tile.
bool encode_kv_view(CUtensorMap* map, const void* kv_pool, int32_t num_blocks, int32_t block_size,
                    int32_t num_kv_heads, int32_t head_dim, uint32_t chunks) {
  const uint64_t D = (uint64_t)head_dim;
  const uint64_t pool_rows = (uint64_t)2 * num_blocks * block_size;
  const uint64_t dims[4] = {64, pool_rows, (uint64_t)num_kv_heads, D / 64};
  const uint64_t strides[3] = {(uint64_t)num_kv_heads * D * 2, D * 2, 128};
  const uint32_t box[4] = {64, 16, 1, chunks};
  return encode_4d(map, kv_pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// q [T][H][D] with a box of {64, G, 128/G} (one 128-row Q tile per chunk).
bool encode_q_tiles(CUtensorMap* map, const void* q, int32_t num_tokens, int32_t num_heads,
                    int32_t num_kv_heads, int32_t head_dim) {
  const uint64_t D = (uint64_t)head_dim;
  const int32_t group = num_heads / num_kv_heads;
  return encode_3d(map, q, D, num_heads, num_tokens, D * 2, (uint64_t)num_heads * D * 2, 64,
                   (uint32_t)group, (uint32_t)(128 / group), CU_TENSOR_MAP_SWIZZLE_128B);
}

// Encode the plan's TMA tensor maps (needs the driver; still enqueues nothing).
pkv_status encode_plan(AttnPlan* a) {
  const AttnParams& p = a->p;
  if (!encode_kv_view(&a->kv_rows, p.kv_pool, p.num_blocks, p.block_size, p.num_kv_heads,
                      p.head_dim, (uint32_t)(p.head_dim / 64)))
    return PKV_ERR_CUDA;
  if (a->prefill &&
      (!encode_q_tiles(&a->q_map, p.q, p.num_tokens, p.num_heads, p.num_kv_heads, p.head_dim) ||
       !encode_kv_view(&a->kv_box, p.kv_pool, p.num_blocks, p.block_size, p.num_kv_heads,
                       p.head_dim, 1)))
    return PKV_ERR_CUDA;
  return PKV_OK;
}

// Point the plan at a caller's workspace after checking its size and alignment.
pkv_status bind_workspace(AttnPlan* a, void* workspace, size_t workspace_bytes) {
  if (!workspace || workspace_bytes < a->wl.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PKV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  a->p.sched = reinterpret_cast<int32_t*>(ws + a->wl.sched_off);
  if (a->ordered) a->p.order = reinterpret_cast<int32_t*>(ws + a->wl.order_off);
  if (a->p.num_parts > 1) {
    a->p.ws_out = reinterpret_cast<float*>(ws);
    a->p.ws_lse = reinterpret_cast<float*>(ws + a->wl.lse_off);
  }
  return PKV_OK;
}

// Whether some request may be short enough for the decode kernel: with
// every request at most max_query_len queries long and num_tokens in all,
// n_short requests of at most decode_max_q queries need
// n_short * (max_query_len - decode_max_q) <= num_seqs * max_query_len - num_tokens.
bool may_have_decode(const AttnParams& p) {
  return (int64_t)p.num_seqs * p.max_query_len - p.num_tokens >=
         (int64_t)p.max_query_len - p.decode_max_q;
}

// Enqueue a planned call, all on the caller's stream: the decode grid (and
// its split-KV merge grid) when no request is longer than the decode kernel
// takes; otherwise the prefill grid, then -- unless no request can be short
// -- the decode grid right behind it (programmatic dependent launch). The
// prefill grid keeps its share of the SMs and leaves the rest to the decode
// grid, which launches as soon as every prefill CTA has started or left;
// the decode grid completes only after the prefill grid has (see
// AttnParams::after_prefill), so the call completes when every grid has.
pkv_status launch_plan(const AttnPlan& a, cudaStream_t st) {
  if (!a.prefill)
    return pkv::launch_decode_mma(a.p, a.kv_rows, st) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  AttnParams pp = a.p;
  const bool decode = may_have_decode(a.p);
  if (decode) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKV_ERR_CUDA;
    pp.shared_sms = sms;
  } else {
    pp.no_decode = 1;
  }
  if (pkv::launch_prefill(pp, a.q_map, a.kv_box, st) != cudaSuccess) return PKV_ERR_CUDA;
  if (!decode) return PKV_OK;
  AttnParams d = a.p;
  d.after_prefill = 1;
  return pkv::launch_decode_mma(d, a.kv_rows, st) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

namespace pkv {
pkv_status attention_with_scratch(float* out, float* out_lse, const void* q, const void* kv_pool,
                                  const int32_t* block_table, int32_t max_blocks_per_seq,
                                  const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                                  int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
                                  int32_t max_seq_len, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                  float scale, int32_t partition_size, int32_t* dev_status,
                                  void* stream, size_t scratch_bytes,
                                  cudaError_t (*scratch)(void**)) {
  AttnPlan a;
  pkv_status s = plan_attention(&a, out, out_lse, q, kv_pool, block_table, max_blocks_per_seq,
                                cu_seqlens_q, seq_lens, num_seqs, num_tokens, max_query_len,
                                max_seq_len, num_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, scale, partition_size, nullptr, nullptr, dev_status);
  if (s != PKV_OK || a.empty) return s;
  if (a.wl.total > scratch_bytes) return PKV_ERR_WORKSPACE;
  if ((s = encode_plan(&a)) != PKV_OK) return s;
  void* base = nullptr;
  if (scratch(&base) != cudaSuccess) return PKV_ERR_CUDA;
  if ((s = bind_workspace(&a, base, scratch_bytes)) != PKV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the work tickets must start at zero (an interrupted earlier call may
  // have left them otherwise)
  if (cudaMemsetAsync(a.p.sched, 0, kSchedBytes, st) != cudaSuccess) return PKV_ERR_CUDA;
  return launch_plan(a, st);
}

}  // namespace pkv

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_NO_BLOCKS: return "block pool exhausted";
    default: return "unknown status";
  }
}

int32_t pkv_abi_version(void) { return 1; }

pkv_status pkv_kv_cache_write(void* kv_pool, const void* k_new, const void* v_new,
                              const int32_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                              int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                              int32_t* dev_status, void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!kv_pool || !k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned16(kv_pool) || !aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
  if (((int64_t)num_kv_heads * head_dim) % 8 != 0) return PKV_ERR_UNSUPPORTED;
  pkv::KvWriteParams p;
  p.pool = kv_pool;
  p.k_new = k_new;
  p.v_new = v_new;
  p.slot_mapping = slot_mapping;
  p.num_tokens = num_tokens;
  p.num_slots = (int64_t)num_blocks * block_size;
  p.row_vecs = num_kv_heads * head_dim / 8;
  p.status = dev_status;
  return pkv::launch_kv_write(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK
                                                                                    : PKV_ERR_CUDA;
}

size_t pkv_attention_workspace_size(int32_t num_seqs, int32_t num_tokens, int32_t num_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t max_seq_len,
                                    int32_t partition_size) {
  (void)num_kv_heads;
  int32_t ps = 0, np = 1;
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0) return 0;
  if (!resolve_partition(max_seq_len, partition_size, &ps, &np) || np > kMaxParts) return 0;
  return workspace_layout(num_seqs, num_heads, head_dim, np,
                          decode_ordered(num_seqs, num_tokens))
      .total;
}

pkv_status pkv_paged_attention_varlen(float* out, float* out_lse, const void* q,
                                      const void* kv_pool, const int32_t* block_table,
                                      int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                                      const int32_t* seq_lens, int32_t num_seqs,
                                      int32_t num_tokens, int32_t max_query_len,
                                      int32_t max_seq_len, int32_t num_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                      int32_t num_blocks, float scale, int32_t partition_size,
                                      void* workspace, size_t workspace_bytes,
                                      int32_t* dev_status, void* stream) {
  AttnPlan a;
  pkv_status s = plan_attention(&a, out, out_lse, q, kv_pool, block_table, max_blocks_per_seq,
                                cu_seqlens_q, seq_lens, num_seqs, num_tokens, max_query_len,
                                max_seq_len, num_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, scale, partition_size, nullptr, nullptr, dev_status);
  if (s != PKV_OK || a.empty) return s;
  if ((s = bind_workspace(&a, workspace, workspace_bytes)) != PKV_OK) return s;
  if ((s = encode_plan(&a)) != PKV_OK) return s;
  return launch_plan(a, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_paged_attention_varlen_append(
    float* out, float* out_lse, const void* q, void* kv_pool, const void* k_new, const void* v_new,
    const int32_t* slot_mapping, const int32_t* block_table, int32_t max_blocks_per_seq,
    const int32_t* cu_seqlens_q, const int32_t* seq_lens, int32_t num_seqs, int32_t num_tokens,
    int32_t max_query_len, int32_t max_seq_len, int32_t num_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale, int32_t partition_size,
    void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  // every check of both parts before the first launch
  AttnPlan a;
  pkv_status s = plan_attention(&a, out, out_lse, q, kv_pool, block_table, max_blocks_per_seq,
                                cu_seqlens_q, seq_lens, num_seqs, num_tokens, max_query_len,
                                max_seq_len, num_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, scale, partition_size, nullptr, nullptr, dev_status);
  if (s != PKV_OK || a.empty) return s;
  if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new))
    return PKV_ERR_INVALID_ARG;
  if ((s = bind_workspace(&a, workspace, workspace_bytes)) != PKV_OK) return s;
  if ((s = encode_plan(&a)) != PKV_OK) return s;
  pkv::KvWriteParams w;
  w.pool = kv_pool;
  w.k_new = k_new;
  w.v_new = v_new;
  w.slot_mapping = slot_mapping;
  w.num_tokens = num_tokens;
  w.num_slots = (int64_t)num_blocks * block_size;
  w.row_vecs = num_kv_heads * head_dim / 8;
  w.status = dev_status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (pkv::launch_kv_write(w, st) != cudaSuccess) return PKV_ERR_CUDA;
  a.p.early_pool = 1;
  return launch_plan(a, st);
}

pkv_status pkv_paged_attention_varlen_range(
    float* out, float* out_lse, const void* q, const void* kv_pool, const int32_t* block_table,
    int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q, const int32_t* seq_lens,
    const int32_t* key_start_pos, const int32_t* query_start_pos, int32_t num_seqs,
    int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
    int32_t partition_size, void* workspace, size_t workspace_bytes, int32_t* dev_status,
    void* stream) {
  if (num_tokens > 0 && (!key_start_pos || !query_start_pos)) return PKV_ERR_INVALID_ARG;
  AttnPlan a;
  pkv_status s = plan_attention(&a, out, out_lse, q, kv_pool, block_table, max_blocks_per_seq,
                                cu_seqlens_q, seq_lens, num_seqs, num_tokens, max_query_len,
                                max_seq_len, num_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, scale, partition_size, key_start_pos,
                                query_start_pos, dev_status);
  if (s != PKV_OK || a.empty) return s;
  if ((s = bind_workspace(&a, workspace, workspace_bytes)) != PKV_OK) return s;
  if ((s = encode_plan(&a)) != PKV_OK) return s;
  return launch_plan(a, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_copy_blocks(void* kv_pool, const int32_t* copy_src, const int32_t* copy_dst,
                           int32_t num_copies, int32_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, int32_t head_dim, int32_t* dev_status,
                           void* stream) {
  if (num_copies < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_copies == 0) return PKV_OK;
  if (!kv_pool || !copy_src || !copy_dst || !aligned16(kv_pool)) return PKV_ERR_INVALID_ARG;
  const int64_t block_bytes = (int64_t)block_size * num_kv_heads * head_dim * 2;
  if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_copies > 65535 || block_bytes / 16 / 1024 > 65535) return PKV_ERR_UNSUPPORTED;
  return pkv::launch_copy_blocks(kv_pool, copy_src, copy_dst, num_copies, num_blocks,
                                 block_bytes / 16, dev_status,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

size_t pkv_cascade_workspace_size(int32_t num_seqs, int32_t num_prefix_groups,
                                  int32_t max_group_size, int32_t max_prefix_len,
                                  int32_t max_tail_len, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim) {
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  if (num_heads % num_kv_heads != 0) return 0;
  return cascade_layout(num_seqs, num_prefix_groups, max_group_size, max_prefix_len, max_tail_len,
                        num_heads, num_kv_heads, head_dim)
      .total;
}

pkv_status pkv_cascade_decode(float* out, float* out_lse, const void* q, const void* kv_pool,
                              int32_t num_prefix_groups, const int32_t* group_starts,
                              const int32_t* prefix_lens, const int32_t* prefix_tables,
                              int32_t max_prefix_blocks, int32_t max_group_size,
                              int32_t max_prefix_len, const int32_t* tail_tables,
                              int32_t max_tail_blocks, const int32_t* tail_lens,
                              int32_t max_tail_len, int32_t num_seqs, int32_t num_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int32_t num_blocks, float scale, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (num_seqs < 0 || num_prefix_groups < 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !kv_pool || !tail_tables || !tail_lens) return PKV_ERR_INVALID_ARG;
  if (num_prefix_groups > 0 && (!group_starts || !prefix_lens || !prefix_tables ||
                                max_prefix_blocks <= 0 || max_group_size <= 0 ||
                                max_prefix_len < 0))
    return PKV_ERR_INVALID_ARG;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return PKV_ERR_INVALID_ARG;
  if (max_tail_len < 1 || max_tail_blocks <= 0) return PKV_ERR_INVALID_ARG;
  const int32_t group = num_heads / num_kv_heads;
  if (num_prefix_groups > 0 && max_prefix_len > 0 &&
      (group > 128 || (128 % group) != 0 || !pkv::prefill_fits(num_prefix_groups, head_dim)))
    return PKV_ERR_UNSUPPORTED;
  if ((int64_t)max_prefix_blocks * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const CascadeLayout c = cascade_layout(num_seqs, num_prefix_groups, max_group_size,
                                         max_prefix_len, max_tail_len, num_heads, num_kv_heads,
                                         head_dim);
  if (!workspace || workspace_bytes < c.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PKV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  float* part_out = reinterpret_cast<float*>(ws);
  float* part_lse = reinterpret_cast<float*>(ws + c.lse_off);
  const int64_t bh = (int64_t)num_seqs * num_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool prefixes = num_prefix_groups > 0 && max_prefix_len > 0;

  // Every check and tensor-map encoding happens before the first launch.
  // Tails: ordinary decode over each request's private blocks, one query per
  // request (request i is query i: no cu_seqlens array; tail_lens stands in
  // for it in the planning checks), into partial slot 0 -- or straight into
  // `out` when there is no prefix.
  AttnPlan tails;
  pkv_status s = plan_attention(
      &tails, prefixes ? part_out : out, prefixes ? part_lse : out_lse, q, kv_pool, tail_tables,
      max_tail_blocks, tail_lens, tail_lens, num_seqs, num_seqs, 1, max_tail_len, num_heads,
      num_kv_heads, head_dim, block_size, num_blocks, scale, -1, nullptr, nullptr, dev_status);
  if (s != PKV_OK) return s;
  tails.p.cu_seqlens = nullptr;
  if ((s = bind_workspace(&tails, ws + c.ws_off, c.ws_bytes)) != PKV_OK) return s;
  if ((s = encode_plan(&tails)) != PKV_OK) return s;
  if (!prefixes) return launch_plan(tails, st);
  // Prefixes: every group's queries against its shared blocks, once, on the
  // tensor cores (the prefill kernel in prefix mode), cut into key segments
  // written to partial slots 1 .. S.
  AttnParams p = tails.p;
  CUtensorMap q_map{}, kv_box{};
  p.out = part_out + bh * head_dim;
  p.out_lse = part_lse + bh;
  p.block_table = prefix_tables;
  p.cu_seqlens = group_starts;
  p.seq_lens = prefix_lens;
  p.max_blocks = max_prefix_blocks;
  p.num_seqs = num_prefix_groups;
  p.num_tokens = num_seqs;
  p.max_query_len = max_group_size;
  p.max_seq_len = max_prefix_len;
  p.part_size = 0;
  p.num_parts = 1;
  p.ws_out = nullptr;
  p.ws_lse = nullptr;
  p.sched = reinterpret_cast<int32_t*>(ws + c.ws_off + c.ws_sched_off);
  p.decode_max_q = 0;  // the prefix pass takes every group
  p.decode_max_rows = 0;
  p.prefix_mode = 1;
  p.kv_splits = c.splits;
  p.split_out_stride = bh * head_dim;
  p.split_lse_stride = bh;
  if (!encode_q_tiles(&q_map, q, num_seqs, num_heads, num_kv_heads, head_dim) ||
      !encode_kv_view(&kv_box, kv_pool, num_blocks, block_size, num_kv_heads, head_dim, 1))
    return PKV_ERR_CUDA;

  // 1. the prefix pass (its grid sized for about a fifth of the SMs);
  // 2. right behind it, on the SMs it leaves, the tails (their grid
  // completes only after the prefix pass has); 3. every request's tail and
  // prefix segments merged by log-sum-exp
  if (pkv::launch_prefill(p, q_map, kv_box, st) != cudaSuccess) return PKV_ERR_CUDA;
  AttnParams d = tails.p;
  d.after_prefill = 1;
  if (pkv::launch_decode_mma(d, tails.kv_rows, st) != cudaSuccess) return PKV_ERR_CUDA;
  return pkv::launch_cascade_merge(out, out_lse, part_out, part_lse, bh, num_heads, head_dim,
                                   group_starts, prefix_lens, num_prefix_groups, c.splits,
                                   st) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

pkv_status pkv_lse_merge(float* out, float* out_lse, const float* part_out, const float* part_lse,
                         int32_t num_parts, int32_t num_tokens, int32_t num_heads,
                         int32_t head_dim, void* stream) {
  if (num_parts < 1 || num_tokens < 0 || num_heads < 1 || head_dim < 1) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!out || !part_out || !part_lse) return PKV_ERR_INVALID_ARG;
  if (head_dim % 4 != 0 || head_dim > 512) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(out) || !aligned16(part_out)) return PKV_ERR_INVALID_ARG;
  return pkv::launch_lse_merge(out, out_lse, part_out, part_lse, num_parts,
                               (int64_t)num_tokens * num_heads, head_dim,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // extern "C"
