// prefill_tc.cu -- paged causal attention for query_len > 1 requests
// (prefill chunks), on the 5th-generation tensor cores (tcgen05).
//
// Method (sources as cited in include/pkv.h):
//   page 1 §04: prefill is a dense matrix product (compute-bound); GQA index
//     map kv_head = q_head / (num_heads / num_kv_heads); flattened queries
//     separated by cu_seqlens.
//   page 1 §07 / page 2 step 5: chunked prefill -- a chunk's queries attend
//     to the already cached context plus the chunk itself.
//   page 2 step 4: causal mask; query j of a request with seq_len L and
//     query_len q sits at position L - q + j and sees keys 0 .. L - q + j.
//   page 3 §3.4: FlashAttention -- S and P stay on chip, tile by tile, exact.
//
// GB300 design:
//   * persistent CTAs, one per SM: every CTA builds the list of work items in
//     shared memory (heaviest request first) and takes items dynamically
//     from a global ticket counter in the workspace; an item is (request, KV
//     head, two consecutive query tiles A and B of 128/G queries each), later
//     items (more keys) first. Tensor memory and barriers are set up once
//     per CTA; requests short enough for the decode kernel (1 ..
//     decode_max_q queries) give no items here. When a decode grid shares
//     the call, the grid keeps about its share of the SMs (prefill tiles
//     against decode bytes) and its other CTAs leave at once;
//   * a Q tile is 128 rows = (128/G queries) x (G heads sharing the KV head),
//     so one pass over the K/V pages serves the whole GQA group, and both Q
//     tiles of the item share every K/V tile loaded;
//   * Q, K and V arrive by TMA with the 128-byte swizzle the MMA descriptors
//     read: Q in {64, G, 128/G} boxes, a 128-key K or V tile as 8 boxes of 16
//     keys (one page run; block ids from block_table) per 64-column chunk,
//     issued by one thread per role (warp 14: Q and K, warp 15: V) into
//     2-stage rings. Warps 8-11, one on each SM sub-partition (a stage is
//     ready when its slowest converter is), convert each V stage to fp16 in
//     place, zeroing rows not loaded or past the needed keys;
//   * S = Q K^T (M=128, N=64, K=head_dim, bf16) and O += P V (M=128,
//     N=head_dim, K=16 per step, fp16) run as tcgen05.mma kind::f16 with
//     fp32 accumulation in tensor memory: per Q tile two S buffers of 64
//     columns and O (2 x (64 + 64 + 128) = 512 columns). P is written back
//     as fp16 pairs over the S columns it came from and is the A operand
//     straight from TMEM;
//   * one issuing thread per Q tile (warps 12, 13): QK^T of the next S tile
//     is issued right behind the PV of the current one, so S of tile j+1 is
//     ready while the softmax works on tile j, and the softmax warps go from
//     one tile to the next without waiting for the tensor core;
//   * two softmax warpgroups, one per Q tile; thread r of a warpgroup owns
//     TMEM lane (= Q row) r: it loads the row's 64 scores into registers
//     (one TMEM round trip), takes the maximum, computes the probabilities
//     with the exp2-domain online softmax (lazy rescale when the maximum
//     grows by more than 8), stores them as fp16 pairs and adds the rounded
//     values to the row sum (so that O and l see the same weights); O is
//     rescaled in TMEM when needed; a tile every key of which is visible to
//     the warp's rows skips the mask and uses packed fp32x2 arithmetic;
//   * every wait is bounded; on a timeout the CTA drains its copies and
//     MMAs, frees its TMEM and leaves with PKV_DEV_TIMEOUT set.
#include <math.h>

#include "common.cuh"
#include "launch.h"

#ifdef PKV_TEST_HOLD_ARRIVAL
// Test builds only: while set, softmax warp 0 of CTA 0 withholds its P-ready
// arrival for its first tile, so that the MMA thread's bounded wait runs out.
__device__ int g_pkv_test_hold_prefill;
extern "C" int pkv_test_hold_prefill(int on) {
  return (int)cudaMemcpyToSymbol(g_pkv_test_hold_prefill, &on, sizeof(int));
}
#endif

namespace pkv {
namespace {

constexpr int kBM = 128;                             // Q rows per tile
constexpr int kQT = 2;                               // Q tiles per work item
constexpr int kBN = 128;                             // keys per K/V tile (one ring stage)
constexpr int kSN = 64;                              // keys per S tile (half a K/V tile)
constexpr int kSB = 2;                               // S buffers per Q tile
constexpr int kNS = 2;                               // stages of each of the K and V rings
constexpr int kSub = 16;                             // keys per TMA box
constexpr int kSoftmaxThreads = kQT * kBM;           // warps 0 .. 7 (warpgroups 0, 1)
constexpr int kConvWarp0 = kSoftmaxThreads / 32;     // warps 8-11: V to fp16 (one per sub-partition)
constexpr int kMmaWarp = kConvWarp0 + 4;             // warps 12, 13: MMA issue for Q tiles A, B
constexpr int kProdWarp0 = kMmaWarp + 2;             // warp 14: Q and K tiles
constexpr int kVWarp0 = kProdWarp0 + 1;              // warp 15: V tiles
constexpr int kConverters = 4 * 32;
__device__ __forceinline__ int converter_slot(int warp) {
  return warp - kConvWarp0;
}
constexpr int kThreads = 512;                        // four warpgroups
// registers per thread: launched with 128; the softmax warpgroups take 152,
// the producer / MMA warpgroups give theirs down to 104 (2*152 + 2*104 = 4*128)
constexpr int kSoftmaxRegs = 152;
constexpr int kOtherRegs = 104;
static_assert(2 * kSoftmaxRegs + 2 * kOtherRegs == 4 * (65536 / kThreads),
              "the register split adds up to the launch's registers");
constexpr uint32_t kTmemCols = 512;
constexpr int kRing = 4;  // work items announced ahead of the roles that consume them
// readers of an announced item: the V producer warp, the two MMA threads,
// the eight softmax warps and the four converter warps (one lane each)
constexpr int kItemReaders = 1 + kQT + kSoftmaxThreads / 32 + kConverters / 32;
constexpr float kRescaleThreshold = 8.f;
constexpr uint32_t kFullMask = 0xffffffffu;

// The work list handed out by the tickets. For batches of at most
// kSortMax requests it holds the requests that have work, heaviest first
// (by the key tiles of their heaviest unit): an approximate
// longest-processing-time-first schedule, since a CTA takes the next ticket
// when it finishes an item (in request order the longest prefill chunks came
// last and left most SMs idle for their tail). Larger batches keep request
// order. Shared-memory ints: key, candidate, order and prefix arrays of
// B + 1 each when sorted, else the prefix array alone.
constexpr int kSortMax = 2048;
__host__ __device__ constexpr size_t work_list_ints(int num_seqs) {
  return num_seqs <= kSortMax ? 4 * ((size_t)num_seqs + 1) : (size_t)num_seqs + 1;
}

template <int D>
struct PrefillLayout {
  static constexpr int NCH = D / 64;                       // 128-byte column chunks of a row
  static constexpr int CH_BYTES = 128 * 128;               // one chunk of 128 rows
  static constexpr int TILE_BYTES = NCH * CH_BYTES;        // one Q, K or V tile
  static constexpr int Q_OFF = 0;                          // [kQT] Q tiles of the item
  static constexpr int K_OFF = Q_OFF + kQT * TILE_BYTES;   // [kNS] K tiles
  static constexpr int V_OFF = K_OFF + kNS * TILE_BYTES;   // [kNS] V tiles
  static constexpr int BAR_OFF = V_OFF + kNS * TILE_BYTES;
  static constexpr int PREF_OFF = BAR_OFF + 512;   // the work list (see WorkList)
  // keep one CTA per SM (each CTA allocates all 512 TMEM columns)
  static size_t bytes(int num_seqs) {
    const size_t need = 1024 + PREF_OFF + work_list_ints(num_seqs) * 4;
    return need > 120 * 1024 ? need : 120 * 1024;
  }
  // TMEM columns of Q tile x: its two S buffers of kSN columns (P written
  // in place), then O
  __device__ static constexpr uint32_t s_col(int x, int b) {
    return 256u * (uint32_t)x + (uint32_t)(b * kSN);
  }
  __device__ static constexpr uint32_t o_col(int x) { return 256u * (uint32_t)x + 128u; }
  // P of keys 16*kk .. 16*kk+15 inside an S buffer: fp16 pairs in 8 columns
  __device__ static constexpr uint32_t p_col(int kk) { return 8u * (uint32_t)kk; }
};
static_assert(kQT * (kSB * kSN + 128) <= (int)kTmemCols, "S and O of every Q tile fit in TMEM");

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kNS], k_empty[kNS];
  uint64_t v_full[kNS], v_empty[kNS];
  uint64_t v_landed[kNS];  // V copies arrived (bf16), not yet converted
  uint64_t s_full[kQT][kSB];  // QK^T of the S tile landed in buffer b of S_x
  // the warpgroup stored P(g) of Q tile x (and rescaled O_x): barrier
  // [x][g & 1], phase g >> 1. Two barriers, alternating by S tile: the
  // softmax may run a tile ahead of the issuer (it waits for the previous PV
  // only to rescale O), but not two (P(g + 2) needs QK(g + 2), issued after
  // PV(g)), so a barrier is never two phases past its waiter.
  uint64_t p_ready[kQT][2];
  // PV(g) of Q tile x finished (O_x stable): barrier [x][g & 1], phase g >> 1.
  // Two barriers, alternating by S tile: a waiter for PV(g) then always finds
  // the barrier at PV(g)'s phase or the one after (PV(g - 2) is complete once
  // S(g + 1) has been seen, PV(g + 2) cannot be issued before P(g + 2)), so
  // the softmax needs to wait only when it rescales O.
  uint64_t o_done[kQT][2];
  uint64_t o_free[kQT];   // the warpgroup's epilogue has read O_x
  uint64_t mma_done;
  uint64_t item_full[kRing], item_empty[kRing];
  int32_t item_id[kRing];  // work item taken from the global ticket counter, -1: none left
  uint32_t tmem_base;
  int32_t abort;
  int32_t scan[kThreads / 32];
  uint32_t v_mask[kNS];  // boxes of the V stage that were loaded (bit b: keys 16b .. 16b+15)
  float red[2][kThreads / 32];
};

static_assert(sizeof(Bars) <= 512, "the barriers fit below the work list");

struct PrefillItem {
  int req, kvh, j0, j1, t0, qlen, L, kv_end, n_tiles;
  int n_sub;  // S tiles of kSN keys: the needed keys of the n_tiles K/V tiles (at least 1)
  int qpos0;  // position of the request's first query among its keys
  int jb;   // first key tile of the item (a key segment in prefix mode)
  int seg;  // key segment (prefix mode), else 0
};

static_assert(kBN == 128, "prefix segments count 128-key tiles");

// Work units (pairs of query tiles) of request r (0 for requests of at most
// decode_max_q queries, which the decode kernel takes);
// bad lengths flagged by CTA 0. QP = queries per unit.
__device__ __forceinline__ int prefill_units(const AttnParams& p, int r, int QP, bool flag) {
  const int32_t t0 = __ldg(p.cu_seqlens + r), t1 = __ldg(p.cu_seqlens + r + 1);
  if (t0 < 0 || t1 < t0 || t1 > p.num_tokens) {
    if (flag) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return 0;
  }
  const int32_t qlen = t1 - t0;
  if (p.prefix_mode) {  // a prefix group: qlen queries, all seeing L keys
    const int32_t L = __ldg(p.seq_lens + r);
    if (qlen > p.max_query_len || L < 0 || L > p.max_seq_len || L > p.max_blocks * p.block_size) {
      if (flag) set_status(p.status, PKV_DEV_BAD_LENGTHS);
      return 0;
    }
    if (qlen < 1 || L == 0) return 0;
    return ((qlen + QP - 1) / QP) * prefix_segment_count(L, p.kv_splits);
  }
  if (qlen <= p.decode_max_q) {  // short requests run on the decode kernel
    if (p.no_decode && qlen > 0 && flag) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return 0;
  }
  const int32_t L = __ldg(p.seq_lens + r);
  const bool bad_range =
      p.key_start ? (L < 1 || __ldg(p.key_start + r) < 0 || __ldg(p.query_start + r) < 0)
                  : L < qlen;
  if (qlen > p.max_query_len || bad_range || L > p.max_seq_len ||
      L > p.max_blocks * p.block_size) {
    if (flag) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return 0;
  }
  return (qlen + QP - 1) / QP;
}

// Key tiles of request r's heaviest work unit (its last queries see the
// most keys), for the heaviest-first order; call only for requests with work.
__device__ __forceinline__ int prefill_weight(const AttnParams& p, int r) {
  const int32_t L = __ldg(p.seq_lens + r);
  if (p.prefix_mode) return prefix_tiles_per_segment(L, p.kv_splits);
  const int32_t qlen = __ldg(p.cu_seqlens + r + 1) - __ldg(p.cu_seqlens + r);
  int64_t end = L;  // ordinary call: the last query sees every key
  if (p.key_start) {
    end = (int64_t)__ldg(p.query_start + r) - __ldg(p.key_start + r) + qlen;
    end = end < 0 ? 0 : (end > L ? L : end);
  }
  return (int)((end + kBN - 1) / kBN);
}

// Exclusive prefix sum of one value per thread over the CTA; *total gets the
// sum. All threads; two __syncthreads.
__device__ __forceinline__ int block_exclusive_scan(int v, int32_t* scan, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scan[warp] = incl;
  __syncthreads();
  int base = 0, all = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) base += scan[w];
    all += scan[w];
  }
  __syncthreads();
  *total = all;
  return base + incl - v;
}

// The work list in shared memory: positions 0 .. n-1 in the order their units
// are handed out; request of position k = sorted ? order[k] : k; units
// before position k = pref[k], pref[n] = total.
struct WorkList {
  const int* order;
  const int* pref;
  int n;
  bool sorted;
};

// Builds the work list (all threads); returns it and sets *total_units.
__device__ __forceinline__ WorkList prefill_work_list(const AttnParams& p, int* base,
                                                      int32_t* scan, int QP, int* total_units) {
  const int B = p.num_seqs;
  const int tid = threadIdx.x;
  const bool flag = blockIdx.x == 0;
  const int per = (B + kThreads - 1) / kThreads;
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  WorkList wl;
  if (B > kSortMax) {  // request order: pref over every request
    int* pref = base;
    int sum = 0;
    for (int r = r0; r < r1; ++r) sum += prefill_units(p, r, QP, flag);
    int total = 0;
    int run = block_exclusive_scan(sum, scan, &total);
    for (int r = r0; r < r1; ++r) {
      pref[r] = run;
      run += prefill_units(p, r, QP, false);
    }
    if (tid == kThreads - 1) pref[B] = total;
    __syncthreads();
    *total_units = total;
    wl.order = nullptr;
    wl.pref = pref;
    wl.n = B;
    wl.sorted = false;
    return wl;
  }
  int* key = base;               // [B] weight of each request with work, -1 otherwise
  int* cand = base + (B + 1);    // [n] requests with work, in request order
  int* order = cand + (B + 1);   // [n] the same, heaviest first
  int* pref = order + (B + 1);   // [n + 1]
  int cnt = 0;
  for (int r = r0; r < r1; ++r) {
    const bool work = prefill_units(p, r, QP, flag) > 0;
    key[r] = work ? prefill_weight(p, r) : -1;
    cnt += work ? 1 : 0;
  }
  int n = 0;
  int pos = block_exclusive_scan(cnt, scan, &n);
  for (int r = r0; r < r1; ++r)
    if (key[r] >= 0) cand[pos++] = r;
  __syncthreads();
  // rank among the candidates: heavier first, ties by request index
  for (int i = tid; i < n; i += kThreads) {
    const int r = cand[i], k = key[r];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const int r2 = cand[j], k2 = key[r2];
      rank += (k2 > k || (k2 == k && r2 < r)) ? 1 : 0;
    }
    order[rank] = r;
  }
  __syncthreads();
  const int per2 = (n + kThreads - 1) / kThreads;
  const int k0 = min(n, tid * per2), k1 = min(n, k0 + per2);
  int sum = 0;
  for (int k = k0; k < k1; ++k) sum += prefill_units(p, order[k], QP, false);
  int total = 0;
  int run = block_exclusive_scan(sum, scan, &total);
  for (int k = k0; k < k1; ++k) {
    pref[k] = run;
    run += prefill_units(p, order[k], QP, false);
  }
  if (tid == kThreads - 1) pref[n] = total;
  __syncthreads();
  *total_units = total;
  wl.order = order;
  wl.pref = pref;
  wl.n = n;
  wl.sorted = true;
  return wl;
}

// Calibration of the SM split of a mixed call, measured on GB300: a
// 128-key tile pair (two Q tiles) takes ~4800 cycles of an SM in this
// kernel; the decode kernel streams ~40 bytes of K/V per cycle of an SM
// when it has only some of the SMs. (Swept on a mixed step of 48 decodes
// and four 512-query chunks: 3000, 3800, 4800, 5800 and 6300 cycles gave
// 312, 285, 269, 271 and 272 us per call; with the current kernel 4400, 4800,
// 5100 and 5400 gave 273.5, 270.0, 270.0 and 271.2 us on one box.)
constexpr float kPairCycles = 4800.f;
constexpr float kDecodeBytesPerCycle = 40.f;

// The CTAs of this grid that take prefill work when a decode grid shares the
// SMs: out of p.shared_sms, the prefill work's share of the estimated SM
// time (its tile pairs against the decode requests' K/V bytes), at least 1.
// All threads (two __syncthreads); every CTA computes the same value.
__device__ __noinline__ int prefill_share(const AttnParams& p, int QP, float (*red)[kThreads / 32]) {
  const int B = p.num_seqs;
  const int per = (B + kThreads - 1) / kThreads;
  const int r0 = min(B, (int)threadIdx.x * per), r1 = min(B, r0 + per);
  float pairs = 0.f, dkeys = 0.f;
  for (int r = r0; r < r1; ++r) {
    const int32_t t0 = __ldg(p.cu_seqlens + r), qlen = __ldg(p.cu_seqlens + r + 1) - t0;
    const int32_t L = __ldg(p.seq_lens + r);
    if (qlen < 1 || L < 1 || L > p.max_seq_len) continue;
    if (qlen <= p.decode_max_q) {
      dkeys += (float)L;
      continue;
    }
    int64_t q0 = (int64_t)L - qlen;  // position of the first query among the keys
    if (p.key_start) q0 = (int64_t)__ldg(p.query_start + r) - __ldg(p.key_start + r);
    for (int j1 = min(qlen, QP);; j1 = min(qlen, j1 + QP)) {
      const int64_t end = max((int64_t)0, min((int64_t)L, q0 + j1));
      pairs += (float)max((int64_t)1, (end + kBN - 1) / kBN);
      if (j1 == qlen) break;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pairs += __shfl_xor_sync(kFullMask, pairs, o);
    dkeys += __shfl_xor_sync(kFullMask, dkeys, o);
  }
  if (lane == 0) {
    red[0][warp] = pairs;
    red[1][warp] = dkeys;
  }
  __syncthreads();
  float pt = 0.f, dt = 0.f;
  for (int w = 0; w < kThreads / 32; ++w) {
    pt += red[0][w];
    dt += red[1][w];
  }
  __syncthreads();
  const float a = dt * (float)(p.num_kv_heads * p.head_dim * 4) / kDecodeBytesPerCycle;
  const float b = pt * (float)p.num_kv_heads * kPairCycles;
  const int S = p.shared_sms;
  const int keep = a + b > 0.f ? S - (int)((float)S * a / (a + b) + 0.5f) : S;
  return max(1, min(S, keep));
}

__device__ __forceinline__ PrefillItem prefill_item(const AttnParams& p, const WorkList& wl, int QP,
                                                    int it) {
  PrefillItem d;
  const int u = it / p.num_kv_heads;
  d.kvh = it - u * p.num_kv_heads;
  int lo = 0, hi = wl.n;  // largest lo with pref[lo] <= u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (wl.pref[mid] <= u)
      lo = mid;
    else
      hi = mid;
  }
  const int req = wl.sorted ? wl.order[lo] : lo;
  const int local = u - wl.pref[lo];
  d.req = req;
  d.t0 = __ldg(p.cu_seqlens + req);
  d.qlen = __ldg(p.cu_seqlens + req + 1) - d.t0;
  d.L = __ldg(p.seq_lens + req);
  const int ntq = (d.qlen + QP - 1) / QP;
  d.qpos0 = d.L - d.qlen;
  if (p.prefix_mode) {
    const int segs = prefix_segment_count(d.L, p.kv_splits);
    const int tps = prefix_tiles_per_segment(d.L, p.kv_splits);
    d.seg = local % segs;
    d.j0 = (local / segs) * QP;
    d.j1 = min(d.qlen, d.j0 + QP);
    d.kv_end = d.L;  // every query sees the whole prefix
    d.jb = d.seg * tps;
    d.n_tiles = min((d.L + kBN - 1) / kBN, d.jb + tps) - d.jb;
    d.n_sub = max(1, (min(d.L, (d.jb + d.n_tiles) * kBN) - d.jb * kBN + kSN - 1) / kSN);
    return d;
  }
  const int qt = ntq - 1 - local;  // later (heavier) units first
  d.j0 = qt * QP;
  d.j1 = min(d.qlen, d.j0 + QP);
  if (p.key_start) {  // key range: the queries' positions come from the caller
    const int64_t rel = (int64_t)__ldg(p.query_start + req) - __ldg(p.key_start + req);
    d.qpos0 = (int)max((int64_t)-(1 << 30), min((int64_t)(1 << 30), rel));
  }
  // keys [0, kv_end) are needed; at least one tile runs (fully masked when no
  // key is visible) so that the item's rows are written
  d.kv_end = max(0, min(d.L, d.qpos0 + d.j1));
  d.n_tiles = max(1, (d.kv_end + kBN - 1) / kBN);
  d.n_sub = max(1, (d.kv_end + kSN - 1) / kSN);
  d.jb = 0;
  d.seg = 0;
  return d;
}

// Work items are handed out dynamically: the first producer warp takes the
// next ticket from the global counter p.sched[0] and announces it in a small
// ring; every other role reads the same sequence from the ring. A CTA that
// finishes counts itself in p.sched[1]; the last one resets both counters, so
// they are zero again for the next call.
__device__ __forceinline__ int take_item(Bars* bars, const AttnParams& p, int total, int k,
                                         volatile int32_t* abort) {
  const int slot = k % kRing;
  bool w = true;
  if (k >= kRing)
    w = mbar_wait(smem_addr(&bars->item_empty[slot]), ((k / kRing) - 1) & 1, p.status, abort);
  int it = -1;
  if (w) {
    const int t = atomicAdd(p.sched, 1);
    it = t < total ? t : -1;
  }
  *reinterpret_cast<volatile int32_t*>(&bars->item_id[slot]) = it;
  mbar_arrive(smem_addr(&bars->item_full[slot]));
  return it;
}

__device__ __forceinline__ int read_item(Bars* bars, const AttnParams& p, int k,
                                         volatile int32_t* abort) {
  const int slot = k % kRing;
  int it = -1;
  if (mbar_wait(smem_addr(&bars->item_full[slot]), (k / kRing) & 1, p.status, abort))
    it = *reinterpret_cast<volatile int32_t*>(&bars->item_id[slot]);
  mbar_arrive(smem_addr(&bars->item_empty[slot]));
  return it;
}

// 32 bytes to global memory in one store (the address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(float* p, float a, float b, float c, float d, float e,
                                             float f, float g, float h) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(a),
               "f"(b), "f"(c), "f"(d), "f"(e), "f"(f), "f"(g), "f"(h)
               : "memory");
}

// Two fp32 values as fp16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// acc += both fp16 halves of h (exactly, in fp32).
__device__ __forceinline__ void add_f16x2_to(float& a, float& b, uint32_t h) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
      : "+f"(a), "+f"(b)
      : "r"(h));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// One 16-byte piece of a V tile (8 bf16 values) converted in place to fp16
// (exact for |v| < 65536: fp16 keeps bf16's 8 significant bits); the
// exponent fields seen are folded into emax (per 16-bit half) for the range
// check.
__device__ __forceinline__ void v_piece_to_f16(uint32_t addr, uint32_t& emax) {
  uint32_t w[4];
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(addr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("max.u16x2 %0, %0, %1;" : "+r"(emax) : "r"(w[i] & 0x7f807f80u));
    w[i] = pack_f16x2(bf16_lo(w[i]), bf16_hi(w[i]));
  }
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3])
               : "memory");
}

template <int R>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

__device__ __forceinline__ void cta_finished(const AttnParams& p) {  // one thread
  __threadfence();
  if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
    p.sched[0] = 0;
    p.sched[1] = 0;
    __threadfence();
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap kv_map, const AttnParams p) {
  using Lay = PrefillLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + Lay::BAR_OFF);
  int* list_base = reinterpret_cast<int*>(smem + Lay::PREF_OFF);

  griddep_wait();  // the KV write (and all earlier work) has landed
  griddep_launch_dependents();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.num_heads / p.num_kv_heads;
  const int QT = kBM / G;   // queries per Q tile
  const int QP = kQT * QT;  // queries per work item

  // ---- setup: barriers (first producer warp), work list (all), TMEM (MMA warp)
  if (warp == kProdWarp0 && lane == 0) {
    mbar_init(smem_addr(&bars->q_full), 1);
    mbar_init(smem_addr(&bars->q_empty), kQT);  // one commit per MMA thread
    for (int s = 0; s < kNS; ++s) {
      mbar_init(smem_addr(&bars->k_full[s]), 1);  // the producer's arrival + TMA bytes
      mbar_init(smem_addr(&bars->k_empty[s]), kQT);
      mbar_init(smem_addr(&bars->v_full[s]), kConverters);
      mbar_init(smem_addr(&bars->v_empty[s]), kQT);
      mbar_init(smem_addr(&bars->v_landed[s]), 1);
    }
    for (int x = 0; x < kQT; ++x) {
      for (int b = 0; b < kSB; ++b) mbar_init(smem_addr(&bars->s_full[x][b]), 1);
      for (int b = 0; b < 2; ++b)  // one arrival per softmax warp
        mbar_init(smem_addr(&bars->p_ready[x][b]), kBM / 32);
      for (int b = 0; b < 2; ++b) mbar_init(smem_addr(&bars->o_done[x][b]), 1);
      mbar_init(smem_addr(&bars->o_free[x]), kBM / 32);
    }
    mbar_init(smem_addr(&bars->mma_done), kQT);
    for (int k = 0; k < kRing; ++k) {
      mbar_init(smem_addr(&bars->item_full[k]), 1);
      mbar_init(smem_addr(&bars->item_empty[k]), kItemReaders);
    }
    bars->abort = 0;
    fence_barrier_init();
  }
  int total_units = 0;
  const WorkList wl = prefill_work_list(p, list_base, bars->scan, QP, &total_units);  // syncs
  const int total = total_units * p.num_kv_heads;
  const int active = p.shared_sms > 0 ? prefill_share(p, QP, bars->red) : (int)gridDim.x;  // syncs
  if ((int)blockIdx.x >= min(total, active)) {  // uniform; nothing allocated yet
    if (threadIdx.x == 0) cta_finished(p);
    return;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int32_t* abort = &bars->abort;

  const uint32_t q_s = smem_addr(smem + Lay::Q_OFF);
  const uint32_t k_s = smem_addr(smem + Lay::K_OFF);
  const uint32_t v_s = smem_addr(smem + Lay::V_OFF);

  // Each role changes its register budget at the top of its own branch (no
  // control-flow merge between the change and the code that relies on it):
  // warpgroups 2 (converters) and 3 (MMA issue, copies) give registers
  // back, warpgroups 0 and 1 (softmax) take them.
  if (warp >= kConvWarp0) {
    setmaxnreg_dec<kOtherRegs>();
    // ===== producers: Q and the K tiles (warp 14), the V tiles (warp 15),
    // all by TMA =====
    // A 128-key tile is 8 boxes of 16 keys (a 16-key run never crosses a
    // page: block_size is a multiple of 16), each box one TMA copy per
    // 64-column chunk, landing 128-byte-swizzled in the layout the MMA
    // descriptors read. Boxes wholly past the needed keys, or in a page
    // whose id is bad, are not loaded: K rows there are masked by the
    // softmax (bad-block K rows are zeroed here), V rows are zeroed by the
    // converter warps (P is 0 there, but 0 * NaN is not 0).
    if (warp == kProdWarp0 || warp == kVWarp0) {
      const bool vrole = warp == kVWarp0;
      const int32_t half_rows = vrole ? p.num_blocks * p.block_size : 0;  // first V row of the view
      const uint32_t ring = vrole ? v_s : k_s;
      if (lane == 0) {
        prefetch_tmap(&kv_map);
        if (!vrole) prefetch_tmap(&q_map);
      }
      int gi = 0, gt = 0, armed = 0, q_issued = 0;
      bool ok = true, bad_block = false;
      for (;; ++gi) {
        int it = -1;
        if (lane == 0)
          it = vrole ? read_item(bars, p, gi, abort) : take_item(bars, p, total, gi, abort);
        it = __shfl_sync(kFullMask, it, 0);
        if (it < 0) break;
        const PrefillItem d = prefill_item(p, wl, QP, it);
        const int32_t* bt = p.block_table + (int64_t)d.req * p.max_blocks;
        if (!vrole) {
          int w = 1;
          if (lane == 0 && gi >= 1)  // the previous item's QK^T products are done with Q
            w = mbar_wait(smem_addr(&bars->q_empty), (gi - 1) & 1, p.status, abort);
          ok = __shfl_sync(kFullMask, w, 0) != 0;
          if (!ok) break;
          if (lane == 0) {
            // rows past the last token read as zeros; rows of the next request
            // are loaded but belong to no valid output row
            mbar_arrive_expect_tx(smem_addr(&bars->q_full), kQT * Lay::TILE_BYTES);
            for (int x = 0; x < kQT; ++x)
              for (int c = 0; c < Lay::NCH; ++c)
                tma_load_3d(q_s + x * Lay::TILE_BYTES + c * Lay::CH_BYTES, &q_map,
                            smem_addr(&bars->q_full), c * 64, d.kvh * G, d.t0 + d.j0 + x * QT);
          }
          ++q_issued;
        }
        int32_t ids = -1;
        for (int j = 0; j < d.n_tiles; ++j, ++gt) {
          const int jj = d.jb + j;  // key tile
          if ((j & 3) == 0) {  // block ids of the next 4 tiles, one 16-key box per lane
            const int key = (jj * (kBN / kSub) + lane) * kSub;
            ids = (key < d.kv_end) ? __ldg(bt + key / p.block_size) : -1;
          }
          // lane b < 8: box b of the tile -- loaded or not, and its first row
          const int b = lane & 7;
          const int32_t id = __shfl_sync(kFullMask, ids, (j & 3) * (kBN / kSub) + b);
          const int key = jj * kBN + b * kSub;
          const bool in_range = lane < 8 && key < d.kv_end;
          const bool good = in_range && id >= 0 && id < p.num_blocks;
          bad_block |= in_range && !good;
          const uint32_t load = __ballot_sync(kFullMask, good);
          const uint32_t zero = vrole ? 0u : __ballot_sync(kFullMask, in_range && !good);
          const int32_t row = good ? half_rows + id * p.block_size + key % p.block_size : 0;
          const int st = gt % kNS;
          uint64_t* empty = vrole ? &bars->v_empty[st] : &bars->k_empty[st];
          uint64_t* full = vrole ? &bars->v_landed[st] : &bars->k_full[st];
          int w = 1;
          if (lane == 0 && gt >= kNS)
            w = mbar_wait(smem_addr(empty), ((gt / kNS) - 1) & 1, p.status, abort);
          ok = __shfl_sync(kFullMask, w, 0) != 0;
          if (!ok) break;
          const uint32_t dst0 = ring + st * Lay::TILE_BYTES;
          if (zero) {  // K rows of a bad page read as zeros
            fence_proxy_async_smem();
            constexpr int UNITS = Lay::NCH * kSub * 8;  // 16-byte units of one box
            for (int i = lane; i < (kBN / kSub) * UNITS; i += 32) {
              const int bx = i / UNITS, u = i % UNITS;
              if ((zero >> bx) & 1)
                st_shared_zero16(dst0 + (u / (kSub * 8)) * Lay::CH_BYTES + bx * kSub * 128 +
                                 (u % (kSub * 8)) * 16);
            }
            fence_proxy_async_smem();
          }
          if (vrole && lane == 0) *reinterpret_cast<volatile uint32_t*>(&bars->v_mask[st]) = load;
          __syncwarp();
          if (lane == 0)
            mbar_arrive_expect_tx(smem_addr(full), __popc(load) * Lay::NCH * kSub * 128);
#pragma unroll
          for (int bb = 0; bb < kBN / kSub; ++bb) {
            const int32_t r = __shfl_sync(kFullMask, row, bb);
            if (lane == 0 && ((load >> bb) & 1))
              for (int c = 0; c < Lay::NCH; ++c)
                tma_load_4d(dst0 + c * Lay::CH_BYTES + bb * kSub * 128, &kv_map, smem_addr(full), 0,
                            r, d.kvh, c);
          }
          armed = gt + 1;
        }
        if (!ok) break;
      }
      if (bad_block) set_status(p.status, PKV_DEV_BAD_BLOCK);
      // our copies, and the barrier arrivals they trigger, land before the CTA can exit
      if (lane == 0) {
        uint64_t* landed = vrole ? bars->v_landed : bars->k_full;
        for (int g = max(0, armed - kNS); g < armed; ++g)
          mbar_wait(smem_addr(&landed[g % kNS]), (g / kNS) & 1, nullptr);
        if (!vrole && q_issued > 0)
          mbar_wait(smem_addr(&bars->q_full), (q_issued - 1) & 1, nullptr);
      }
    } else if (warp != kMmaWarp && warp != kMmaWarp + 1) {
      // ===== converters (warps 8-11, one per SM sub-partition): each landed
      // V stage to fp16 in place =====
      // piece i of a stage (row i / RP, 16-byte column unit i % RP) is
      // converted by converter thread i mod 128 (rows not loaded, or past
      // the needed keys, are zeroed); the stage is then published to the
      // tensor core's (async) proxy
      constexpr int RP = D / 8;
      const int ct = converter_slot(warp) * 32 + lane;
      uint32_t emax = 0;  // V exponent fields seen (range check)
      int gt = 0;
      bool ok = true;
      for (int gi = 0; ok; ++gi) {
        int it = -1;
        if (lane == 0) it = read_item(bars, p, gi, abort);
        it = __shfl_sync(kFullMask, it, 0);
        if (it < 0) break;
        const PrefillItem d = prefill_item(p, wl, QP, it);
        for (int j = 0; j < d.n_tiles; ++j, ++gt) {
          const int st = gt % kNS;
          int w = 1;
          if (lane == 0)
            w = mbar_wait(smem_addr(&bars->v_landed[st]), (gt / kNS) & 1, p.status, abort);
          ok = __shfl_sync(kFullMask, w, 0) != 0;
          if (!ok) break;
          const uint32_t base = v_s + st * Lay::TILE_BYTES;
          const uint32_t load = *reinterpret_cast<volatile uint32_t*>(&bars->v_mask[st]);
          const int nvalid = d.kv_end - (d.jb + j) * kBN;  // rows below it are needed keys
#pragma unroll 4
          for (int i = ct; i < kBN * RP; i += kConverters) {
            const int k = i / RP, pc = i % RP;
            const uint32_t a = base + (pc >> 3) * Lay::CH_BYTES + k * 128 +
                               (((uint32_t)(pc & 7) ^ (uint32_t)(k & 7)) << 4);
            if (k < nvalid && ((load >> (k / kSub)) & 1u))
              v_piece_to_f16(a, emax);
            else
              st_shared_zero16(a);
          }
          fence_proxy_async_smem();
          mbar_arrive(smem_addr(&bars->v_full[st]));
        }
      }
      // a bf16 exponent field >= 143 is a magnitude >= 2^16 (or inf / NaN)
      if ((emax & 0xffffu) >= 0x4780u || (emax >> 16) >= 0x4780u)
        set_status(p.status, PKV_DEV_V_RANGE);
    } else if (lane == 0) {
      // ============ MMA issuers: one thread of warp 12 for Q tile A, one of
      // warp 13 for Q tile B ============
      // Each issues its own tile's products in order over S tiles of kSN
      // keys (the halves of the K/V tiles): QK(0) and QK(1) into the two S
      // buffers, then for every S tile j: PV(j), QK(j+2). S tile j+1 is
      // thus computed while the softmax works on j, and the softmax
      // warpgroup goes from one tile to the next without waiting for the
      // tensor core. A buffer holds P(j) until PV(j) has read it; tcgen05
      // operations of one thread run in issue order, so QK(j+2) into the
      // same buffer may follow PV(j) at once. The two threads' MMAs
      // interleave on the tensor core. A K or V stage is released when both
      // threads' products that read it are done (two commits); so is Q.
      // Descriptors and barrier addresses are computed once; an operand
      // offset only adds to the start-address field (16-byte units).
      const int x = warp - kMmaWarp;
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kBM, kSN, false, false);
      constexpr uint32_t idesc_pv = umma_idesc_f16(kBM, D, false, true);
      const uint64_t qd = smem_desc_sw128(q_s + x * Lay::TILE_BYTES, 16, 1024);
      uint64_t kdesc[kNS], vdesc[kNS];
      uint32_t k_empty_b[kNS], v_empty_b[kNS];
#pragma unroll
      for (int st = 0; st < kNS; ++st) {
        kdesc[st] = smem_desc_sw128(k_s + st * Lay::TILE_BYTES, 16, 1024);
        vdesc[st] = smem_desc_sw128(v_s + st * Lay::TILE_BYTES, Lay::CH_BYTES, 1024);
        k_empty_b[st] = smem_addr(&bars->k_empty[st]);
        v_empty_b[st] = smem_addr(&bars->v_empty[st]);
      }
      static_assert(kNS == 2 && kSB == 2 && kBN == 2 * kSN, "two-way selects below");
      const uint32_t s_full_b[kSB] = {smem_addr(&bars->s_full[x][0]),
                                      smem_addr(&bars->s_full[x][1])};
      const uint32_t o_done_b[2] = {smem_addr(&bars->o_done[x][0]),
                                    smem_addr(&bars->o_done[x][1])};
      const uint32_t s_tmem = tmem + Lay::s_col(x, 0);
      const uint32_t o_tmem = tmem + Lay::o_col(x);
      constexpr uint32_t kHalf16 = (kSN * 128) >> 4;  // rows of half a K/V tile, in 16-byte units
      // S(g) = Q_x K^T over half h of K/V tile kt; `rel`: the last S tile
      // that reads the K stage
      auto issue_qk = [&](int g, int kt, int h, bool rel) {
        tc_fence_after();
        const uint32_t d_tmem = s_tmem + (uint32_t)((g & 1) * kSN);
        const uint64_t kd = ((kt & 1) ? kdesc[1] : kdesc[0]) + (h ? kHalf16 : 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off16 = ((kk >> 2) * Lay::CH_BYTES + (kk & 3) * 32) >> 4;
          umma_ss(d_tmem, qd + off16, kd + off16, idesc_qk, kk > 0);
        }
        if (rel) umma_commit((kt & 1) ? k_empty_b[1] : k_empty_b[0]);
        umma_commit((g & 1) ? s_full_b[1] : s_full_b[0]);
      };
      // O_x += P(g) V over half h of K/V tile kt (fp16 P and V; the
      // converters fenced their V writes to the async proxy before
      // publishing the stage)
      auto issue_pv = [&](int g, int kt, int h, bool first, bool rel) {
        tc_fence_after();
        const uint32_t p_tmem = s_tmem + (uint32_t)((g & 1) * kSN);
        const uint64_t vd = ((kt & 1) ? vdesc[1] : vdesc[0]) + (h ? kHalf16 : 0u);
#pragma unroll
        for (int kk = 0; kk < kSN / 16; ++kk)
          umma_ts(o_tmem, p_tmem + Lay::p_col(kk), vd + (uint32_t)((kk * 16 * 128) >> 4), idesc_pv,
                  (!first || kk > 0) ? 1u : 0u);
        if (rel) umma_commit((kt & 1) ? v_empty_b[1] : v_empty_b[0]);
        umma_commit((g & 1) ? o_done_b[1] : o_done_b[0]);
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return mbar_wait(smem_addr(bar), parity, p.status, abort);
      };
      bool ok = true;
      int gi = 0, gt = 0, gs = 0;  // items, K/V tiles, S tiles so far
      for (; ok; ++gi) {
        const int it = read_item(bars, p, gi, abort);
        if (it < 0) break;
        const PrefillItem d = prefill_item(p, wl, QP, it);
        const int ns = d.n_sub;
        // both S buffers are free: the previous item's PVs were issued first
        ok = wait(&bars->q_full, gi & 1) && wait(&bars->k_full[gt % kNS], (gt / kNS) & 1);
        if (!ok) break;
        issue_qk(gs, gt, 0, ns == 1);
        if (ns > 1) issue_qk(gs + 1, gt, 1, true);
        if (ns <= 2) umma_commit(smem_addr(&bars->q_empty));  // Q of this item no longer read
        for (int j = 0; ok && j < ns; ++j) {
          const int g = gs + j, kt = gt + (j >> 1), h = j & 1;
          // the first PV of an item overwrites O_x: the previous item's
          // epilogue must have read it
          ok = wait(&bars->p_ready[x][g & 1], (g >> 1) & 1) &&
               (h || wait(&bars->v_full[kt % kNS], (kt / kNS) & 1)) &&
               (j > 0 || gi == 0 || wait(&bars->o_free[x], (gi - 1) & 1));
          if (!ok) break;
          issue_pv(g, kt, h, j == 0, h || j == ns - 1);
          if (j + 2 < ns) {
            const int kt2 = gt + ((j + 2) >> 1);
            ok = h || wait(&bars->k_full[kt2 % kNS], (kt2 / kNS) & 1);
            if (!ok) break;
            issue_qk(g + 2, kt2, h, h || j + 2 == ns - 1);
            if (j + 2 == ns - 1) umma_commit(smem_addr(&bars->q_empty));
          }
        }
        gt += d.n_tiles;
        gs += ns;
      }
      // every MMA issued so far (by both threads) has completed before TMEM
      // is released
      umma_commit(smem_addr(&bars->mma_done));
      mbar_wait(smem_addr(&bars->mma_done), 0, nullptr);
    }
  } else {
    setmaxnreg_inc<kSoftmaxRegs>();
    // ====== softmax + epilogue: warpgroup x owns Q tile x, thread r owns row r ======
    const int x = warp >> 2;
    const int r = threadIdx.x & (kBM - 1);
    const int rq = r / G;  // query of the row inside its tile
    const int g = r % G;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t sa0 = tmem + lane_base + Lay::s_col(x, 0);
    const uint32_t oa = tmem + lane_base + Lay::o_col(x);
    const float sl2 = p.scale_log2;
    const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
    bool ok = true;
    int gs = 0;  // S tiles of this Q tile so far (all items)
    for (int k = 0; ok; ++k) {
      int it = -1;
      if (lane == 0) it = read_item(bars, p, k, abort);
      it = __shfl_sync(kFullMask, it, 0);
      if (it < 0) break;
      const PrefillItem d = prefill_item(p, wl, QP, it);
      const int qj = d.j0 + x * QT + rq;
      const bool row_valid = qj < d.j1;
      // the row's last visible key (a key range may end before the query)
      const int pos =
          (row_valid && !p.prefix_mode) ? min(d.qpos0 + qj, d.kv_end - 1) : (d.kv_end - 1);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < d.n_sub; ++j) {
        const int gg = gs + j;
        const uint32_t sa = sa0 + (uint32_t)((gg & 1) * kSN);
        ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->s_full[x][gg & 1]), (gg >> 1) & 1,
                                             p.status, abort));
        if (!ok) break;
        tc_fence_after();
        const int lim = pos - (d.jb * kBN + j * kSN);  // keys c <= lim of this tile are visible
        // the row's kSN scores in registers: one TMEM round trip
        uint32_t u[kSN];
        PKV_TMEM_LD32(sa, u);
        PKV_TMEM_LD32(sa + 32, (u + 32));
        tmem_wait_ld();
        float alpha = 1.f, rsa = 0.f, rsb = 0.f;
        bool resc;
        if (__all_sync(kFullMask, lim >= kSN - 1)) {
          // ---- every key of the tile is visible to every row of the warp:
          // row maximum (two independent chains of 3-input maxima), then the
          // probabilities as fp16 pairs, written over the first half of the
          // S columns; the row sum adds the rounded values, so that O and l
          // see the same weights
          float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
          for (int c = 0; c < kSN / 2; c += 2) {
            mxa = max3(mxa, __uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1]));
            mxb = max3(mxb, __uint_as_float(u[2 * c + 2]), __uint_as_float(u[2 * c + 3]));
          }
          const float mnew = fmaxf(m, fmaxf(mxa, mxb) * sl2);
          resc = mnew > m + kRescaleThreshold;
          if (resc) {
            alpha = fast_exp2(m - mnew);  // 0 on the first tile
            m = mnew;
          }
          const float2 sl2x2 = make_float2(sl2, sl2);
          const float2 negm = make_float2(-m, -m);
#pragma unroll
          for (int ch = 0; ch < kSN / 32; ++ch) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float2 x2 = __ffma2_rn(make_float2(__uint_as_float(u[32 * ch + 2 * c]),
                                                       __uint_as_float(u[32 * ch + 2 * c + 1])),
                                           sl2x2, negm);
              pk[c] = pack_f16x2(fast_exp2(x2.x), fast_exp2(x2.y));
              add_f16x2_to(rsa, rsb, pk[c]);
            }
            PKV_TMEM_ST16(sa + ch * 16, pk);
          }
        } else {
          // ---- a diagonal tile: hide the keys after each row's position
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < kSN; ++c)
            if (c <= lim) mx = fmaxf(mx, __uint_as_float(u[c]));
          const float mnew = fmaxf(m, mx * sl2);
          resc = mnew > m + kRescaleThreshold;
          if (resc) {
            alpha = fast_exp2(m - mnew);  // 0 on the first tile
            m = mnew;
          }
#pragma unroll
          for (int ch = 0; ch < kSN / 32; ++ch) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int c0 = 32 * ch + 2 * c;
              float p0 = fast_exp2(fmaf(__uint_as_float(u[c0]), sl2, -m));
              float p1 = fast_exp2(fmaf(__uint_as_float(u[c0 + 1]), sl2, -m));
              if (c0 > lim) p0 = 0.f;
              if (c0 + 1 > lim) p1 = 0.f;
              pk[c] = pack_f16x2(p0, p1);
              add_f16x2_to(rsa, rsb, pk[c]);
            }
            PKV_TMEM_ST16(sa + ch * 16, pk);
          }
        }
        tmem_wait_st();
        l = l * alpha + (rsa + rsb);
        if (j > 0 && __any_sync(kFullMask, resc)) {
          // O_x is rescaled once the previous tile's PV has finished writing it
          ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->o_done[x][(gg - 1) & 1]),
                                               ((gg - 1) >> 1) & 1, p.status, abort));
          if (!ok) break;
          tc_fence_after();
          {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              PKV_TMEM_LD32(oa + 32 * c, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
              PKV_TMEM_ST32(oa + 32 * c, v);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        __syncwarp();  // the warp's P (and O) stores precede its one arrival
#ifdef PKV_TEST_HOLD_ARRIVAL
        if (g_pkv_test_hold_prefill && blockIdx.x == 0 && warp == 0 && gg == 0) continue;
#endif
        if (lane == 0) mbar_arrive(smem_addr(&bars->p_ready[x][gg & 1]));
      }
      if (!ok) break;
      // ---- epilogue of the item: O / l -> out, lse
      const int last = gs + d.n_sub - 1;
      ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->o_done[x][last & 1]),
                                           (last >> 1) & 1, p.status, abort));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* orow = p.out + d.seg * p.split_out_stride +
                    ((int64_t)(d.t0 + qj) * p.num_heads + d.kvh * G + g) * D;
      // each thread writes its own row: 32-byte stores (whole sectors) when
      // `out` allows them (row offsets are multiples of 32 bytes), else 16-byte
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        PKV_TMEM_LD32(oa + 32 * c, u);
        tmem_wait_ld();
        if (row_valid) {
          if (out32) {
#pragma unroll
            for (int e = 0; e < 32; e += 8)
              st_global_v8(orow + 32 * c + e, __uint_as_float(u[e]) * inv,
                           __uint_as_float(u[e + 1]) * inv, __uint_as_float(u[e + 2]) * inv,
                           __uint_as_float(u[e + 3]) * inv, __uint_as_float(u[e + 4]) * inv,
                           __uint_as_float(u[e + 5]) * inv, __uint_as_float(u[e + 6]) * inv,
                           __uint_as_float(u[e + 7]) * inv);
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(orow + 32 * c + e) =
                  make_float4(__uint_as_float(u[e]) * inv, __uint_as_float(u[e + 1]) * inv,
                              __uint_as_float(u[e + 2]) * inv, __uint_as_float(u[e + 3]) * inv);
          }
        }
      }
      if (row_valid && p.out_lse)
        p.out_lse[d.seg * p.split_lse_stride + (int64_t)(d.t0 + qj) * p.num_heads + d.kvh * G + g] =
            (m + fast_log2(l)) * kLn2;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bars->o_free[x]));  // the MMA may overwrite O_x now
      gs += d.n_sub;
    }
  }

  // ---- teardown: all tcgen05 work of the CTA is complete; release TMEM
  // (its address read again from shared memory: the roles ran with
  // different register budgets)
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == kMmaWarp) {
    const Bars* b = reinterpret_cast<const Bars*>(
        ((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023)) +
        Lay::BAR_OFF);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(*reinterpret_cast<const volatile uint32_t*>(&b->tmem_base), kTmemCols);
  }
  if (threadIdx.x == 0) cta_finished(p);
}

template <int D>
cudaError_t launch_prefill_d(const AttnParams& p, const CUtensorMap& q_map,
                             const CUtensorMap& kv_map, cudaStream_t stream) {
  using Lay = PrefillLayout<D>;
  const size_t smem = Lay::bytes(p.num_seqs);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kernel = prefill_kernel<D>;
  static SmemLimit limit;
  if (cudaError_t e = limit.ensure(reinterpret_cast<const void*>(kernel), 227 * 1024);
      e != cudaSuccess)
    return e;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int G = p.num_heads / p.num_kv_heads;
  const int QP = kQT * (kBM / G);
  const int64_t bound = (int64_t)p.num_seqs * ((p.max_query_len + QP - 1) / QP) * p.num_kv_heads *
                        (p.prefix_mode ? p.kv_splits : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(bound < sms ? bound : sms));  // one CTA per SM (TMEM, smem)
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, q_map, kv_map, p);
}

}  // namespace

bool prefill_fits(int32_t num_seqs, int32_t head_dim) {
  if (num_seqs < 0) return false;
  if (head_dim == 128) return PrefillLayout<128>::bytes(num_seqs) <= 227 * 1024;
  if (head_dim == 64) return PrefillLayout<64>::bytes(num_seqs) <= 227 * 1024;
  return false;
}

cudaError_t launch_prefill(const AttnParams& p, const CUtensorMap& q_map,
                           const CUtensorMap& kv_map, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_prefill_d<128>(p, q_map, kv_map, stream);
  if (p.head_dim == 64) return launch_prefill_d<64>(p, q_map, kv_map, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
