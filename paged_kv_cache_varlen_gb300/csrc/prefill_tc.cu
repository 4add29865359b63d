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
//   * persistent CTAs, one per SM: every CTA builds the per-request prefix
//     sum of work items in shared memory and takes items dynamically from a
//     global ticket counter in the workspace (the busiest SM had 1.6x the
//     mean work under a static round-robin); an item is (request, KV head,
//     two consecutive query tiles A and B of 128/G queries each), later
//     items (more keys) first. Tensor memory and barriers are set up once per CTA;
//     requests short enough for the decode kernel (1 .. decode_max_q
//     queries) give no items here;
//   * a Q tile is 128 rows = (128/G queries) x (G heads sharing the KV head),
//     so one pass over the K/V pages serves the whole GQA group, and both Q
//     tiles of the item share every K/V tile loaded: the gather from L2 (the
//     bound of this kernel, ~12 B/cycle per SM) is paid once per two tiles;
//   * Q arrives by TMA ({64, G, 128/G} boxes, 128-byte swizzle). K and V
//     tiles of 128 keys are gathered page by page (block ids from
//     block_table) by two producer warps with 16-byte cp.async copies
//     written straight into the 128-byte-swizzled layout the MMA descriptors
//     read (keys past the needed range are zero-filled), in separate 2-stage
//     rings. (Paged 16-key TMA boxes were slower: ~200 cycles per 2 KB box
//     per SM);
//   * S = Q K^T (M=128, N=128, K=head_dim) and O += P V (M=128, N=head_dim,
//     K=128) run as tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) issued
//     by one thread. Tensor memory holds S_A, S_B, O_A, O_B (4 x 128
//     columns); P is written back in place over the S columns it came from,
//     as a bf16 high part and a bf16 remainder (P ~= hi + lo to ~2^-16
//     relative; O accumulates hi*V + lo*V -- a single bf16 rounding of P puts
//     few-key rows up to ~4e-3 off the exact result); P is the A operand
//     straight from TMEM;
//   * two softmax warpgroups, one per Q tile; thread r of a warpgroup owns
//     TMEM lane (= Q row) r: pass 1 reads S in 32-column pieces for the row
//     maximum, pass 2 re-reads them, applies the causal mask and the
//     exp2-domain online softmax (lazy rescale when the maximum grows by more
//     than 8) and stores P; O is rescaled in TMEM when needed. While one
//     warpgroup computes its softmax, the tensor core works on the other
//     tile's products (ping-pong);
//   * warps 8-9 produce loads, warp 10 issues the MMAs in a fixed order that
//     alternates the two Q tiles (PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1)),
//     so one tile's softmax overlaps the other tile's products;
//   * the softmax of a tile every key of which is visible to the warp's rows
//     skips the mask and uses packed fp32x2 arithmetic; P's bf16 high part
//     and remainder are cut by bit operations (truncation: hi + lo is p to
//     2^-14 relative) instead of conversions;
//   * every wait is bounded; on a timeout the CTA drains its copies and
//     MMAs, frees its TMEM and leaves with PKV_DEV_TIMEOUT set.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kBM = 128;                             // Q rows per tile
constexpr int kQT = 2;                               // Q tiles per work item
constexpr int kBN = 128;                             // keys per KV tile
constexpr int kNS = 2;                               // stages of each of the K and V rings
constexpr int kSub = 16;                             // keys per gathered sub-block
constexpr int kSoftmaxThreads = kQT * kBM;           // warps 0 .. 4*kQT-1
constexpr int kProducers = 64;                       // two K/V producer warps
constexpr int kProdWarp0 = kSoftmaxThreads / 32;     // first producer warp (also issues Q)
constexpr int kMmaWarp = kProdWarp0 + kProducers / 32;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kRing = 4;  // work items announced ahead of the roles that consume them
// readers of an announced item: the second producer warp, the MMA thread and
// the eight softmax warps (one lane each)
constexpr int kItemReaders = 1 + 1 + kSoftmaxThreads / 32;
constexpr float kRescaleThreshold = 8.f;
constexpr uint32_t kFullMask = 0xffffffffu;

template <int D>
struct PrefillLayout {
  static constexpr int NCH = D / 64;                       // 128-byte column chunks of a row
  static constexpr int CH_BYTES = 128 * 128;               // one chunk of 128 rows
  static constexpr int TILE_BYTES = NCH * CH_BYTES;        // one Q, K or V tile
  static constexpr int Q_OFF = 0;                          // [kQT] Q tiles of the item
  static constexpr int K_OFF = Q_OFF + kQT * TILE_BYTES;   // [kNS] K tiles
  static constexpr int V_OFF = K_OFF + kNS * TILE_BYTES;   // [kNS] V tiles
  static constexpr int BAR_OFF = V_OFF + kNS * TILE_BYTES;
  static constexpr int PREF_OFF = BAR_OFF + 512;
  // keep one CTA per SM (each CTA allocates all 512 TMEM columns)
  static size_t bytes(int num_seqs) {
    const size_t need = 1024 + PREF_OFF + (size_t)(num_seqs + 1) * 4;
    return need > 120 * 1024 ? need : 120 * 1024;
  }
  // TMEM columns: S of tile x (P written in place), then O of tile x
  __device__ static constexpr uint32_t s_col(int x) { return 128u * (uint32_t)x; }
  __device__ static constexpr uint32_t o_col(int x) { return 128u * (uint32_t)(kQT + x); }
  // P of keys 16*kk .. 16*kk+15 inside an S buffer: each 32-key piece holds
  // 16 columns of packed hi then 16 columns of packed lo
  __device__ static constexpr uint32_t p_hi_col(int kk) {
    return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8);
  }
};
static_assert(kQT * 2 * 128 <= (int)kTmemCols, "S and O of every Q tile fit in TMEM");

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kNS], k_empty[kNS];
  uint64_t v_full[kNS], v_empty[kNS];
  uint64_t s_full[kQT];   // QK^T of the tile landed in S_x
  uint64_t p_ready[kQT];  // the warpgroup stored P_x (and rescaled O_x)
  uint64_t o_done[kQT];   // PV of the tile finished (S_x free, O_x stable)
  uint64_t o_free[kQT];   // the warpgroup's epilogue has read O_x
  uint64_t mma_done;
  uint64_t item_full[kRing], item_empty[kRing];
  int32_t item_id[kRing];  // work item taken from the global ticket counter, -1: none left
  uint32_t tmem_base;
  int32_t abort;
  int32_t scan[kThreads / 32];
};

struct PrefillItem {
  int req, kvh, j0, j1, t0, qlen, L, kv_end, n_tiles;
  int qpos0;  // position of the request's first query among its keys
  int jb;   // first key tile of the item (a key segment in prefix mode)
  int seg;  // key segment (prefix mode), else 0
};

// Prefix mode: the keys of a prefix of L tokens are cut into segments of
// tiles_per_segment tiles; segment_count of them are non-empty.
__device__ __forceinline__ int prefix_tiles_per_segment(int L, int splits) {
  const int t = (L + kBN - 1) / kBN;
  return (t + splits - 1) / splits;
}
__device__ __forceinline__ int prefix_segment_count(int L, int splits) {
  const int t = (L + kBN - 1) / kBN;
  const int tps = prefix_tiles_per_segment(L, splits);
  return tps > 0 ? (t + tps - 1) / tps : 0;
}

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
  if (qlen <= p.decode_max_q) return 0;  // short requests run on the decode kernel
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

// pref[r] = work units of requests before r; pref[B] = total. All threads.
__device__ __forceinline__ int prefill_prefix(const AttnParams& p, int* pref, int32_t* scan,
                                              int QP) {
  const int B = p.num_seqs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool flag = blockIdx.x == 0;
  const int per = (B + kThreads - 1) / kThreads;
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  int sum = 0;
  for (int r = r0; r < r1; ++r) sum += prefill_units(p, r, QP, flag);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += scan[w];
  int run = base + incl - sum;
  for (int r = r0; r < r1; ++r) {
    pref[r] = run;
    run += prefill_units(p, r, QP, false);
  }
  if (tid == kThreads - 1) pref[B] = run;
  __syncthreads();
  return pref[B];
}

__device__ __forceinline__ PrefillItem prefill_item(const AttnParams& p, const int* pref, int QP,
                                                    int it) {
  PrefillItem d;
  const int u = it / p.num_kv_heads;
  d.kvh = it - u * p.num_kv_heads;
  int lo = 0, hi = p.num_seqs;  // largest lo with pref[lo] <= u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= u)
      lo = mid;
    else
      hi = mid;
  }
  d.req = lo;
  d.t0 = __ldg(p.cu_seqlens + lo);
  d.qlen = __ldg(p.cu_seqlens + lo + 1) - d.t0;
  d.L = __ldg(p.seq_lens + lo);
  const int ntq = (d.qlen + QP - 1) / QP;
  d.qpos0 = d.L - d.qlen;
  if (p.prefix_mode) {
    const int segs = prefix_segment_count(d.L, p.kv_splits);
    const int tps = prefix_tiles_per_segment(d.L, p.kv_splits);
    const int local = u - pref[lo];
    d.seg = local % segs;
    d.j0 = (local / segs) * QP;
    d.j1 = min(d.qlen, d.j0 + QP);
    d.kv_end = d.L;  // every query sees the whole prefix
    d.jb = d.seg * tps;
    d.n_tiles = min((d.L + kBN - 1) / kBN, d.jb + tps) - d.jb;
    return d;
  }
  const int qt = ntq - 1 - (u - pref[lo]);  // later (heavier) units first
  d.j0 = qt * QP;
  d.j1 = min(d.qlen, d.j0 + QP);
  if (p.key_start) {  // key range: the queries' positions come from the caller
    const int64_t rel = (int64_t)__ldg(p.query_start + lo) - __ldg(p.key_start + lo);
    d.qpos0 = (int)max((int64_t)-(1 << 30), min((int64_t)(1 << 30), rel));
  }
  // keys [0, kv_end) are needed; at least one tile runs (fully masked when no
  // key is visible) so that the item's rows are written
  d.kv_end = max(0, min(d.L, d.qpos0 + d.j1));
  d.n_tiles = max(1, (d.kv_end + kBN - 1) / kBN);
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
    prefill_kernel(const __grid_constant__ CUtensorMap q_map, const AttnParams p) {
  using Lay = PrefillLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + Lay::BAR_OFF);
  int* pref = reinterpret_cast<int*>(smem + Lay::PREF_OFF);

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
    mbar_init(smem_addr(&bars->q_empty), 1);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(smem_addr(&bars->k_full[s]), kProducers);
      mbar_init(smem_addr(&bars->k_empty[s]), 1);
      mbar_init(smem_addr(&bars->v_full[s]), kProducers);
      mbar_init(smem_addr(&bars->v_empty[s]), 1);
    }
    for (int x = 0; x < kQT; ++x) {
      mbar_init(smem_addr(&bars->s_full[x]), 1);
      mbar_init(smem_addr(&bars->p_ready[x]), kBM / 32);  // one arrival per softmax warp
      mbar_init(smem_addr(&bars->o_done[x]), 1);
      mbar_init(smem_addr(&bars->o_free[x]), kBM / 32);
    }
    mbar_init(smem_addr(&bars->mma_done), 1);
    for (int k = 0; k < kRing; ++k) {
      mbar_init(smem_addr(&bars->item_full[k]), 1);
      mbar_init(smem_addr(&bars->item_empty[k]), kItemReaders);
    }
    bars->abort = 0;
    fence_barrier_init();
  }
  const int total = prefill_prefix(p, pref, bars->scan, QP) * p.num_kv_heads;  // syncs
  if ((int)blockIdx.x >= total) {  // uniform; nothing allocated yet
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

  if (warp >= kProdWarp0 && warp < kMmaWarp) {
    // ===== producers: Q by TMA (one thread), K/V by cp.async (64 threads) =====
    // Thread pt copies 16-byte piece pc of the rows of keys pk0, pk0 + KSTEP,
    // ... of every tile into the 128-byte-swizzled layout the MMA descriptors
    // expect (the piece at column unit u of row r lands at unit u ^ (r & 7)).
    // Keys past the needed range and rows of bad blocks are filled with
    // zeros (so V rows there never poison O: P is 0 there, 0 * NaN is not).
    constexpr int RP = D / 8;               // 16-byte pieces per K or V row
    constexpr int KSTEP = kProducers / RP;  // keys per round
    constexpr int NIT = kBN / KSTEP;        // rounds per tile
    static_assert(kSub % KSTEP == 0, "a round stays inside one 16-key sub-block");
    const int pt = threadIdx.x - kSoftmaxThreads;
    const int pc = pt % RP;
    const int pk0 = pt / RP;
    const uint32_t col_off = (uint32_t)((pc >> 3) * Lay::CH_BYTES);
    const uint32_t pcc = (uint32_t)(pc & 7);
    const int64_t row_bytes = (int64_t)p.num_kv_heads * D * 2;
    const uint8_t* pool = static_cast<const uint8_t*>(p.kv_pool);
    const int64_t v_half = (int64_t)p.num_blocks * p.block_size * row_bytes;
    const bool qlead = pt == 0;
    if (qlead) prefetch_tmap(&q_map);
    int gi = 0, gt = 0, armed = 0, q_issued = 0;
    bool ok = true, bad_block = false;
    for (;; ++gi) {
      int it = -1;
      if (lane == 0)
        it = warp == kProdWarp0 ? take_item(bars, p, total, gi, abort)
                                : read_item(bars, p, gi, abort);
      it = __shfl_sync(kFullMask, it, 0);
      if (it < 0) break;
      const PrefillItem d = prefill_item(p, pref, QP, it);
      const int32_t* bt = p.block_table + (int64_t)d.req * p.max_blocks;
      if (warp == kProdWarp0) {
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
      const int64_t head_off = (int64_t)d.kvh * D * 2 + pc * 16;
      int32_t ids = -1;
      for (int j = 0; j < d.n_tiles; ++j, ++gt) {
        const int jj = d.jb + j;  // key tile
        if ((j & 3) == 0) {  // block ids of the next 4 tiles, one 16-key sub-block per lane
          const int key = (jj * (kBN / kSub) + lane) * kSub;
          ids = (key < d.kv_end) ? __ldg(bt + key / p.block_size) : -1;
        }
        // byte offset in the K half of the pool of each sub-block's first row
        // for this thread's piece, or -1 (zero fill)
        int64_t sub_off[kBN / kSub];
#pragma unroll
        for (int sb = 0; sb < kBN / kSub; ++sb) {
          const int32_t id = __shfl_sync(kFullMask, ids, (j & 3) * (kBN / kSub) + sb);
          const int key = jj * kBN + sb * kSub;
          sub_off[sb] = -1;
          if (key < d.kv_end) {
            if (id < 0 || id >= p.num_blocks)
              bad_block = true;
            else
              sub_off[sb] = ((int64_t)id * p.block_size + key % p.block_size) * row_bytes + head_off;
          }
        }
        const int st = gt % kNS;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint64_t* empty = half ? &bars->v_empty[st] : &bars->k_empty[st];
          uint64_t* full = half ? &bars->v_full[st] : &bars->k_full[st];
          int w = 1;
          if (lane == 0 && gt >= kNS)
            w = mbar_wait(smem_addr(empty), ((gt / kNS) - 1) & 1, p.status, abort);
          ok = __shfl_sync(kFullMask, w, 0) != 0;
          if (!ok) break;
          fence_proxy_async_smem();  // the MMAs' reads of this stage precede our writes
          const uint32_t dst0 = (half ? v_s : k_s) + st * Lay::TILE_BYTES + col_off;
          const int64_t base = half ? v_half : 0;
#pragma unroll
          for (int i = 0; i < NIT; ++i) {
            const int k = pk0 + KSTEP * i;
            const int sb = (KSTEP * i) / kSub;
            const bool valid = sub_off[sb] >= 0 && jj * kBN + k < d.kv_end;
            const uint8_t* src =
                valid ? pool + base + sub_off[sb] + (int64_t)(k % kSub) * row_bytes : pool;
            cp_async_16(dst0 + k * 128 + ((pcc ^ (uint32_t)(k & 7)) << 4), src, valid ? 16u : 0u);
          }
          cp_async_arrive_noinc(smem_addr(full));
        }
        if (!ok) break;
        armed = gt + 1;
      }
    }
    if (bad_block) set_status(p.status, PKV_DEV_BAD_BLOCK);
    // our copies, and the barrier arrivals they trigger, land before the CTA can exit
    cp_async_wait_all();
    if (lane == 0) {
      for (int g = max(0, armed - kNS); g < armed; ++g) {
        mbar_wait(smem_addr(&bars->k_full[g % kNS]), (g / kNS) & 1, nullptr);
        mbar_wait(smem_addr(&bars->v_full[g % kNS]), (g / kNS) & 1, nullptr);
      }
      if (warp == kProdWarp0 && q_issued > 0)
        mbar_wait(smem_addr(&bars->q_full), (q_issued - 1) & 1, nullptr);
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA issuer (one thread) =================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kBM, D, false, true);
      bool ok = true;
      int gi = 0, gt = 0;
      // S_x = Q_x K_g^T (the K stage is released after the last Q tile's product)
      auto issue_qk = [&](int x, int g) {
        fence_proxy_async_smem();  // K was written by cp.async (generic proxy)
        tc_fence_after();
        const uint32_t d_tmem = tmem + Lay::s_col(x);
        const uint32_t qb = q_s + x * Lay::TILE_BYTES;
        const uint32_t kb = k_s + (g % kNS) * Lay::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Lay::CH_BYTES + (kk & 3) * 32;
          umma_ss(d_tmem, smem_desc_sw128(qb + off, 16, 1024),
                  smem_desc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0);
        }
        if (x == kQT - 1) umma_commit(smem_addr(&bars->k_empty[g % kNS]));
        umma_commit(smem_addr(&bars->s_full[x]));
      };
      // O_x += P_x V_g (P as bf16 high parts, then the remainders)
      auto issue_pv = [&](int x, int g, bool first) {
        fence_proxy_async_smem();  // V was written by cp.async (generic proxy)
        tc_fence_after();
        const uint32_t s_base = tmem + Lay::s_col(x);
        const uint32_t o_base = tmem + Lay::o_col(x);
        const uint32_t v_base = v_s + (g % kNS) * Lay::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t b = smem_desc_sw128(v_base + kk * 16 * 128, Lay::CH_BYTES, 1024);
          umma_ts(o_base, s_base + Lay::p_hi_col(kk), b, idesc_pv, (!first || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t b = smem_desc_sw128(v_base + kk * 16 * 128, Lay::CH_BYTES, 1024);
          umma_ts(o_base, s_base + Lay::p_hi_col(kk) + 16, b, idesc_pv, 1u);
        }
        if (x == kQT - 1) umma_commit(smem_addr(&bars->v_empty[g % kNS]));
        umma_commit(smem_addr(&bars->o_done[x]));
      };
      // Fixed issue order per item: QK_A(0), QK_B(0), then for every tile j
      // PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1). After the first tile this
      // puts the two warpgroups half a period apart: the softmax of one Q
      // tile runs while the tensor core works through the other tile's PV
      // and next QK^T, instead of both softmaxes running at once and the
      // tensor core idling meanwhile.
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return mbar_wait(smem_addr(bar), parity, p.status, abort);
      };
      for (; ok; ++gi) {
        const int it = read_item(bars, p, gi, abort);
        if (it < 0) break;
        const PrefillItem d = prefill_item(p, pref, QP, it);
        const int n = d.n_tiles;
        ok = wait(&bars->q_full, gi & 1) && wait(&bars->k_full[gt % kNS], (gt / kNS) & 1);
        // S_x is reused after PV of the previous item's last tile: in issue order
        for (int x = 0; ok && x < kQT; ++x) issue_qk(x, gt);
        if (!ok) break;
        if (n == 1) umma_commit(smem_addr(&bars->q_empty));  // Q of this item no longer read
        for (int j = 0; ok && j < n; ++j) {
          const int g = gt + j;
          for (int x = 0; ok && x < kQT; ++x) {
            // the first PV of an item overwrites O_x: the previous item's
            // epilogue must have read it
            ok = wait(&bars->p_ready[x], g & 1) &&
                 wait(&bars->v_full[g % kNS], (g / kNS) & 1) &&
                 (j > 0 || gi == 0 || wait(&bars->o_free[x], (gi - 1) & 1));
            if (!ok) break;
            issue_pv(x, g, j == 0);
            if (j + 1 < n) {
              // S_x holds P_x(j) until this PV has read it: tcgen05.mma
              // operations issued by one thread run in issue order, so the
              // next QK^T into S_x may follow the PV at once
              ok = wait(&bars->k_full[(g + 1) % kNS], ((g + 1) / kNS) & 1);
              if (!ok) break;
              issue_qk(x, g + 1);
              if (x == kQT - 1 && j + 2 == n) umma_commit(smem_addr(&bars->q_empty));
            }
          }
        }
        gt += n;
      }
      // every MMA issued so far has completed before TMEM is released
      umma_commit(smem_addr(&bars->mma_done));
      mbar_wait(smem_addr(&bars->mma_done), 0, nullptr);
    }
  } else {
    // ====== softmax + epilogue: warpgroup x owns Q tile x, thread r owns row r ======
    const int x = warp >> 2;
    const int r = threadIdx.x & (kBM - 1);
    const int rq = r / G;  // query of the row inside its tile
    const int g = r % G;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t sa = tmem + lane_base + Lay::s_col(x);
    const uint32_t oa = tmem + lane_base + Lay::o_col(x);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int gt = 0;
    for (int k = 0; ok; ++k) {
      int it = -1;
      if (lane == 0) it = read_item(bars, p, k, abort);
      it = __shfl_sync(kFullMask, it, 0);
      if (it < 0) break;
      const PrefillItem d = prefill_item(p, pref, QP, it);
      const int qj = d.j0 + x * QT + rq;
      const bool row_valid = qj < d.j1;
      // the row's last visible key (a key range may end before the query)
      const int pos =
          (row_valid && !p.prefix_mode) ? min(d.qpos0 + qj, d.kv_end - 1) : (d.kv_end - 1);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < d.n_tiles; ++j) {
        const int gg = gt + j;
        ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->s_full[x]), gg & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
        const int lim = pos - (d.jb + j) * kBN;  // keys c <= lim of this tile are visible
        float alpha = 1.f, rs;
        bool resc;
        if (__all_sync(kFullMask, lim >= kBN - 1)) {
          // ---- every key of the tile is visible to every row of the warp
          // pass 1: row maximum (four independent chains)
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
          for (int ch = 0; ch < kBN / 32; ++ch) {
            uint32_t u[32];
            PKV_TMEM_LD32(sa + ch * 32, u);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], __uint_as_float(u[c]));
          }
          const float mnew = fmaxf(m, fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2);
          resc = mnew > m + kRescaleThreshold;
          if (resc) {
            alpha = fast_exp2(m - mnew);  // 0 on the first tile
            m = mnew;
          }
          // pass 2: probabilities in place as packed bf16 hi | lo, where hi
          // keeps the top 16 bits of p and lo = p - hi (exact) is truncated
          // the same way: hi + lo is p to 2^-14 relative
          const float2 sl2x2 = make_float2(sl2, sl2);
          const float2 negm = make_float2(-m, -m);
          const float2 minus1 = make_float2(-1.f, -1.f);
          float2 rsa = make_float2(0.f, 0.f), rsb = make_float2(0.f, 0.f);
#pragma unroll 1
          for (int ch = 0; ch < kBN / 32; ++ch) {
            uint32_t u[32];
            PKV_TMEM_LD32(sa + ch * 32, u);
            tmem_wait_ld();
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float2 x2 = __ffma2_rn(
                  make_float2(__uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1])), sl2x2, negm);
              const float2 p2 = make_float2(fast_exp2(x2.x), fast_exp2(x2.y));
              if (c & 1)
                rsb = __fadd2_rn(rsb, p2);
              else
                rsa = __fadd2_rn(rsa, p2);
              const uint32_t b0 = __float_as_uint(p2.x), b1 = __float_as_uint(p2.y);
              const float2 hi2 = make_float2(__uint_as_float(b0 & 0xffff0000u),
                                             __uint_as_float(b1 & 0xffff0000u));
              const float2 lo2 = __ffma2_rn(hi2, minus1, p2);
              pk[c] = __byte_perm(b0, b1, 0x7632);
              pk[16 + c] = __byte_perm(__float_as_uint(lo2.x), __float_as_uint(lo2.y), 0x7632);
            }
            PKV_TMEM_ST32(sa + ch * 32, pk);
          }
          tmem_wait_st();
          rs = (rsa.x + rsb.x) + (rsa.y + rsb.y);
        } else {
          // ---- a diagonal tile: hide the keys after each row's position
          // pass 1: row maximum over the visible keys
          float mx = -INFINITY;
#pragma unroll 1
          for (int ch = 0; ch < kBN / 32; ++ch) {
            uint32_t u[32];
            PKV_TMEM_LD32(sa + ch * 32, u);
            tmem_wait_ld();
            const int vis = lim - ch * 32;
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c <= vis) mx = fmaxf(mx, __uint_as_float(u[c]));
          }
          const float mnew = fmaxf(m, mx * sl2);
          resc = mnew > m + kRescaleThreshold;
          if (resc) {
            alpha = fast_exp2(m - mnew);  // 0 on the first tile
            m = mnew;
          }
          // pass 2: probabilities, stored in place as packed bf16 hi | lo
          rs = 0.f;
#pragma unroll 1
          for (int ch = 0; ch < kBN / 32; ++ch) {
            uint32_t u[32];
            PKV_TMEM_LD32(sa + ch * 32, u);
            tmem_wait_ld();
            uint32_t pk[32];
            const int vis = lim - ch * 32;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              float p0 = fast_exp2(fmaf(__uint_as_float(u[2 * c]), sl2, -m));
              float p1 = fast_exp2(fmaf(__uint_as_float(u[2 * c + 1]), sl2, -m));
              if (2 * c > vis) p0 = 0.f;
              if (2 * c + 1 > vis) p1 = 0.f;
              rs += p0 + p1;
              pk[c] = pack_bf16x2(p0, p1);
              pk[16 + c] = pack_bf16x2(p0 - bf16_lo(pk[c]), p1 - bf16_hi(pk[c]));
            }
            PKV_TMEM_ST32(sa + ch * 32, pk);
          }
          tmem_wait_st();
        }
        l = l * alpha + rs;
        if (gg > 0) {
          // the previous tile's PV has finished writing O_x
          ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->o_done[x]), (gg - 1) & 1,
                                               p.status, abort));
          if (!ok) break;
          tc_fence_after();
          if (j > 0 && __any_sync(kFullMask, resc)) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t u[32];
              PKV_TMEM_LD32(oa + 32 * c, u);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
              PKV_TMEM_ST32(oa + 32 * c, u);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        __syncwarp();  // the warp's P (and O) stores precede its one arrival
        if (lane == 0) mbar_arrive(smem_addr(&bars->p_ready[x]));
      }
      if (!ok) break;
      // ---- epilogue of the item: O / l -> out, lse
      const int last = gt + d.n_tiles - 1;
      ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->o_done[x]), last & 1, p.status,
                                           abort));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* orow = p.out + d.seg * p.split_out_stride +
                    ((int64_t)(d.t0 + qj) * p.num_heads + d.kvh * G + g) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        PKV_TMEM_LD32(oa + 32 * c, u);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + 32 * c + e) =
                make_float4(__uint_as_float(u[e]) * inv, __uint_as_float(u[e + 1]) * inv,
                            __uint_as_float(u[e + 2]) * inv, __uint_as_float(u[e + 3]) * inv);
        }
      }
      if (row_valid && p.out_lse)
        p.out_lse[d.seg * p.split_lse_stride + (int64_t)(d.t0 + qj) * p.num_heads + d.kvh * G + g] =
            (m + fast_log2(l)) * kLn2;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bars->o_free[x]));  // the MMA may overwrite O_x now
      gt += d.n_tiles;
    }
  }

  // ---- teardown: all tcgen05 work of the CTA is complete; release TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) cta_finished(p);
}

template <int D>
cudaError_t launch_prefill_d(const AttnParams& p, const CUtensorMap& q_map, cudaStream_t stream) {
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
  return cudaLaunchKernelEx(&cfg, kernel, q_map, p);
}

}  // namespace

cudaError_t launch_prefill(const AttnParams& p, const CUtensorMap& q_map, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_prefill_d<128>(p, q_map, stream);
  if (p.head_dim == 64) return launch_prefill_d<64>(p, q_map, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
