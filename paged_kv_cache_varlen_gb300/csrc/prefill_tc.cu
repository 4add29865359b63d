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
//     sum of work items in shared memory and takes items blockIdx.x,
//     blockIdx.x + gridDim.x, ...; an item is (request, KV head, tile of
//     128/G queries), later query tiles (more keys) first. Tensor memory and
//     barriers are set up once per CTA, and no CTA is launched for decode
//     requests;
//   * the Q tile is 128 rows = (128/G queries) x (G heads sharing the KV
//     head), so one pass over the K/V pages serves the whole GQA group;
//   * Q arrives by TMA ({64, G, 128/G} boxes, 128-byte swizzle, double
//     buffered across items). K and V tiles of 128 keys are gathered page by
//     page (block ids from block_table) by two producer warps with 16-byte
//     cp.async copies written straight into the 128-byte-swizzled layout the
//     MMA descriptors read (keys past the needed range are zero-filled), in
//     separate 2-stage rings: a K stage is released as soon as its QK^T is
//     done, a V stage after its PV. (Paged 16-key TMA boxes were slower: the
//     TMA unit takes ~200 cycles per 2 KB box per SM, cp.async ~12 B/cycle);
//   * S = Q K^T (M=128, N=128, K=head_dim) and O += P V (M=128, N=head_dim,
//     K=128) run as tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) issued
//     by one thread; S is triple-buffered in tensor memory and P is written
//     back in place over the S columns it came from, as a bf16 high part and
//     a bf16 remainder (P ~= hi + lo to ~2^-16 relative; O accumulates
//     hi*V + lo*V -- a single bf16 rounding of P puts few-key rows up to
//     ~4e-3 off the exact result); P is the A operand straight from TMEM;
//   * four softmax warps own one TMEM lane (= one Q row) per thread: pass 1
//     reads S in 32-column pieces for the row maximum, pass 2 re-reads them,
//     applies the causal mask and the exp2-domain online softmax (lazy
//     rescale when the maximum grows by more than 8) and stores P; O is
//     rescaled in TMEM when needed;
//   * warps 4-5 produce loads, warp 6 issues the MMAs, polling so that QK^T
//     of tile j+1 and PV of tile j each go as soon as their inputs are ready
//     (QK^T first: the softmax waits for it); QK^T of tile j+1 overlaps the
//     softmax of tile j;
//   * every wait is bounded; on a timeout the CTA drains its copies and
//     MMAs, frees its TMEM and leaves with PKV_DEV_TIMEOUT set.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kBM = 128;  // Q rows per tile
constexpr int kBN = 128;  // keys per KV tile
constexpr int kNS = 2;    // stages of each of the K and V rings
constexpr int kSub = 16;  // keys per paged TMA box
constexpr int kProducers = 64;  // threads of the two K/V producer warps
constexpr int kMmaWarp = 6;
constexpr int kThreads = 224;   // 4 softmax warps, 2 producer warps, 1 MMA warp
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.f;
constexpr uint32_t kFullMask = 0xffffffffu;

template <int D>
struct PrefillLayout {
  static constexpr int NCH = D / 64;                       // 128-byte column chunks of a row
  static constexpr int CH_BYTES = 128 * 128;               // one chunk of 128 rows
  static constexpr int TILE_BYTES = NCH * CH_BYTES;        // one Q, K or V tile
  static constexpr int Q_OFF = 0;                          // [2] Q tiles
  static constexpr int K_OFF = Q_OFF + 2 * TILE_BYTES;     // [kNS] K tiles
  static constexpr int V_OFF = K_OFF + kNS * TILE_BYTES;   // [kNS] V tiles
  static constexpr int BAR_OFF = V_OFF + kNS * TILE_BYTES;
  static constexpr int PREF_OFF = BAR_OFF + 256;
  // keep one CTA per SM (each CTA allocates all 512 TMEM columns)
  static size_t bytes(int num_seqs) {
    const size_t need = 1024 + PREF_OFF + (size_t)(num_seqs + 1) * 4;
    return need > 120 * 1024 ? need : 120 * 1024;
  }
  // TMEM columns: S triple-buffered (P written in place), then O
  __device__ static constexpr uint32_t s_col(int b) { return 128u * (uint32_t)b; }
  static constexpr uint32_t O_COL = 384;
  // P of keys 16*kk .. 16*kk+15 inside an S buffer: each 32-key piece holds
  // 16 columns of packed hi then 16 columns of packed lo
  __device__ static constexpr uint32_t p_hi_col(int kk) {
    return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8);
  }
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kNS], k_empty[kNS];
  uint64_t v_full[kNS], v_empty[kNS];
  uint64_t s_full[3];
  uint64_t o_done[3];
  uint64_t p_ready;
  uint64_t o_free;
  uint64_t mma_done;
  uint32_t tmem_base;
  int32_t abort;
  int32_t scan[kThreads / 32];
};

struct PrefillItem {
  int req, kvh, j0, j1, t0, qlen, L, kv_end, n_tiles;
};

// Query tiles of request r (0 for decode requests); bad lengths flagged by
// CTA 0.
__device__ __forceinline__ int prefill_units(const AttnParams& p, int r, int QT, bool flag) {
  const int32_t t0 = __ldg(p.cu_seqlens + r), t1 = __ldg(p.cu_seqlens + r + 1);
  if (t0 < 0 || t1 < t0 || t1 > p.num_tokens) {
    if (flag) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return 0;
  }
  const int32_t qlen = t1 - t0;
  if (qlen < 2) return 0;  // decode requests run on the decode kernel
  const int32_t L = __ldg(p.seq_lens + r);
  if (qlen > p.max_query_len || L < qlen || L > p.max_seq_len ||
      L > p.max_blocks * p.block_size) {
    if (flag) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return 0;
  }
  return (qlen + QT - 1) / QT;
}

// pref[r] = query tiles of requests before r; pref[B] = total. All threads.
__device__ __forceinline__ int prefill_prefix(const AttnParams& p, int* pref, int32_t* scan,
                                              int QT) {
  const int B = p.num_seqs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool flag = blockIdx.x == 0;
  const int per = (B + kThreads - 1) / kThreads;
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  int sum = 0;
  for (int r = r0; r < r1; ++r) sum += prefill_units(p, r, QT, flag);
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
    run += prefill_units(p, r, QT, false);
  }
  if (tid == kThreads - 1) pref[B] = run;
  __syncthreads();
  return pref[B];
}

__device__ __forceinline__ PrefillItem prefill_item(const AttnParams& p, const int* pref, int QT,
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
  const int ntq = (d.qlen + QT - 1) / QT;
  const int qt = ntq - 1 - (u - pref[lo]);  // later (heavier) query tiles first
  d.j0 = qt * QT;
  d.j1 = min(d.qlen, d.j0 + QT);
  d.kv_end = d.L - d.qlen + d.j1;  // keys [0, kv_end) are needed
  d.n_tiles = (d.kv_end + kBN - 1) / kBN;
  return d;
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
  int* pref = reinterpret_cast<int*>(smem + Lay::PREF_OFF);

  griddep_wait();  // the KV write (and all earlier work) has landed
  griddep_launch_dependents();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.num_heads / p.num_kv_heads;
  const int QT = kBM / G;  // queries per tile

  // ---- setup: barriers (warp 4), work list (all), TMEM (MMA warp)
  if (warp == 4 && lane == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&bars->q_full[b]), 1);
      mbar_init(smem_addr(&bars->q_empty[b]), 1);
    }
    for (int s = 0; s < kNS; ++s) {
      mbar_init(smem_addr(&bars->k_full[s]), kProducers);
      mbar_init(smem_addr(&bars->k_empty[s]), 1);
      mbar_init(smem_addr(&bars->v_full[s]), kProducers);
      mbar_init(smem_addr(&bars->v_empty[s]), 1);
    }
    for (int b = 0; b < 3; ++b) {
      mbar_init(smem_addr(&bars->s_full[b]), 1);
      mbar_init(smem_addr(&bars->o_done[b]), 1);
    }
    mbar_init(smem_addr(&bars->p_ready), 128);
    mbar_init(smem_addr(&bars->o_free), 128);
    mbar_init(smem_addr(&bars->mma_done), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  const int total = prefill_prefix(p, pref, bars->scan, QT) * p.num_kv_heads;  // syncs
  if ((int)blockIdx.x >= total) return;  // uniform; nothing allocated yet
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

  if (warp == 4 || warp == 5) {
    // ============ producers: Q by TMA (one thread), K/V by cp.async (64 threads) ============
    // Thread pt copies 16-byte piece pc of the rows of keys pk0, pk0 + KSTEP, ...
    // of every tile into the 128-byte-swizzled layout the MMA descriptors
    // expect (the piece at column unit u of row r lands at unit u ^ (r & 7)).
    // Keys past the needed range and rows of bad blocks are filled with
    // zeros (so V rows there never poison O).
    constexpr int RP = D / 8;                // 16-byte pieces per K or V row
    constexpr int KSTEP = kProducers / RP;   // keys per round
    constexpr int NIT = kBN / KSTEP;         // rounds per tile
    static_assert(kSub % KSTEP == 0, "a round stays inside one 16-key sub-block");
    const int pt = threadIdx.x - 4 * 32;
    const int pc = pt % RP;
    const int pk0 = pt / RP;
    const uint32_t col_off = (uint32_t)((pc >> 3) * Lay::CH_BYTES);
    const uint32_t pcc = (uint32_t)(pc & 7);
    const int64_t row_bytes = (int64_t)p.num_kv_heads * D * 2;
    const uint8_t* pool = static_cast<const uint8_t*>(p.kv_pool);
    const int64_t v_half = (int64_t)p.num_blocks * p.block_size * row_bytes;
    const bool qlead = threadIdx.x == 4 * 32;
    if (qlead) prefetch_tmap(&q_map);
    int gi = 0, gt = 0, q_issued = 0, armed = 0;
    bool ok = true, bad_block = false;
    for (int it = blockIdx.x; ok && it < total; it += gridDim.x, ++gi) {
      const PrefillItem d = prefill_item(p, pref, QT, it);
      const int32_t* bt = p.block_table + (int64_t)d.req * p.max_blocks;
      if (warp == 4) {
        const int qb = gi & 1;
        int w = 1;
        if (lane == 0 && gi >= 2)
          w = mbar_wait(smem_addr(&bars->q_empty[qb]), ((gi >> 1) - 1) & 1, p.status, abort);
        ok = __shfl_sync(kFullMask, w, 0) != 0;
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_addr(&bars->q_full[qb]), Lay::TILE_BYTES);
          for (int c = 0; c < Lay::NCH; ++c)
            tma_load_3d(q_s + qb * Lay::TILE_BYTES + c * Lay::CH_BYTES, &q_map,
                        smem_addr(&bars->q_full[qb]), c * 64, d.kvh * G, d.t0 + d.j0);
        }
        ++q_issued;
      }
      const int64_t head_off = (int64_t)d.kvh * D * 2 + pc * 16;
      int32_t ids = -1;
      for (int j = 0; j < d.n_tiles; ++j, ++gt) {
        if ((j & 3) == 0) {  // block ids of the next 4 tiles, one 16-key sub-block per lane
          const int key = (j * (kBN / kSub) + lane) * kSub;
          ids = (key < d.kv_end) ? __ldg(bt + key / p.block_size) : -1;
        }
        // byte offset in the K half of the pool of each sub-block's first row
        // for this thread's piece, or -1 (zero fill)
        int64_t sub_off[kBN / kSub];
#pragma unroll
        for (int sb = 0; sb < kBN / kSub; ++sb) {
          const int32_t id = __shfl_sync(kFullMask, ids, (j & 3) * (kBN / kSub) + sb);
          const int key = j * kBN + sb * kSub;
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
            const bool valid = sub_off[sb] >= 0 && j * kBN + k < d.kv_end;
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
      if (warp == 4)
        for (int g = max(0, q_issued - 2); g < q_issued; ++g)
          mbar_wait(smem_addr(&bars->q_full[g & 1]), (g >> 1) & 1, nullptr);
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA issuer (one thread) =================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kBM, D, false, true);
      bool ok = true;
      int gi = 0, gt = 0;
      // S_g = Q K_g^T into S buffer g % 3 (P of tile g - 3 lived there)
      auto qk_ready = [&](int g) -> bool {
        return (g < 3 || mbar_test(smem_addr(&bars->o_done[g % 3]), ((g / 3) - 1) & 1)) &&
               mbar_test(smem_addr(&bars->k_full[g % kNS]), (g / kNS) & 1);
      };
      auto issue_qk = [&](int g, uint32_t q_base) {
        fence_proxy_async_smem();  // K was written by cp.async (generic proxy)
        tc_fence_after();
        const uint32_t d_tmem = tmem + Lay::s_col(g % 3);
        const uint32_t kb = k_s + (g % kNS) * Lay::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Lay::CH_BYTES + (kk & 3) * 32;
          umma_ss(d_tmem, smem_desc_sw128(q_base + off, 16, 1024),
                  smem_desc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0);
        }
        umma_commit(smem_addr(&bars->k_empty[g % kNS]));
        umma_commit(smem_addr(&bars->s_full[g % 3]));
      };
      // O += P_g V_g (P as bf16 high parts, then the remainders)
      auto issue_pv = [&](int g, bool first) {
        fence_proxy_async_smem();  // V was written by cp.async (generic proxy)
        tc_fence_after();
        const uint32_t s_base = tmem + Lay::s_col(g % 3);
        const uint32_t v_base = v_s + (g % kNS) * Lay::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t b = smem_desc_sw128(v_base + kk * 16 * 128, Lay::CH_BYTES, 1024);
          umma_ts(tmem + Lay::O_COL, s_base + Lay::p_hi_col(kk), b, idesc_pv,
                  (!first || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t b = smem_desc_sw128(v_base + kk * 16 * 128, Lay::CH_BYTES, 1024);
          umma_ts(tmem + Lay::O_COL, s_base + Lay::p_hi_col(kk) + 16, b, idesc_pv, 1u);
        }
        umma_commit(smem_addr(&bars->v_empty[g % kNS]));
        umma_commit(smem_addr(&bars->o_done[g % 3]));
      };
      for (int it = blockIdx.x; ok && it < total; it += gridDim.x, ++gi) {
        const PrefillItem d = prefill_item(p, pref, QT, it);
        const int qb = gi & 1;
        const uint32_t q_base = q_s + qb * Lay::TILE_BYTES;
        ok = mbar_wait(smem_addr(&bars->q_full[qb]), (gi >> 1) & 1, p.status, abort) &&
             (gt < 3 || mbar_wait(smem_addr(&bars->o_done[gt % 3]), ((gt / 3) - 1) & 1, p.status,
                                  abort)) &&
             mbar_wait(smem_addr(&bars->k_full[gt % kNS]), (gt / kNS) & 1, p.status, abort);
        if (!ok) break;
        issue_qk(gt, q_base);
        for (int j = 0; ok && j < d.n_tiles; ++j) {
          const int g = gt + j;
          // QK^T of the next tile and PV of this one, whichever can go first
          // (QK^T first when both can: the softmax waits for it)
          bool want_qk = j + 1 < d.n_tiles;
          bool want_pv = true;
          if (!want_qk) umma_commit(smem_addr(&bars->q_empty[qb]));  // Q no longer read
          const uint64_t t0 = globaltimer();
          for (uint32_t spin = 0; want_qk || want_pv; ++spin) {
            if (want_qk && qk_ready(g + 1)) {
              issue_qk(g + 1, q_base);
              want_qk = false;
              continue;
            }
            if (want_pv && mbar_test(smem_addr(&bars->p_ready), g & 1) &&
                mbar_test(smem_addr(&bars->v_full[g % kNS]), (g / kNS) & 1) &&
                (j > 0 || gi == 0 || mbar_test(smem_addr(&bars->o_free), (gi - 1) & 1))) {
              issue_pv(g, j == 0);  // the previous item's epilogue has read O
              want_pv = false;
              continue;
            }
            if ((spin & 63) == 63) {
              if (*abort) {
                ok = false;
                break;
              }
              if (globaltimer() - t0 > PKV_WAIT_TIMEOUT_NS) {
                set_status(p.status, PKV_DEV_TIMEOUT);
                *abort = 1;
                ok = false;
                break;
              }
            }
          }
        }
        gt += d.n_tiles;
      }
      // every MMA issued so far has completed before TMEM is released
      umma_commit(smem_addr(&bars->mma_done));
      mbar_wait(smem_addr(&bars->mma_done), 0, nullptr);
    }
  } else {
    // ================= softmax + epilogue: thread r owns Q row r =================
    const int r = threadIdx.x;
    const int rq = r / G;  // query of the row inside the tile
    const int g = r % G;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int gt = 0;
    for (int it = blockIdx.x; ok && it < total; it += gridDim.x) {
      const PrefillItem d = prefill_item(p, pref, QT, it);
      const int qj = d.j0 + rq;
      const bool row_valid = qj < d.j1;
      const int pos = row_valid ? (d.L - d.qlen + qj) : (d.kv_end - 1);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < d.n_tiles; ++j) {
        const int gg = gt + j;
        const int sb = gg % 3;
        ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->s_full[sb]), (gg / 3) & 1,
                                             p.status, abort));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = tmem + lane_base + Lay::s_col(sb);
        const int lim = pos - j * kBN;  // keys c <= lim of this tile are visible
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
        float alpha = 1.f;
        const bool resc = mnew > m + kRescaleThreshold;
        if (resc) {
          alpha = fast_exp2(m - mnew);  // 0 on the first tile
          m = mnew;
        }
        // pass 2: probabilities, stored in place as packed bf16 hi | lo
        float rs = 0.f;
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
        l = l * alpha + rs;
        if (gg > 0) {
          // the previous tile's PV has finished writing O
          const int pv = gg - 1;
          ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->o_done[pv % 3]), (pv / 3) & 1,
                                               p.status, abort));
          if (!ok) break;
          tc_fence_after();
          if (j > 0 && __any_sync(kFullMask, resc)) {
            const uint32_t oa = tmem + lane_base + Lay::O_COL;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t u[32];
              PKV_TMEM_LD32(oa + 32 * c, u);
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) u[x] = __float_as_uint(__uint_as_float(u[x]) * alpha);
              PKV_TMEM_ST32(oa + 32 * c, u);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        mbar_arrive(smem_addr(&bars->p_ready));
      }
      if (!ok) break;
      // ---- epilogue of the item: O / l -> out, lse
      const int last = gt + d.n_tiles - 1;
      ok = __all_sync(kFullMask, mbar_wait(smem_addr(&bars->o_done[last % 3]), (last / 3) & 1,
                                           p.status, abort));
      if (!ok) break;
      tc_fence_after();
      const uint32_t oa = tmem + lane_base + Lay::O_COL;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* orow = p.out + ((int64_t)(d.t0 + qj) * p.num_heads + d.kvh * G + g) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        PKV_TMEM_LD32(oa + 32 * c, u);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            *reinterpret_cast<float4*>(orow + 32 * c + x) =
                make_float4(__uint_as_float(u[x]) * inv, __uint_as_float(u[x + 1]) * inv,
                            __uint_as_float(u[x + 2]) * inv, __uint_as_float(u[x + 3]) * inv);
        }
      }
      if (row_valid && p.out_lse)
        p.out_lse[(int64_t)(d.t0 + qj) * p.num_heads + d.kvh * G + g] =
            (m + fast_log2(l)) * kLn2;
      tc_fence_before();
      mbar_arrive(smem_addr(&bars->o_free));  // the MMA may overwrite O now
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
}

template <int D>
cudaError_t launch_prefill_d(const AttnParams& p, const CUtensorMap& q_map,
                             const CUtensorMap& kv_map, cudaStream_t stream) {
  using Lay = PrefillLayout<D>;
  const size_t smem = Lay::bytes(p.num_seqs);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kernel = prefill_kernel<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int G = p.num_heads / p.num_kv_heads;
  const int QT = kBM / G;
  const int64_t bound = (int64_t)p.num_seqs * ((p.max_query_len + QT - 1) / QT) * p.num_kv_heads;
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

cudaError_t launch_prefill(const AttnParams& p, const CUtensorMap& q_map,
                           const CUtensorMap& kv_map, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_prefill_d<128>(p, q_map, kv_map, stream);
  if (p.head_dim == 64) return launch_prefill_d<64>(p, q_map, kv_map, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
