// decode.cu -- paged attention for query_len == 1 requests (decode).
//
// Method (sources as cited in include/pkv.h):
//   page 1 §04: GQA, kv_head = q_head / (num_heads / num_kv_heads); the six
//     attention steps; decode is a matrix-vector product whose cost is
//     moving the whole KV cache from HBM, so it is bandwidth-bound.
//   page 1 §02 / page 2 (PagedAttention deep-dive): block_table maps the
//     request's logical blocks to physical pool blocks.
//   page 2 step 4: causal mask. For decode the single query sits at
//     position seq_len - 1 and sees every cached key, including its own.
//   page 3 §3.4: fused, exact attention (online softmax; scores never
//     leave the SM).
//   page 1 §07: a long context is split into partitions whose partial
//     results are renormalised by log-sum-exp.
//
// GB300 design:
//   * one CTA = (request, KV head, head subgroup, partition); the CTA holds
//     the HG query heads that share that KV head, so each K/V byte of the
//     partition is read from HBM exactly once;
//   * each of the 4 warps owns SPW private pipeline slots; a slot holds one
//     16-token chunk of K and V for this KV head (16 rows of D bf16 at a
//     row stride of Hkv*D*2 bytes in the pool), fetched by one TMA tile
//     load each into shared memory and completed on the slot's mbarrier.
//     Warp w processes chunks w, w+4, w+8, ... and refills a slot as soon as
//     it has consumed it;
//   * inside a warp, LPT lanes cooperate on one token: each lane holds
//     64/HG elements of every query head of the group (pre-scaled by
//     scale*log2 e) and of the output accumulators, as float pairs for the
//     packed fp32x2 FMA; the LPT partial dot products are reduced by a
//     transpose-reduce over xor shuffles that leaves each lane with the full
//     score of ONE head, so each lane runs the online softmax of one head
//     and the probabilities are broadcast back for P*V;
//   * online softmax in the exp2 domain with lazy rescaling: the running
//     maximum only moves when a score exceeds it by more than 8 (a factor
//     256), which keeps the rescale off the common path and is exact up to
//     rounding; chunks whose 16 tokens are all valid take a check-free path;
//   * the lane groups of a warp merge by shuffles, the warps through shared
//     memory; a single-partition request is written directly. A split
//     request writes its normalised partial and log-sum-exp to the
//     workspace, and the last partition CTA to finish (an atomic counter per
//     (request, head group), reset by that CTA) merges all partials by
//     log-sum-exp -- no second kernel launch;
//   * programmatic dependent launch: the kernel may start while the KV
//     write that precedes it is finishing; it waits for that grid before
//     reading anything, then lets the next kernel launch.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kChunk = 16;  // tokens per TMA box and per pipeline stage
constexpr int kWarps = 4;
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr uint32_t kFull = 0xffffffffu;

template <int D, int HG>
struct DecodeGeometry {
  static constexpr int LPT = HG * D / 64;  // lanes per token
  static constexpr int DPL = D / LPT;      // elements of D per lane (= 64 / HG)
  static constexpr int CPL = DPL / 8;      // 16-byte vectors per lane per row
  static constexpr int TPW = 32 / LPT;     // tokens per warp per pass
  static constexpr int NPASS = (kChunk + TPW - 1) / TPW;
  static constexpr int ROW = D * 2;        // bytes of one K or V row
  static constexpr int SLOT = 2 * kChunk * ROW;
  static constexpr int LOG_HG = HG == 1 ? 0 : HG == 2 ? 1 : HG == 4 ? 2 : 3;
  static_assert(LPT >= HG && LPT <= 32 && (32 % LPT) == 0, "bad lanes per token");
  static_assert(CPL >= 1, "at least one 16-byte vector per lane");
};

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(bf16_lo(w), bf16_hi(w));
}

// Reduce the HG partial dot products v[] of one token over its LPT lanes so
// that the lane ends up with the full score of one head, returned. The head
// a lane holds is own_head(s) for its position s in the token's lane group.
template <int D, int HG>
__device__ __forceinline__ float transpose_reduce(const float (&v)[HG], int s) {
  using Geo = DecodeGeometry<D, HG>;
  float a[HG];
#pragma unroll
  for (int g = 0; g < HG; ++g) a[g] = v[g];
#pragma unroll
  for (int k = 0; k < Geo::LOG_HG; ++k) {
    const int off = Geo::LPT >> (k + 1);
    const bool hi = (s & off) != 0;
#pragma unroll
    for (int i = 0; i < (HG >> (k + 1)); ++i) {
      const float keep = hi ? a[i + (HG >> (k + 1))] : a[i];
      const float send = hi ? a[i] : a[i + (HG >> (k + 1))];
      a[i] = keep + __shfl_xor_sync(kFull, send, off);
    }
  }
#pragma unroll
  for (int off = Geo::LPT >> (Geo::LOG_HG + 1); off > 0; off >>= 1)
    a[0] += __shfl_xor_sync(kFull, a[0], off);
  return a[0];
}

template <int D, int HG>
__device__ __forceinline__ int own_head(int s) {
  using Geo = DecodeGeometry<D, HG>;
  int h = 0;
#pragma unroll
  for (int k = 0; k < Geo::LOG_HG; ++k)
    if (s & (Geo::LPT >> (k + 1))) h += HG >> (k + 1);
  return h;
}

// Position inside a token's lane group of the lane that holds head g.
template <int D, int HG>
__device__ __forceinline__ int owner_offset(int g) {
  using Geo = DecodeGeometry<D, HG>;
  int s = 0;
#pragma unroll
  for (int k = 0; k < Geo::LOG_HG; ++k)
    if (g & (HG >> (k + 1))) s += Geo::LPT >> (k + 1);
  return s;
}

// Per-warp running state of the online softmax.
template <int D, int HG>
struct WarpState {
  static constexpr int NP = DecodeGeometry<D, HG>::DPL / 2;
  float2 q[HG][NP];  // query slices, scaled by scale*log2(e)
  float2 o[HG][NP];  // unnormalised output slices
  float m;           // running max of this lane's own head (log2 units)
  float l;           // running sum of this lane's own head
};

// One 16-token chunk. Each lane group owns NPASS tokens of the chunk (one per
// pass). Phase A computes their scores (independent dot products and
// transpose-reduces, so their latencies overlap), phase B makes one
// online-softmax update for all of them, phase C accumulates P*V.
template <int D, int HG, bool FULL>
__device__ __forceinline__ void decode_chunk(WarpState<D, HG>& st, const uint8_t* kbase,
                                             const uint8_t* vbase, int key0, int kend,
                                             bool chunk_ok, int s, int tg, int group_base) {
  using Geo = DecodeGeometry<D, HG>;
  constexpr int LPT = Geo::LPT, CPL = Geo::CPL, TPW = Geo::TPW, NPASS = Geo::NPASS;
  float sc[NPASS];
  bool valid[NPASS];
#pragma unroll
  for (int pass = 0; pass < NPASS; ++pass) {
    const int tok = pass * TPW + tg;
    valid[pass] = FULL || (chunk_ok && tok < kChunk && key0 + tok < kend);
    const int row = tok < kChunk ? tok : kChunk - 1;
    float2 acc[HG];
#pragma unroll
    for (int g = 0; g < HG; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const uint4 w =
          *reinterpret_cast<const uint4*>(kbase + row * Geo::ROW + (c * LPT + s) * 16);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 k2 = bf16x2_to_float2(ws[e]);
#pragma unroll
        for (int g = 0; g < HG; ++g) acc[g] = __ffma2_rn(st.q[g][c * 4 + e], k2, acc[g]);
      }
    }
    float part[HG];
#pragma unroll
    for (int g = 0; g < HG; ++g) part[g] = acc[g].x + acc[g].y;
    sc[pass] = transpose_reduce<D, HG>(part, s);
    if (!valid[pass]) sc[pass] = -INFINITY;
  }

  float mx = sc[0];
#pragma unroll
  for (int pass = 1; pass < NPASS; ++pass) mx = fmaxf(mx, sc[pass]);
  const float mn = fmaxf(st.m, mx);
  const bool need = mn > st.m + kRescaleThreshold;
  if (__any_sync(kFull, need)) {
    const float alpha = need ? fast_exp2(st.m - mn) : 1.f;  // 0 when m = -inf
    if (need) {
      st.l *= alpha;
      st.m = mn;
    }
#pragma unroll
    for (int g = 0; g < HG; ++g) {
      const float a = __shfl_sync(kFull, alpha, group_base + owner_offset<D, HG>(g));
      const float2 a2 = make_float2(a, a);
#pragma unroll
      for (int i = 0; i < WarpState<D, HG>::NP; ++i) st.o[g][i] = __fmul2_rn(st.o[g][i], a2);
    }
  }
  float pr[NPASS];
#pragma unroll
  for (int pass = 0; pass < NPASS; ++pass) {
    pr[pass] = valid[pass] ? fast_exp2(sc[pass] - st.m) : 0.f;
    st.l += pr[pass];
  }

#pragma unroll
  for (int pass = 0; pass < NPASS; ++pass) {
    const int tok = pass * TPW + tg;
    const int row = tok < kChunk ? tok : kChunk - 1;
    float pg[HG];
#pragma unroll
    for (int g = 0; g < HG; ++g)
      pg[g] = __shfl_sync(kFull, pr[pass], group_base + owner_offset<D, HG>(g));
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      uint4 w = *reinterpret_cast<const uint4*>(vbase + row * Geo::ROW + (c * LPT + s) * 16);
      if (!valid[pass]) w = make_uint4(0u, 0u, 0u, 0u);  // masked rows may hold NaN
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 v2 = bf16x2_to_float2(ws[e]);
#pragma unroll
        for (int g = 0; g < HG; ++g)
          st.o[g][c * 4 + e] = __ffma2_rn(v2, make_float2(pg[g], pg[g]), st.o[g][c * 4 + e]);
      }
    }
  }
}

template <int D, int HG, int SPW, int MINB>
__global__ void __launch_bounds__(kWarps * 32, MINB)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const AttnParams p) {
  using Geo = DecodeGeometry<D, HG>;
  constexpr int LPT = Geo::LPT, DPL = Geo::DPL, CPL = Geo::CPL, TPW = Geo::TPW;
  constexpr int NP = DPL / 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* slots = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * SPW * Geo::SLOT);
  int* flag = reinterpret_cast<int*>(bars + kWarps * SPW);

  // Everything below may read the pool the preceding KV write produces.
  griddep_wait();
  griddep_launch_dependents();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int group = p.num_heads / p.num_kv_heads;
  const int nsub = group / HG;
  const int kvh = blockIdx.x / nsub;
  const int h0 = kvh * group + (blockIdx.x % nsub) * HG;
  const int part = blockIdx.y;
  const int i = blockIdx.z;
  const bool leader = (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0);

  const int32_t t0 = p.cu_seqlens[i];
  const int32_t t1 = p.cu_seqlens[i + 1];
  if (t0 < 0 || t1 < t0 || t1 > p.num_tokens) {
    if (leader) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return;
  }
  if (t1 - t0 != 1) return;  // not a decode request
  const int32_t L = p.seq_lens[i];
  if (L < 1 || L > p.max_seq_len || L > p.max_blocks * p.block_size) {
    if (leader) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return;
  }
  const int32_t kbeg = part * p.part_size;
  if (kbeg >= L) return;
  const int32_t kend = min(L, kbeg + p.part_size);
  const int nchunks = (kend - kbeg + kChunk - 1) / kChunk;
  const int my_chunks = (nchunks - warp + kWarps - 1) / kWarps;

  if (lane == 0) {
    for (int s = 0; s < SPW; ++s) mbar_init(smem_addr(&bars[warp * SPW + s]), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&kv_map);
  __syncwarp();

  const int32_t* bt = p.block_table + (int64_t)i * p.max_blocks;
  // lane j of the warp caches the block id of the warp's chunk (kb + j)
  auto load_ids = [&](int kb) -> int32_t {
    const int k = kb + lane;
    if (k >= my_chunks) return -1;
    const int c = warp + k * kWarps;
    return __ldg(bt + (kbeg + c * kChunk) / p.block_size);
  };
  const int32_t nrows = p.num_blocks * p.block_size;
  auto issue = [&](int k, int32_t id) {  // lane 0 only
    const int slot = k % SPW;
    const uint32_t bar = smem_addr(&bars[warp * SPW + slot]);
    if (id < 0 || id >= p.num_blocks) {
      set_status(p.status, PKV_DEV_BAD_BLOCK);
      mbar_arrive(bar);  // no bytes: the chunk is skipped (masked)
      return;
    }
    const uint32_t dst = smem_addr(slots + (warp * SPW + slot) * Geo::SLOT);
    const int key0 = kbeg + (warp + k * kWarps) * kChunk;
    const int32_t row = id * p.block_size + key0 % p.block_size;
    mbar_arrive_expect_tx(bar, Geo::SLOT);
    tma_load_3d(dst, &kv_map, bar, 0, kvh, row);
    tma_load_3d(dst + kChunk * Geo::ROW, &kv_map, bar, 0, kvh, row + nrows);
  };

  int32_t ids_cur = load_ids(0);
  int32_t ids_next = load_ids(32);
  int issued = 0;
  for (int k = 0; k < SPW && k < my_chunks; ++k) {
    const int32_t id = __shfl_sync(kFull, ids_cur, k);
    if (lane == 0) issue(k, id);
    ++issued;
  }

  const int s = lane % LPT;
  const int tg = lane / LPT;
  const int group_base = tg * LPT;

  WarpState<D, HG> st;
#pragma unroll
  for (int g = 0; g < HG; ++g) {
    const uint4* qrow =
        reinterpret_cast<const uint4*>(p.q + ((int64_t)t0 * p.num_heads + h0 + g) * D);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const uint4 w = __ldg(qrow + c * LPT + s);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = bf16x2_to_float2(ws[e]);
        st.q[g][c * 4 + e] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
      }
    }
#pragma unroll
    for (int e = 0; e < NP; ++e) st.o[g][e] = make_float2(0.f, 0.f);
  }
  st.m = -INFINITY;
  st.l = 0.f;

  int kb = 0;
  int consumed = 0;
  for (int k = 0; k < my_chunks; ++k) {
    if (k - kb == 32) {
      kb += 32;
      ids_cur = ids_next;
      ids_next = load_ids(kb + 32);
    }
    const int slot = k % SPW;
    const bool ok =
        __all_sync(kFull, mbar_wait(smem_addr(&bars[warp * SPW + slot]), (k / SPW) & 1, p.status));
    if (!ok) break;
    consumed = k + 1;
    const int32_t id = __shfl_sync(kFull, ids_cur, k - kb);
    const bool chunk_ok = (id >= 0 && id < p.num_blocks);
    const int key0 = kbeg + (warp + k * kWarps) * kChunk;
    const uint8_t* kbase = slots + (warp * SPW + slot) * Geo::SLOT;
    const uint8_t* vbase = kbase + kChunk * Geo::ROW;

    if (chunk_ok && key0 + kChunk <= kend && TPW <= kChunk)
      decode_chunk<D, HG, true>(st, kbase, vbase, key0, kend, true, s, tg, group_base);
    else
      decode_chunk<D, HG, false>(st, kbase, vbase, key0, kend, chunk_ok, s, tg, group_base);
    __syncwarp();
    const int kn = k + SPW;
    if (kn < my_chunks) {
      const int32_t idn = (kn - kb < 32) ? __shfl_sync(kFull, ids_cur, kn - kb)
                                         : __shfl_sync(kFull, ids_next, kn - kb - 32);
      if (lane == 0) {
        fence_proxy_async_smem();  // our reads of the slot precede the refill
        issue(kn, idn);
      }
      ++issued;
    }
  }
  // After an abandoned wait, let this warp's copies in flight land before the
  // CTA leaves (bounded as well).
  for (int k = consumed; k < issued; ++k)
    mbar_wait(smem_addr(&bars[warp * SPW + (k % SPW)]), (k / SPW) & 1, nullptr);

  // every lane gathers the running (m, l) of all HG heads of its token group
  float m[HG], l[HG];
#pragma unroll
  for (int g = 0; g < HG; ++g) {
    m[g] = __shfl_sync(kFull, st.m, group_base + owner_offset<D, HG>(g));
    l[g] = __shfl_sync(kFull, st.l, group_base + owner_offset<D, HG>(g));
  }
  // merge the warp's token groups (lanes tg differ) by xor shuffles
#pragma unroll
  for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
    for (int g = 0; g < HG; ++g) {
      const float mo = __shfl_xor_sync(kFull, m[g], off);
      const float lo = __shfl_xor_sync(kFull, l[g], off);
      const float M = fmaxf(m[g], mo);
      const float a = (m[g] == -INFINITY) ? 0.f : fast_exp2(m[g] - M);
      const float b = (mo == -INFINITY) ? 0.f : fast_exp2(mo - M);
      l[g] = a * l[g] + b * lo;
#pragma unroll
      for (int e = 0; e < NP; ++e) {
        const float ox = __shfl_xor_sync(kFull, st.o[g][e].x, off);
        const float oy = __shfl_xor_sync(kFull, st.o[g][e].y, off);
        st.o[g][e] = make_float2(a * st.o[g][e].x + b * ox, a * st.o[g][e].y + b * oy);
      }
      m[g] = M;
    }
  }

  __syncthreads();  // every warp is done with its slots: reuse them
  float* red_o = reinterpret_cast<float*>(smem);       // [kWarps][HG][D]
  float* red_ml = red_o + kWarps * HG * D;             // [kWarps][HG][2]
  if (tg == 0) {
#pragma unroll
    for (int g = 0; g < HG; ++g) {
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float* dst = red_o + (warp * HG + g) * D + (c * LPT + s) * 8 + 2 * e;
          dst[0] = st.o[g][c * 4 + e].x;
          dst[1] = st.o[g][c * 4 + e].y;
        }
      if (s == 0) {
        red_ml[(warp * HG + g) * 2] = m[g];
        red_ml[(warp * HG + g) * 2 + 1] = l[g];
      }
    }
  }
  __syncthreads();

  const int parts_i = (L + p.part_size - 1) / p.part_size;
  for (int idx = threadIdx.x; idx < HG * D; idx += kWarps * 32) {
    const int g = idx / D;
    const int d = idx - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_ml[(w * HG + g) * 2]);
    float wsum = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = red_ml[(w * HG + g) * 2];
      if (mw == -INFINITY) continue;
      const float a = fast_exp2(mw - M);
      wsum += a * red_ml[(w * HG + g) * 2 + 1];
      acc += a * red_o[(w * HG + g) * D + d];
    }
    const float val = wsum > 0.f ? acc / wsum : 0.f;
    const float lse = wsum > 0.f ? (M + fast_log2(wsum)) * kLn2 : -INFINITY;
    const int h = h0 + g;
    if (parts_i == 1) {
      p.out[((int64_t)t0 * p.num_heads + h) * D + d] = val;
      if (d == 0 && p.out_lse) p.out_lse[(int64_t)t0 * p.num_heads + h] = lse;
    } else {
      const int64_t r = ((int64_t)i * p.num_parts + part) * p.num_heads + h;
      p.ws_out[r * D + d] = val;
      if (d == 0) p.ws_lse[r] = lse;
    }
  }
  if (parts_i == 1) return;

  // ---- split request: the last partition CTA of (request, head group) merges
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // publish this CTA's partial before counting it
    const int old = atomicAdd(&p.ws_cnt[(int64_t)i * gridDim.x + blockIdx.x], 1);
    *flag = (old == parts_i - 1);
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();  // see every other partition's partial
  float* mg = red_ml;  // [HG] maxima of the partial lse (reuses shared memory)
  const int64_t row0 = (int64_t)i * p.num_parts * p.num_heads;
  for (int g = warp; g < HG; g += kWarps) {
    float M = -INFINITY;
    for (int pp = lane; pp < parts_i; pp += 32)
      M = fmaxf(M, __ldcg(p.ws_lse + row0 + (int64_t)pp * p.num_heads + h0 + g));
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    if (lane == 0) mg[g] = M;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < HG * D / 4; idx += kWarps * 32) {
    const int g = idx / (D / 4);
    const int d4 = idx - g * (D / 4);
    const float M = mg[g];
    const int h = h0 + g;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll 4
      for (int pp = 0; pp < parts_i; ++pp) {
        const int64_t r = row0 + (int64_t)pp * p.num_heads + h;
        const float w = fast_exp2((__ldcg(p.ws_lse + r) - M) * kLog2e);  // 0 for an empty part
        const float4 o = __ldcg(reinterpret_cast<const float4*>(p.ws_out + r * D) + d4);
        wsum += w;
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    reinterpret_cast<float4*>(p.out + ((int64_t)t0 * p.num_heads + h) * D)[d4] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (d4 == 0 && p.out_lse)
      p.out_lse[(int64_t)t0 * p.num_heads + h] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
  }
  if (threadIdx.x == 0) p.ws_cnt[(int64_t)i * gridDim.x + blockIdx.x] = 0;  // ready for reuse
}

template <int D, int HG, int SPW, int MINB>
cudaError_t launch_decode_t(const AttnParams& p, const CUtensorMap& kv_map, cudaStream_t stream) {
  using Geo = DecodeGeometry<D, HG>;
  const size_t smem = kWarps * SPW * Geo::SLOT + kWarps * SPW * sizeof(uint64_t) + 16;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, HG, SPW, MINB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int group = p.num_heads / p.num_kv_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_kv_heads * (group / HG), p.num_parts, p.num_seqs);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, HG, SPW, MINB>, kv_map, p);
}

// Occupancy per shape: 3 CTAs per SM (168 registers per thread, 2 slots per
// warp). The larger head groups would like ~210 registers and spill a few
// values at 168, but measured on GB300 the 12 resident warps still beat
// 2 CTAs per SM without spills by ~12 % (the kernel is latency-bound).
#ifndef PKV_DECODE_TIGHT_MINB
#define PKV_DECODE_TIGHT_MINB 3
#endif
template <int D, int HG>
struct DecodeOccupancy {
  static constexpr bool kWide = (D == 128 && HG >= 2) || (D == 64 && HG >= 4);
  static constexpr int MINB = kWide ? PKV_DECODE_TIGHT_MINB : 3;
  static constexpr int SPW = MINB == 3 ? 2 : 3;
};

template <int D, int HG>
cudaError_t launch_decode_g(const AttnParams& p, const CUtensorMap& kv_map, cudaStream_t stream) {
  using Occ = DecodeOccupancy<D, HG>;
  return launch_decode_t<D, HG, Occ::SPW, Occ::MINB>(p, kv_map, stream);
}

template <int D>
cudaError_t launch_decode_d(const AttnParams& p, const CUtensorMap& kv_map, cudaStream_t stream) {
  const int group = p.num_heads / p.num_kv_heads;
  if (group % 8 == 0) return launch_decode_g<D, 8>(p, kv_map, stream);
  if (group % 4 == 0) return launch_decode_g<D, 4>(p, kv_map, stream);
  if (group % 2 == 0) return launch_decode_g<D, 2>(p, kv_map, stream);
  return launch_decode_g<D, 1>(p, kv_map, stream);
}

}  // namespace

cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& kv_map, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_decode_d<128>(p, kv_map, stream);
  if (p.head_dim == 64) return launch_decode_d<64>(p, kv_map, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
