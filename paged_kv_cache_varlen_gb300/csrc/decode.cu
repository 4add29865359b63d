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
//     results are renormalised by log-sum-exp (merge.cu).
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
//     it has consumed it, so up to 4*SPW chunks are in flight per CTA;
//   * inside a warp, LPT lanes cooperate on one token: each lane holds
//     64/HG elements of every query head of the group (pre-scaled by
//     scale*log2 e) and of the output accumulators, computes partial dot
//     products with 16-byte shared-memory loads, and the lanes of the token
//     reduce them with xor shuffles;
//   * online softmax in the exp2 domain with lazy rescaling: the running
//     maximum only moves when a score exceeds it by more than 8 (a factor
//     256), which keeps the rescale off the common path and is exact up to
//     rounding;
//   * the lane groups of a warp merge by shuffles, the warps through shared
//     memory; the CTA writes the normalised output row (single partition)
//     or the partition's normalised partial and its log-sum-exp (split).
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kChunk = 16;  // tokens per TMA box and per pipeline stage
constexpr int kWarps = 4;
constexpr float kRescaleThreshold = 8.f;  // log2 units

template <int D, int HG>
struct DecodeGeometry {
  static constexpr int LPT = HG * D / 64;  // lanes per token
  static constexpr int DPL = D / LPT;      // elements of D per lane (= 64 / HG)
  static constexpr int CPL = DPL / 8;      // 16-byte vectors per lane per row
  static constexpr int TPW = 32 / LPT;     // tokens per warp per pass
  static constexpr int NPASS = (kChunk + TPW - 1) / TPW;
  static constexpr int ROW = D * 2;        // bytes of one K or V row
  static constexpr int SLOT = 2 * kChunk * ROW;
  static_assert(LPT >= 1 && LPT <= 32 && (32 % LPT) == 0, "bad lanes per token");
  static_assert(CPL >= 1, "at least one 16-byte vector per lane");
};

template <int D, int HG, int SPW>
__global__ void __launch_bounds__(kWarps * 32, 3)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const AttnParams p) {
  using Geo = DecodeGeometry<D, HG>;
  constexpr int LPT = Geo::LPT, DPL = Geo::DPL, CPL = Geo::CPL, TPW = Geo::TPW;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* slots = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * SPW * Geo::SLOT);

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

  const uint32_t full = 0xffffffffu;
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
    const int32_t id = __shfl_sync(full, ids_cur, k);
    if (lane == 0) issue(k, id);
    ++issued;
  }

  // query heads h0 .. h0+HG-1, this lane's slice of D, scaled by scale*log2(e)
  const int s = lane % LPT;
  const int tg = lane / LPT;
  float q[HG][DPL];
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
        q[g][c * 8 + 2 * e] = bf16_lo(ws[e]) * p.scale_log2;
        q[g][c * 8 + 2 * e + 1] = bf16_hi(ws[e]) * p.scale_log2;
      }
    }
  }
  float o[HG][DPL];
  float m[HG], l[HG];
#pragma unroll
  for (int g = 0; g < HG; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
  }

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
        __all_sync(full, mbar_wait(smem_addr(&bars[warp * SPW + slot]), (k / SPW) & 1, p.status));
    if (!ok) break;
    consumed = k + 1;
    const int32_t id = __shfl_sync(full, ids_cur, k - kb);
    const bool chunk_ok = (id >= 0 && id < p.num_blocks);
    const int key0 = kbeg + (warp + k * kWarps) * kChunk;
    const uint8_t* kbase = slots + (warp * SPW + slot) * Geo::SLOT;
    const uint8_t* vbase = kbase + kChunk * Geo::ROW;

#pragma unroll
    for (int pass = 0; pass < Geo::NPASS; ++pass) {
      const int tok = pass * TPW + tg;
      const bool valid = chunk_ok && tok < kChunk && key0 + tok < kend;
      const int row = tok < kChunk ? tok : kChunk - 1;
      float sc[HG];
#pragma unroll
      for (int g = 0; g < HG; ++g) sc[g] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const uint4 w =
            *reinterpret_cast<const uint4*>(kbase + row * Geo::ROW + (c * LPT + s) * 16);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float k0 = bf16_lo(ws[e]), k1 = bf16_hi(ws[e]);
#pragma unroll
          for (int g = 0; g < HG; ++g) {
            sc[g] = fmaf(q[g][c * 8 + 2 * e], k0, sc[g]);
            sc[g] = fmaf(q[g][c * 8 + 2 * e + 1], k1, sc[g]);
          }
        }
      }
#pragma unroll
      for (int off = LPT / 2; off > 0; off >>= 1)
#pragma unroll
        for (int g = 0; g < HG; ++g) sc[g] += __shfl_xor_sync(full, sc[g], off);

      bool need = false;
      float mn[HG];
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        if (!valid) sc[g] = -INFINITY;
        mn[g] = fmaxf(m[g], sc[g]);
        need |= (mn[g] > m[g] + kRescaleThreshold);
      }
      if (__any_sync(full, need)) {
#pragma unroll
        for (int g = 0; g < HG; ++g) {
          if (mn[g] > m[g] + kRescaleThreshold) {
            const float alpha = fast_exp2(m[g] - mn[g]);  // 0 when m = -inf
            l[g] *= alpha;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[g][e] *= alpha;
            m[g] = mn[g];
          }
        }
      }
      float pr[HG];
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        pr[g] = valid ? fast_exp2(sc[g] - m[g]) : 0.f;
        l[g] += pr[g];
      }
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        uint4 w = *reinterpret_cast<const uint4*>(vbase + row * Geo::ROW + (c * LPT + s) * 16);
        if (!valid) w = make_uint4(0u, 0u, 0u, 0u);  // masked rows may hold NaN
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v0 = bf16_lo(ws[e]), v1 = bf16_hi(ws[e]);
#pragma unroll
          for (int g = 0; g < HG; ++g) {
            o[g][c * 8 + 2 * e] = fmaf(pr[g], v0, o[g][c * 8 + 2 * e]);
            o[g][c * 8 + 2 * e + 1] = fmaf(pr[g], v1, o[g][c * 8 + 2 * e + 1]);
          }
        }
      }
    }
    __syncwarp();
    const int kn = k + SPW;
    if (kn < my_chunks) {
      const int32_t idn = (kn - kb < 32) ? __shfl_sync(full, ids_cur, kn - kb)
                                         : __shfl_sync(full, ids_next, kn - kb - 32);
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

  // merge the warp's token groups (lanes tg differ) by xor shuffles
#pragma unroll
  for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
    for (int g = 0; g < HG; ++g) {
      const float mo = __shfl_xor_sync(full, m[g], off);
      const float lo = __shfl_xor_sync(full, l[g], off);
      const float M = fmaxf(m[g], mo);
      const float a = (m[g] == -INFINITY) ? 0.f : fast_exp2(m[g] - M);
      const float b = (mo == -INFINITY) ? 0.f : fast_exp2(mo - M);
      l[g] = a * l[g] + b * lo;
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        const float oo = __shfl_xor_sync(full, o[g][e], off);
        o[g][e] = a * o[g][e] + b * oo;
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
        for (int e = 0; e < 8; ++e)
          red_o[(warp * HG + g) * D + (c * LPT + s) * 8 + e] = o[g][c * 8 + e];
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
}

template <int D, int HG, int SPW>
cudaError_t launch_decode_t(const AttnParams& p, const CUtensorMap& kv_map, cudaStream_t stream) {
  using Geo = DecodeGeometry<D, HG>;
  const size_t smem = kWarps * SPW * Geo::SLOT + kWarps * SPW * sizeof(uint64_t);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, HG, SPW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int group = p.num_heads / p.num_kv_heads;
  const dim3 grid(p.num_kv_heads * (group / HG), p.num_parts, p.num_seqs);
  decode_kernel<D, HG, SPW><<<grid, kWarps * 32, smem, stream>>>(kv_map, p);
  return cudaGetLastError();
}

constexpr int kSlotsPerWarp = 2;

template <int D>
cudaError_t launch_decode_d(const AttnParams& p, const CUtensorMap& kv_map, cudaStream_t stream) {
  const int group = p.num_heads / p.num_kv_heads;
  if (group % 8 == 0) return launch_decode_t<D, 8, kSlotsPerWarp>(p, kv_map, stream);
  if (group % 4 == 0) return launch_decode_t<D, 4, kSlotsPerWarp>(p, kv_map, stream);
  if (group % 2 == 0) return launch_decode_t<D, 2, kSlotsPerWarp>(p, kv_map, stream);
  return launch_decode_t<D, 1, kSlotsPerWarp>(p, kv_map, stream);
}

}  // namespace

size_t decode_smem_bytes(int head_dim) {
  return (size_t)kWarps * kSlotsPerWarp * (2 * kChunk * head_dim * 2 + sizeof(uint64_t));
}

cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& kv_map, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_decode_d<128>(p, kv_map, stream);
  if (p.head_dim == 64) return launch_decode_d<64>(p, kv_map, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
