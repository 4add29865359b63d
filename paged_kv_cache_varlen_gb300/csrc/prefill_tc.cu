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
// GB300 design (one CTA per (request, KV head, tile of 128/G queries)):
//   * the Q tile is 128 rows = (128/G queries) x (G heads sharing the KV
//     head), so one pass over the K/V pages serves the whole GQA group;
//   * TMA tile loads with 128-byte swizzle: Q once ({64, G, 128/G} boxes),
//     K and V tiles of 128 keys as eight 16-key paged boxes each whose
//     physical block comes from block_table (no multicast);
//   * S = Q K^T (M=128, N=128, K=head_dim) and O += P V (M=128, N=head_dim,
//     K=128) run as tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) issued
//     by one thread; S (double-buffered), P and O live in tensor memory; P
//     is the A operand straight from TMEM. P is split into a bf16 high part
//     and a bf16 remainder, P ~= hi + lo to ~2^-16 relative, and O
//     accumulates hi*V + lo*V: a single bf16 rounding of P alone (2^-9
//     relative) puts few-key rows up to ~4e-3 off the exact result;
//   * four softmax warps own one TMEM lane (= one Q row) per thread: they
//     read S with tcgen05.ld, apply the causal mask and the online softmax
//     (exp2 domain, lazy rescale when the maximum grows by more than 8),
//     write P (hi and lo) with tcgen05.st once the previous tile's PV is
//     done, and rescale O in TMEM when needed;
//   * warp 4 produces TMA loads into a 2-stage K/V ring, warp 5 issues the
//     MMAs; QK^T of tile j+1 overlaps the softmax of tile j;
//   * every wait is bounded; on a timeout the CTA drains its copies and
//     MMAs, frees its TMEM and leaves with PKV_DEV_TIMEOUT set.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kBM = 128;  // Q rows per tile
constexpr int kBN = 128;  // keys per KV tile
constexpr int kNS = 2;    // K/V pipeline stages
constexpr int kSub = 16;  // keys per paged TMA box
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.f;

template <int D>
struct PrefillLayout {
  static constexpr int NCH = D / 64;                 // 128-byte column chunks of a row
  static constexpr int CH_BYTES = 128 * 128;         // one chunk of 128 rows
  static constexpr int Q_BYTES = NCH * CH_BYTES;
  static constexpr int KV_BYTES = NCH * CH_BYTES;    // one K or V tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;                  // [kNS] K tiles
  static constexpr int V_OFF = K_OFF + kNS * KV_BYTES;           // [kNS] V tiles
  static constexpr int BAR_OFF = V_OFF + kNS * KV_BYTES;
  static constexpr int SMEM = BAR_OFF + 256;
  // keep one CTA per SM (each CTA allocates all 512 TMEM columns)
  static constexpr int SMEM_ALLOC = (SMEM + 1024 > 120 * 1024) ? SMEM + 1024 : 120 * 1024;
  // TMEM columns
  __device__ static constexpr uint32_t s_col(int b) { return 128u * (uint32_t)b; }
  static constexpr uint32_t O_COL = 256;
  static constexpr uint32_t P_HI_COL = 256 + D;       // bf16(P), 64 columns
  static constexpr uint32_t P_LO_COL = 256 + D + 64;  // bf16(P - bf16(P)), 64 columns
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kNS];
  uint64_t v_full[kNS];
  uint64_t kv_empty[kNS];
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_done;
  uint64_t mma_done;
  uint32_t tmem_base;
  int32_t abort;
};

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

  griddep_wait();  // the KV write (and all earlier work) has landed
  griddep_launch_dependents();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t full = 0xffffffffu;
  const int G = p.num_heads / p.num_kv_heads;
  const int QT = kBM / G;  // queries per tile
  const int kvh = blockIdx.y;
  const int i = blockIdx.z;
  const bool leader = (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0);

  // ---- request geometry (uniform over the CTA; early exits before any setup)
  const int32_t t0 = p.cu_seqlens[i];
  const int32_t t1 = p.cu_seqlens[i + 1];
  if (t0 < 0 || t1 < t0 || t1 > p.num_tokens) {
    if (leader) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return;
  }
  const int32_t qlen = t1 - t0;
  if (qlen < 2) return;  // decode requests run on the decode kernel
  const int32_t L = p.seq_lens[i];
  if (qlen > p.max_query_len || L < qlen || L > p.max_seq_len ||
      L > p.max_blocks * p.block_size) {
    if (leader) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return;
  }
  const int ntq = (qlen + QT - 1) / QT;
  const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;  // heavier (later) tiles first
  if (qt >= ntq) return;
  const int j0 = qt * QT;
  const int j1 = min(qlen, j0 + QT);
  const int kv_end = L - qlen + j1;  // keys [0, kv_end) are needed
  const int n_tiles = (kv_end + kBN - 1) / kBN;

  // ---- setup: barriers (warp 4), TMEM (warp 5)
  if (warp == 4 && lane == 0) {
    mbar_init(smem_addr(&bars->q_full), 1);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(smem_addr(&bars->k_full[s]), 1);
      mbar_init(smem_addr(&bars->v_full[s]), 1);
      mbar_init(smem_addr(&bars->kv_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&bars->s_full[b]), 1);
      mbar_init(smem_addr(&bars->p_ready[b]), 128);
    }
    mbar_init(smem_addr(&bars->o_done), 1);
    mbar_init(smem_addr(&bars->mma_done), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
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

  if (warp == 4) {
    // ================= TMA producer =================
    const int32_t* bt = p.block_table + (int64_t)i * p.max_blocks;
    const int32_t nrows = p.num_blocks * p.block_size;
    if (lane == 0) {
      prefetch_tmap(&q_map);
      prefetch_tmap(&kv_map);
      mbar_arrive_expect_tx(smem_addr(&bars->q_full), Lay::Q_BYTES);
      for (int c = 0; c < Lay::NCH; ++c)
        tma_load_3d(q_s + c * Lay::CH_BYTES, &q_map, smem_addr(&bars->q_full), c * 64, kvh * G,
                    t0 + j0);
    }
    int32_t ids = -1;
    int issued = 0;
    bool bad_block = false;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % kNS;
      if ((j & 3) == 0) {  // block ids of the next 4 tiles, one 16-key box per lane
        const int key = (j * (kBN / kSub) + lane) * kSub;
        ids = (key < kv_end) ? __ldg(bt + key / p.block_size) : -1;
      }
      int ok = 1;
      if (lane == 0 && j >= kNS)
        ok = mbar_wait(smem_addr(&bars->kv_empty[st]), ((j / kNS) - 1) & 1, p.status, abort);
      ok = __shfl_sync(full, ok, 0);
      if (!ok) break;
      int32_t sub_id[kBN / kSub];
      uint32_t nvalid = 0;
#pragma unroll
      for (int sb = 0; sb < kBN / kSub; ++sb) {
        sub_id[sb] = __shfl_sync(full, ids, (j & 3) * (kBN / kSub) + sb);
        const int key = j * kBN + sb * kSub;
        if (key >= kv_end) {
          sub_id[sb] = -1;
        } else if (sub_id[sb] < 0 || sub_id[sb] >= p.num_blocks) {
          bad_block = true;
          sub_id[sb] = -1;
        } else {
          ++nvalid;
        }
      }
      if (lane == 0) {
        const uint32_t bytes = nvalid * kSub * 128 * Lay::NCH;
        const uint32_t kb = smem_addr(&bars->k_full[st]);
        const uint32_t vb = smem_addr(&bars->v_full[st]);
        mbar_arrive_expect_tx(kb, bytes);
#pragma unroll
        for (int sb = 0; sb < kBN / kSub; ++sb) {
          if (sub_id[sb] < 0) continue;
          const int key = j * kBN + sb * kSub;
          const int32_t row = sub_id[sb] * p.block_size + key % p.block_size;
          for (int c = 0; c < Lay::NCH; ++c)
            tma_load_3d(k_s + st * Lay::KV_BYTES + c * Lay::CH_BYTES + sb * kSub * 128, &kv_map,
                        kb, c * 64, kvh, row);
        }
        mbar_arrive_expect_tx(vb, bytes);
#pragma unroll
        for (int sb = 0; sb < kBN / kSub; ++sb) {
          if (sub_id[sb] < 0) continue;
          const int key = j * kBN + sb * kSub;
          const int32_t row = sub_id[sb] * p.block_size + key % p.block_size + nrows;
          for (int c = 0; c < Lay::NCH; ++c)
            tma_load_3d(v_s + st * Lay::KV_BYTES + c * Lay::CH_BYTES + sb * kSub * 128, &kv_map,
                        vb, c * 64, kvh, row);
        }
      }
      ++issued;
    }
    if (lane == 0) {
      if (bad_block) set_status(p.status, PKV_DEV_BAD_BLOCK);
      // make sure our last copies have landed before the CTA can exit
      for (int j = max(0, issued - kNS); j < issued; ++j) {
        mbar_wait(smem_addr(&bars->k_full[j % kNS]), (j / kNS) & 1, nullptr);
        mbar_wait(smem_addr(&bars->v_full[j % kNS]), (j / kNS) & 1, nullptr);
      }
      mbar_wait(smem_addr(&bars->q_full), 0, nullptr);
    }
  } else if (warp == 5) {
    // ================= MMA issuer (one thread) =================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kBM, D, false, true);
      auto issue_qk = [&](int j) {
        const int st = j % kNS;
        const uint32_t d_tmem = tmem + Lay::s_col(j & 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Lay::CH_BYTES + (kk & 3) * 32;
          const uint64_t a = smem_desc_sw128(q_s + off, 16, 1024);
          const uint64_t b = smem_desc_sw128(k_s + st * Lay::KV_BYTES + off, 16, 1024);
          umma_ss(d_tmem, a, b, idesc_qk, kk > 0);
        }
        umma_commit(smem_addr(&bars->s_full[j & 1]));
      };
      bool ok = mbar_wait(smem_addr(&bars->q_full), 0, p.status, abort) &&
                mbar_wait(smem_addr(&bars->k_full[0]), 0, p.status, abort);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
          ok = mbar_wait(smem_addr(&bars->k_full[(j + 1) % kNS]), ((j + 1) / kNS) & 1, p.status,
                         abort);
          if (!ok) break;
          tc_fence_after();
          issue_qk(j + 1);
        }
        ok = mbar_wait(smem_addr(&bars->p_ready[j & 1]), (j >> 1) & 1, p.status, abort) &&
             mbar_wait(smem_addr(&bars->v_full[j % kNS]), (j / kNS) & 1, p.status, abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t v_base = v_s + (j % kNS) * Lay::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t b = smem_desc_sw128(v_base + kk * 16 * 128, Lay::CH_BYTES, 1024);
          umma_ts(tmem + Lay::O_COL, tmem + Lay::P_HI_COL + kk * 8, b, idesc_pv,
                  (j > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t b = smem_desc_sw128(v_base + kk * 16 * 128, Lay::CH_BYTES, 1024);
          umma_ts(tmem + Lay::O_COL, tmem + Lay::P_LO_COL + kk * 8, b, idesc_pv, 1u);
        }
        umma_commit(smem_addr(&bars->kv_empty[j % kNS]));
        umma_commit(smem_addr(&bars->o_done));
      }
      // every MMA issued so far has completed before TMEM is released
      umma_commit(smem_addr(&bars->mma_done));
      mbar_wait(smem_addr(&bars->mma_done), 0, nullptr);
    }
  } else {
    // ================= softmax + epilogue: thread r owns Q row r =================
    const int r = threadIdx.x;
    const int qj = j0 + r / G;
    const int g = r % G;
    const bool row_valid = qj < j1;
    const int pos = row_valid ? (L - qlen + qj) : (kv_end - 1);
    const int pos_first = L - qlen + j0;  // smallest position in the tile
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = __all_sync(full, mbar_wait(smem_addr(&bars->s_full[j & 1]), (j >> 1) & 1, p.status,
                                      abort));
      if (!ok) break;
      tc_fence_after();
      float f[kBN];
      {
        uint32_t u[kBN];
        const uint32_t sa = tmem + lane_base + Lay::s_col(j & 1);
        PKV_TMEM_LD32(sa + 0, (u + 0));
        PKV_TMEM_LD32(sa + 32, (u + 32));
        PKV_TMEM_LD32(sa + 64, (u + 64));
        PKV_TMEM_LD32(sa + 96, (u + 96));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kBN; ++c) f[c] = __uint_as_float(u[c]);
      }
      const int k0 = j * kBN;
      float mx = -INFINITY;
      if (k0 + kBN - 1 > pos_first) {  // tile touches the diagonal: mask per element
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          if (k0 + c > pos) f[c] = -INFINITY;
          mx = fmaxf(mx, f[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kBN; ++c) mx = fmaxf(mx, f[c]);
      }
      const float mnew = fmaxf(m, mx * sl2);
      float alpha = 1.f;
      const bool resc = mnew > m + kRescaleThreshold;
      if (resc) {
        alpha = fast_exp2(m - mnew);  // 0 on the first tile
        m = mnew;
      }
      float rs = 0.f;
      uint32_t pk[kBN / 2], pl[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN / 2; ++c) {
        const float p0 = fast_exp2(fmaf(f[2 * c], sl2, -m));
        const float p1 = fast_exp2(fmaf(f[2 * c + 1], sl2, -m));
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
        pl[c] = pack_bf16x2(p0 - bf16_lo(pk[c]), p1 - bf16_hi(pk[c]));
      }
      l = l * alpha + rs;
      if (j > 0) {
        // PV of the previous tile must be done: it reads the P buffer we are
        // about to overwrite, and it writes the O we may rescale below.
        ok = __all_sync(full, mbar_wait(smem_addr(&bars->o_done), (j - 1) & 1, p.status, abort));
        if (!ok) break;
        tc_fence_after();
      }
      {
        const uint32_t ph = tmem + lane_base + Lay::P_HI_COL;
        const uint32_t plo = tmem + lane_base + Lay::P_LO_COL;
        PKV_TMEM_ST32(ph + 0, (pk + 0));
        PKV_TMEM_ST32(ph + 32, (pk + 32));
        PKV_TMEM_ST32(plo + 0, (pl + 0));
        PKV_TMEM_ST32(plo + 32, (pl + 32));
        tmem_wait_st();
      }
      if (j == n_tiles - 1 && (kv_end % kBN) != 0) {
        // V rows past the last needed key may hold anything (NaN included);
        // P is 0 there, and 0 * NaN would poison O, so zero them.
        ok = __all_sync(full, mbar_wait(smem_addr(&bars->v_full[j % kNS]), (j / kNS) & 1,
                                        p.status, abort));
        if (!ok) break;
        if (k0 + r >= kv_end) {
          uint8_t* vrow = smem + Lay::V_OFF + (j % kNS) * Lay::KV_BYTES + r * 128;
#pragma unroll
          for (int c = 0; c < Lay::NCH; ++c)
#pragma unroll
            for (int x = 0; x < 8; ++x)
              reinterpret_cast<uint4*>(vrow + c * Lay::CH_BYTES)[x] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      if (j > 0) {
        if (__any_sync(full, resc)) {
          const uint32_t oa = tmem + lane_base + Lay::O_COL;
#pragma unroll
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
      mbar_arrive(smem_addr(&bars->p_ready[j & 1]));
    }
    if (ok) {
      ok = __all_sync(full, mbar_wait(smem_addr(&bars->o_done), (n_tiles - 1) & 1, p.status,
                                      abort));
    }
    if (ok) {
      tc_fence_after();
      const uint32_t oa = tmem + lane_base + Lay::O_COL;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* orow = p.out + ((int64_t)(t0 + qj) * p.num_heads + kvh * G + g) * D;
#pragma unroll
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
        p.out_lse[(int64_t)(t0 + qj) * p.num_heads + kvh * G + g] =
            (m + fast_log2(l)) * kLn2;
    }
  }

  // ---- teardown: all tcgen05 work of the CTA is complete; release TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_prefill_d(const AttnParams& p, const CUtensorMap& q_map,
                             const CUtensorMap& kv_map, cudaStream_t stream) {
  using Lay = PrefillLayout<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int G = p.num_heads / p.num_kv_heads;
  const int QT = kBM / G;
  const dim3 grid((p.max_query_len + QT - 1) / QT, p.num_kv_heads, p.num_seqs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Lay::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_kernel<D>, q_map, kv_map, p);
}

}  // namespace

cudaError_t launch_prefill(const AttnParams& p, const CUtensorMap& q_map,
                           const CUtensorMap& kv_map, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_prefill_d<128>(p, q_map, kv_map, stream);
  if (p.head_dim == 64) return launch_prefill_d<64>(p, q_map, kv_map, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
