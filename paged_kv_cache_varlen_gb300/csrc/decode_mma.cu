// decode_mma.cu -- paged attention for decode requests (query_len == 1) and
// short verification steps (up to 32 (query, head) rows a request), with the
// two products of each 16-token chunk on the warp-level tensor-core path
// (mma.sync m16n8k16: bf16 operands, fp32 accumulation).
//
// Method (sources as cited in include/pkv.h):
//   page 1 §04: GQA, kv_head = q_head / (num_heads / num_kv_heads); decode
//     is a matrix-vector product bound by moving the KV cache from HBM.
//   page 1 §02 / page 2 (PagedAttention deep-dive): block_table maps the
//     request's logical blocks to physical pool blocks.
//   page 2 step 4: causal mask; the single query sits at position
//     seq_len - 1 and sees every cached key, including its own.
//   page 3 §3.4: fused, exact attention (online softmax on chip).
//   page 1 §07: long contexts split into partitions merged by log-sum-exp.
//
// Why tensor cores here: on CUDA cores a GQA group of 4 heads costs ~1024
// fp32 FMAs per (token, KV head) plus bf16 unpacking and shuffles for 512
// bytes of K and V; measured on GB300 that arithmetic, not HBM, bound the
// kernel (issue ~46 % active, ~52 warp instructions per token and KV head).
// The group's query heads form the 16 rows of an m16n8k16 tile, so each
// chunk's QK^T and PV are ~48 MMAs per warp instead, and the kernel is left
// to stream K/V.
//
// GB300 design (the pipeline is the one of the CUDA-core decode kernel):
//   * one CTA = (request, KV head, subgroup of up to 16 (query, head) rows,
//     partition); each K/V byte of a partition is read from HBM once by
//     each subgroup (one subgroup for a decode);
//   * 4 warps, each with SPW private slots; a slot holds one 16-token chunk
//     of K and of V for this KV head, fetched by one TMA load each (box of
//     16 rows x head_dim, laid out as the rows' first 128-byte halves then
//     their second halves, 128-byte swizzle, so that the 8 rows an ldmatrix
//     reads hit 8 different bank groups) and completed on the slot's mbarrier;
//   * S = Q K^T: Q is held as A fragments (rows = heads, zero padded), K
//     rows come in by ldmatrix as B fragments; online softmax in the exp2
//     domain with lazy rescaling (the running maximum moves only when a score
//     exceeds it by more than 8); P goes straight from the accumulator
//     registers into A fragments as a bf16 high part and a bf16 remainder
//     (p ~= hi + lo to ~2^-16), and O += P V
//     with V rows from ldmatrix.trans; V rows of tokens past the context are
//     zeroed first (P is 0 there, and 0 * NaN is not);
//   * end: warps merge through shared memory; a split request's partitions
//     write normalised partials and leave at once, and a small merge grid,
//     launched behind it with programmatic dependent launch, combines them
//     (per-CTA timelines showed the CTA that merged in-kernel spending ~8 us
//     of dependent memory round trips at the end of the grid);
//   * the prologue reads the request's lengths and the first block ids in
//     one round trip, so the first copies leave ~1 round trip earlier;
//   * decode-only batches with several-query requests (at most 256) run
//     longest context first: a one-CTA kernel before the grid ranks the
//     lengths, and grid slice z takes the request of rank z.
#include <math.h>

#include "common.cuh"
#include "launch.h"

#ifdef PKV_TEST_HOLD_ARRIVAL
// Test builds only: while set, warp 0 of the first CTA withholds the copy of
// its second chunk, so that its bounded wait on that chunk runs out.
__device__ int g_pkv_test_hold_decode;
extern "C" int pkv_test_hold_decode(int on) {
  return (int)cudaMemcpyToSymbol(g_pkv_test_hold_decode, &on, sizeof(int));
}
#endif

namespace pkv {
namespace {

constexpr int kChunk = 16;  // tokens per TMA box and per pipeline stage
constexpr int kWarps = 4;
constexpr int kRows = 16;   // MMA rows: query heads of the subgroup, zero padded
constexpr float kRescaleThreshold = 8.f;
constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// Byte offset of 16-byte unit `unit` of row `token` in a 16-row x D tile
// written by TMA with 128-byte swizzle (tile base 1024-byte aligned): the
// tile holds the 16 rows' first 128-byte halves (lines 0..15), then their
// second halves (lines 16..31); inside line q the unit u sits at u ^ (q % 8).
template <int D>
__device__ __forceinline__ uint32_t swz(int token, int unit) {
  const int line = (unit >> 3) * kChunk + token;
  return (uint32_t)(line * 128 + (((unit & 7) ^ (line & 7)) << 4));
}

// UNITQ: one query per request, request i being query i (no cu_seqlens
// array is read). ORDERED: grid slice z takes request p.order[z]. EARLY: the
// grid before this one is the call's own KV write, which let this grid
// launch only once everything before it had completed; it writes only the
// slots of the requests' query positions, so a CTA reads its inputs and the
// keys before its first query's position without waiting for it, and waits
// (the issuing lane of each warp) only before the copy of a chunk that holds
// a query position, and (every thread) before its output stores. Separate
// instantiations, so that every prologue's loads stay branch-free (a
// run-time choice there cost up to 5 %).
template <int D, int SPW, int MINB, bool UNITQ, bool ORDERED, bool EARLY>
__global__ void __launch_bounds__(kWarps * 32, MINB)
    decode_mma_kernel(const __grid_constant__ CUtensorMap kv_map, const AttnParams p) {
  constexpr int KS = D / 16;            // k-steps of QK^T
  constexpr int NT = D / 8;             // n-tiles of PV
  constexpr int HALF = kChunk * D * 2;  // bytes of the K (or V) rows of a chunk
  constexpr int SLOT = 2 * HALF;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* slots = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * SPW * SLOT);

  if (p.after_prefill) {
    // Launched behind a prefill grid, which does not produce anything read
    // here (it started after the preceding KV write had completed): only
    // the extra CTA (z = num_seqs) waits for that grid to complete, so
    // that this grid's completion implies the prefill grid's. The grid that
    // follows launches when every CTA here has finished.
    if ((int)blockIdx.z >= p.num_seqs) {
      if (blockIdx.x == 0 && blockIdx.y == 0) griddep_wait();
      return;
    }
  } else {
    // Everything below may read the pool the preceding KV write produces
    // (EARLY: see above).
    if constexpr (!EARLY) griddep_wait();
    griddep_launch_dependents();
  }

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  // MMA rows of a request: (query j, head g) pairs, j-major, cut into
  // subgroups of 16 rows; one query per request (decode) makes the rows the
  // heads of the GQA group
  const int group = p.num_heads / p.num_kv_heads;
  const int nsub = (p.decode_max_rows + kRows - 1) / kRows;
  const int kvh = blockIdx.x / nsub;
  const int sub = blockIdx.x - kvh * nsub;
  const int part = blockIdx.y;
  const int i = ORDERED ? __ldg(p.order + blockIdx.z) : (int)blockIdx.z;
  const bool leader = (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0);

  // The request's lengths and the block ids of this warp's first chunks are
  // fetched together, one memory round trip before the first copy is issued
  // (the ids are read speculatively, bounded by the table row only).
  const int32_t t0 = UNITQ ? i : __ldg(p.cu_seqlens + i);
  const int32_t t1 = UNITQ ? i + 1 : __ldg(p.cu_seqlens + i + 1);
  const int32_t L = __ldg(p.seq_lens + i);
  const bool ranged = p.key_start != nullptr;
  const int32_t kstart = ranged ? __ldg(p.key_start + i) : 0;
  const int32_t qstart = ranged ? __ldg(p.query_start + i) : 0;
  // several queries (a verification step) take partition 0 only, kbeg = 0
  const int32_t kbeg = part * p.part_size;
  const int32_t* bt = p.block_table + (int64_t)i * p.max_blocks;
  // lane j of the warp caches the block id of the warp's chunk (kb + j)
  auto load_ids = [&](int kb) -> int32_t {
    const int64_t c = warp + (int64_t)(kb + lane) * kWarps;
    const int64_t blk = (kbeg + c * kChunk) / p.block_size;
    return blk < p.max_blocks ? __ldg(bt + blk) : -1;
  };
  int32_t ids_cur = load_ids(0);
  int32_t ids_next = load_ids(32);

  if (t0 < 0 || t1 < t0 || t1 > p.num_tokens) {
    if (leader) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return;
  }
  const int32_t qlen = t1 - t0;
  if (qlen < 1 || qlen > p.decode_max_q) return;  // longer requests run on the prefill kernel
  if (qlen > p.max_query_len) {  // the grid covers only max_query_len queries' rows
    if (leader) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return;
  }
  const int row0 = sub * kRows;
  if (row0 >= qlen * group) return;  // no row of this request in the subgroup
  const int rows = min(kRows, qlen * group - row0);  // rows of this CTA
  if ((ranged ? (L < 1 || kstart < 0 || qstart < 0) : L < qlen) || L > p.max_seq_len ||
      L > p.max_blocks * p.block_size) {
    if (leader) set_status(p.status, PKV_DEV_BAD_LENGTHS);
    return;
  }
  // position of the request's first query among its keys (query j sees keys
  // 0 .. qpos0 + j); a key range may start after a query, which then sees
  // nothing of it
  const int32_t qpos0 =
      ranged ? (int32_t)max(-(1 << 30), min(1 << 30, qstart - kstart)) : L - qlen;
  // several queries: one partition over every key, with the causal limit per
  // row; one query: the split-KV partitions
  if (qlen > 1 && part > 0) return;
  if (kbeg >= L) return;
  const int32_t kend = qlen > 1 ? L : min(L, kbeg + p.part_size);
  const int nchunks = (kend - kbeg + kChunk - 1) / kChunk;
  const int my_chunks = (nchunks - warp + kWarps - 1) / kWarps;

  if (lane == 0) {
    for (int s = 0; s < SPW; ++s) mbar_init(smem_addr(&bars[warp * SPW + s]), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&kv_map);
  __syncwarp();

  const int32_t nrows = p.num_blocks * p.block_size;
  bool waited = false;  // EARLY: this lane has waited for the KV write
  auto issue = [&](int k, int32_t id) {  // lane 0 only
    const int slot = k % SPW;
    const uint32_t bar = smem_addr(&bars[warp * SPW + slot]);
    if (id < 0 || id >= p.num_blocks) {
      set_status(p.status, PKV_DEV_BAD_BLOCK);
      mbar_arrive(bar);  // no bytes: the chunk is skipped (masked)
      return;
    }
    const uint32_t dst = smem_addr(slots + (warp * SPW + slot) * SLOT);
    const int key0 = kbeg + (warp + k * kWarps) * kChunk;
    if constexpr (EARLY) {
      if (!waited && key0 + kChunk > qpos0) {  // the chunk holds a query position
        griddep_wait();
        waited = true;
      }
    }
    const int32_t row = id * p.block_size + key0 % p.block_size;
    mbar_arrive_expect_tx(bar, SLOT);
    tma_load_4d(dst, &kv_map, bar, 0, row, kvh, 0);
    tma_load_4d(dst + HALF, &kv_map, bar, 0, row + nrows, kvh, 0);
  };

  int issued = 0;
  for (int k = 0; k < SPW && k < my_chunks; ++k) {
    const int32_t id = __shfl_sync(kFull, ids_cur, k);
#ifdef PKV_TEST_HOLD_ARRIVAL
    if (g_pkv_test_hold_decode && k == 1 && warp == 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
        blockIdx.z == 0) {
      ++issued;  // counted as issued: the drain below waits for it (and gives up)
      continue;
    }
#endif
    if (lane == 0) issue(k, id);
    ++issued;
  }

  // Q of the subgroup as A fragments: row r = lane / 4 (and r + 8), columns
  // (lane % 4) * 2 + {0, 1} (and + 8) of every 16-wide k-step; rows past the
  // subgroup are zero.
  const int r = lane >> 2;
  const int cq = (lane & 3) * 2;
  // row -> (query, head): the query's token and the causal key limit
  auto row_token = [&](int rr) { return t0 + (row0 + rr) / group; };
  auto row_head = [&](int rr) { return kvh * group + (row0 + rr) % group; };
  auto row_limit = [&](int rr) {  // keys < limit are visible to the row
    return rr < rows ? min(kend, qpos0 + (row0 + rr) / group + 1) : 0;
  };
  uint32_t qa[KS][4];
  {
    const bool lo_ok = r < rows, hi_ok = r + 8 < rows;
    const uint16_t* q_lo = p.q + ((int64_t)row_token(r) * p.num_heads + row_head(r)) * D + cq;
    const uint16_t* q_hi =
        p.q + ((int64_t)row_token(r + 8) * p.num_heads + row_head(r + 8)) * D + cq;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = lo_ok ? __ldg(reinterpret_cast<const uint32_t*>(q_lo + ks * 16)) : 0u;
      qa[ks][1] = hi_ok ? __ldg(reinterpret_cast<const uint32_t*>(q_hi + ks * 16)) : 0u;
      qa[ks][2] = lo_ok ? __ldg(reinterpret_cast<const uint32_t*>(q_lo + ks * 16 + 8)) : 0u;
      qa[ks][3] = hi_ok ? __ldg(reinterpret_cast<const uint32_t*>(q_hi + ks * 16 + 8)) : 0u;
    }
  }
  const int lim0 = row_limit(r), lim1 = row_limit(r + 8);
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running maxima of rows r, r + 8 (log2 units)
  float l0 = 0.f, l1 = 0.f;              // this lane's share of the running sums
  const float sl2 = p.scale_log2;

  // ldmatrix lane addresses inside a tile: K (x4: tokens 0-7 / 8-15 x the
  // two 8-wide halves of a k-step) and V (x4.trans: tokens 0-7 / 8-15 x two
  // 8-wide n-tiles)
  const int mi = lane >> 3;
  const int k_tok = ((mi >> 1) << 3) + (lane & 7), k_unit = mi & 1;
  const int v_tok = ((mi & 1) << 3) + (lane & 7), v_unit = mi >> 1;

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
    const int nvalid = chunk_ok ? min(kChunk, kend - key0) : 0;
    uint8_t* kbase = slots + (warp * SPW + slot) * SLOT;
    uint8_t* vbase = kbase + HALF;
    if (nvalid < kChunk) {
      // rows past the context may hold anything, NaN included: zero those V
      // rows (their P is 0, and 0 * NaN would poison O)
      for (int e = lane; e < (kChunk - nvalid) * (D / 8); e += 32) {
        const int tok = nvalid + e / (D / 8);
        *reinterpret_cast<uint4*>(vbase + swz<D>(tok, e % (D / 8))) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    const uint32_t ka = smem_addr(kbase), va = smem_addr(vbase);

    // ---- S = Q K^T (two 8-token n-tiles)
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b[4];
      ldsm_x4(ka + swz<D>(k_tok, ks * 2 + k_unit), b);
      mma_16816(s[0], qa[ks], b[0], b[1]);
      mma_16816(s[1], qa[ks], b[2], b[3]);
    }
    // ---- mask (past the context, or after the row's own position), chunk
    // maxima (the 4 lanes of a quad share a row)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = nt * 8 + cq + j;
        if (tok >= nvalid || key0 + tok >= lim0) s[nt][j] = -INFINITY;
        if (tok >= nvalid || key0 + tok >= lim1) s[nt][2 + j] = -INFINITY;
        mx0 = fmaxf(mx0, s[nt][j]);
        mx1 = fmaxf(mx1, s[nt][2 + j]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
    const float n0 = fmaxf(m0, __fmul_rn(mx0, sl2)), n1 = fmaxf(m1, __fmul_rn(mx1, sl2));
    const bool r0 = n0 > m0 + kRescaleThreshold, r1 = n1 > m1 + kRescaleThreshold;
    if (__any_sync(kFull, r0 || r1)) {
      const float a0 = r0 ? fast_exp2(m0 - n0) : 1.f;  // 0 when m was -inf
      const float a1 = r1 ? fast_exp2(m1 - n1) : 1.f;
      if (r0) m0 = n0;
      if (r1) m1 = n1;
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[nt][0] *= a0;
        o[nt][1] *= a0;
        o[nt][2] *= a1;
        o[nt][3] *= a1;
      }
    }
    // ---- P = 2^(s * scale * log2 e - m), as bf16 hi + lo A fragments
    const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        // the product rounded exactly as for the maximum, so that the
        // largest score gives p = 1 exactly
        pr[nt][j] = fast_exp2(__fmul_rn(s[nt][j], sl2) - mu0);
        pr[nt][2 + j] = fast_exp2(__fmul_rn(s[nt][2 + j], sl2) - mu1);
      }
    l0 += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
    l1 += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
    uint32_t ah[4], al[4];
    ah[0] = pack_bf16x2(pr[0][0], pr[0][1]);
    ah[1] = pack_bf16x2(pr[0][2], pr[0][3]);
    ah[2] = pack_bf16x2(pr[1][0], pr[1][1]);
    ah[3] = pack_bf16x2(pr[1][2], pr[1][3]);
    al[0] = pack_bf16x2(pr[0][0] - bf16_lo(ah[0]), pr[0][1] - bf16_hi(ah[0]));
    al[1] = pack_bf16x2(pr[0][2] - bf16_lo(ah[1]), pr[0][3] - bf16_hi(ah[1]));
    al[2] = pack_bf16x2(pr[1][0] - bf16_lo(ah[2]), pr[1][1] - bf16_hi(ah[2]));
    al[3] = pack_bf16x2(pr[1][2] - bf16_lo(ah[3]), pr[1][3] - bf16_hi(ah[3]));
    // ---- O += P V (two n-tiles per ldmatrix)
#pragma unroll
    for (int n2 = 0; n2 < NT / 2; ++n2) {
      uint32_t b[4];
      ldsm_x4_trans(va + swz<D>(v_tok, n2 * 2 + v_unit), b);
      mma_16816(o[2 * n2], ah, b[0], b[1]);
      mma_16816(o[2 * n2], al, b[0], b[1]);
      mma_16816(o[2 * n2 + 1], ah, b[2], b[3]);
      mma_16816(o[2 * n2 + 1], al, b[2], b[3]);
    }
    __syncwarp();
    const int kn = k + SPW;
    if (kn < my_chunks) {
      const int32_t idn = (kn - kb < 32) ? __shfl_sync(kFull, ids_cur, kn - kb)
                                         : __shfl_sync(kFull, ids_next, kn - kb - 32);
      if (lane == 0) {
        fence_proxy_async_smem();  // our reads and writes of the slot precede the refill
        issue(kn, idn);
      }
      ++issued;
    }
  }
  // After an abandoned wait, let this warp's copies in flight land before the
  // CTA leaves (bounded as well).
  for (int k = consumed; k < issued; ++k)
    mbar_wait(smem_addr(&bars[warp * SPW + (k % SPW)]), (k / SPW) & 1, nullptr);

  // the quad's lanes hold a row's sum in four pieces
  l0 += __shfl_xor_sync(kFull, l0, 1);
  l0 += __shfl_xor_sync(kFull, l0, 2);
  l1 += __shfl_xor_sync(kFull, l1, 1);
  l1 += __shfl_xor_sync(kFull, l1, 2);

  __syncthreads();  // every warp is done with its slots: reuse them
  if constexpr (EARLY) griddep_wait();  // before the first output store
  // rows padded to D + 8 floats: the quads of 4 consecutive rows store to
  // disjoint banks; rows past the CTA's own are not stored at all
  constexpr int RS = D + 8;
  static_assert((size_t)kWarps * kRows * (RS + 2) * sizeof(float) <= (size_t)kWarps * SPW * SLOT,
                "the reduction buffers fit in the slots they reuse (one slot a warp does not)");
  float* red_o = reinterpret_cast<float*>(smem);       // [kWarps][kRows][RS]
  float* red_ml = red_o + kWarps * kRows * RS;         // [kWarps][kRows][2]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float* dst = red_o + (warp * kRows + r) * RS + nt * 8 + cq;
    if (r < rows) *reinterpret_cast<float2*>(dst) = make_float2(o[nt][0], o[nt][1]);
    if (r + 8 < rows) *reinterpret_cast<float2*>(dst + 8 * RS) = make_float2(o[nt][2], o[nt][3]);
  }
  if ((lane & 3) == 0) {
    red_ml[(warp * kRows + r) * 2] = m0;
    red_ml[(warp * kRows + r) * 2 + 1] = l0;
    red_ml[(warp * kRows + r + 8) * 2] = m1;
    red_ml[(warp * kRows + r + 8) * 2 + 1] = l1;
  }
  __syncthreads();

  const int parts_i = qlen > 1 ? 1 : (L + p.part_size - 1) / p.part_size;
  const int h0 = kvh * group + row0;  // one query: row g is head h0 + g
  for (int idx = threadIdx.x; idx < rows * D; idx += kWarps * 32) {
    const int g = idx / D;
    const int d = idx - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_ml[(w * kRows + g) * 2]);
    float wsum = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = red_ml[(w * kRows + g) * 2];
      if (mw == -INFINITY) continue;
      const float a = fast_exp2(mw - M);
      wsum += a * red_ml[(w * kRows + g) * 2 + 1];
      acc += a * red_o[(w * kRows + g) * RS + d];
    }
    const float val = wsum > 0.f ? acc / wsum : 0.f;
    const float lse = wsum > 0.f ? (M + fast_log2(wsum)) * kLn2 : -INFINITY;
    if (parts_i == 1) {
      const int64_t orow = (int64_t)row_token(g) * p.num_heads + row_head(g);
      p.out[orow * D + d] = val;
      if (d == 0 && p.out_lse) p.out_lse[orow] = lse;
    } else {
      const int h = h0 + g;
      const int64_t rr = ((int64_t)i * p.num_parts + part) * p.num_heads + h;
      p.ws_out[rr * D + d] = val;
      if (d == 0) p.ws_lse[rr] = lse;
    }
  }
}

// Split requests (one query, two or more partitions): the partitions'
// normalised outputs combined by their log-sum-exp (page 1 §07), as a
// separate grid so that no attention CTA waits on the others. WPR warps per
// (request, head) row split the partitions (one row per CTA when WPR > 1,
// four when WPR == 1); lanes hold float4 slices of D. Each warp makes one
// pass with a running maximum, so its partitions' loads can all be in
// flight; the warps then combine through shared memory.
template <int D, int WPR>
__global__ void __launch_bounds__(128 * (WPR == 1 ? 1 : WPR / 4))
    decode_merge_kernel(const AttnParams p) {
  constexpr int R = WPR == 1 ? 4 : 1;  // rows per CTA
  constexpr int RS = D + 4;  // floats per warp record: D, max, sum (16-byte multiple)
  __shared__ __align__(16) float red[WPR > 1 ? WPR * RS : 4];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.x * R + (R > 1 ? warp : 0);
  const int wr = R > 1 ? 0 : warp;  // this warp's share of the row's partitions
  const int i = blockIdx.y;
  // The lengths are inputs that the attention grid does not write. This grid
  // starts only once every attention CTA has passed its own wait on the
  // grids before it, so they are final; they are read (through L2) while the
  // attention grid is still running, off the path after its completion.
  const int32_t t0 = p.cu_seqlens ? __ldcg(p.cu_seqlens + i) : i;
  const int32_t t1 = p.cu_seqlens ? __ldcg(p.cu_seqlens + i + 1) : i + 1;
  const int32_t L = __ldcg(p.seq_lens + i);
  griddep_wait();  // the attention grid and its partials are complete
  griddep_launch_dependents();
  if (h >= p.num_heads) return;  // (uniform over the CTA when WPR > 1)
  // requests the attention kernel rejected (and flagged) or did not split
  if (t0 < 0 || t1 != t0 + 1 || t1 > p.num_tokens) return;
  if (L < 1 || L > p.max_seq_len || L > p.max_blocks * p.block_size) return;
  const int parts = (L + p.part_size - 1) / p.part_size;
  if (parts < 2) return;
  const int64_t r0 = (int64_t)i * p.num_parts * p.num_heads + h;
  const bool act = lane < D / 4;
  float M = -INFINITY, wsum = 0.f;  // log2 domain
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int U = 8;  // partitions in flight per warp
  for (int base = wr; base < parts; base += U * WPR) {
    float l[U];
    float4 ov[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int pp = base + u * WPR;
      const int64_t rr = r0 + (int64_t)pp * p.num_heads;
      l[u] = pp < parts ? __ldcg(p.ws_lse + rr) * kLog2e : -INFINITY;
      ov[u] = (pp < parts && act)
                  ? __ldcg(reinterpret_cast<const float4*>(p.ws_out + rr * D) + lane)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (l[u] == -INFINITY) continue;  // past the last partition
      if (l[u] > M) {
        const float c = fast_exp2(M - l[u]);  // 0 while M is -inf
        wsum *= c;
        acc.x *= c;
        acc.y *= c;
        acc.z *= c;
        acc.w *= c;
        M = l[u];
      }
      const float w = fast_exp2(l[u] - M);
      wsum += w;
      acc.x += w * ov[u].x;
      acc.y += w * ov[u].y;
      acc.z += w * ov[u].z;
      acc.w += w * ov[u].w;
    }
  }
  if (WPR > 1) {
    float* mine = red + warp * RS;
    if (act) reinterpret_cast<float4*>(mine)[lane] = acc;
    if (lane == 0) {
      mine[D] = M;
      mine[D + 1] = wsum;
    }
    __syncthreads();
    if (warp != 0) return;
    float Mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < WPR; ++w) Mt = fmaxf(Mt, red[w * RS + D]);
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    wsum = 0.f;
#pragma unroll
    for (int w = 0; w < WPR; ++w) {
      const float mw = red[w * RS + D];
      if (mw == -INFINITY) continue;
      const float c = fast_exp2(mw - Mt);
      wsum += c * red[w * RS + D + 1];
      if (act) {
        const float4 x = reinterpret_cast<const float4*>(red + w * RS)[lane];
        acc.x += c * x.x;
        acc.y += c * x.y;
        acc.z += c * x.z;
        acc.w += c * x.w;
      }
    }
    M = Mt;
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int64_t orow = (int64_t)t0 * p.num_heads + h;
  if (act)
    reinterpret_cast<float4*>(p.out + orow * D)[lane] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lane == 0 && p.out_lse) p.out_lse[orow] = wsum > 0.f ? (M + fast_log2(wsum)) * kLn2 : -INFINITY;
}

#ifndef PKV_DECODE_MMA_MINB
#define PKV_DECODE_MMA_MINB 3
#endif
#ifndef PKV_DECODE_MMA_SPW
#define PKV_DECODE_MMA_SPW 2
#endif

// Longest context first: order[rank] = request, rank by descending seq_len
// (ties by index); one CTA, at most 256 requests. Waits for the grid before
// it (the KV write), so that the decode grid's wait on it covers that too.
__global__ void __launch_bounds__(256) decode_order_kernel(const AttnParams p) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int32_t lens[256];
  const int B = p.num_seqs, t = threadIdx.x;
  if (t < B) lens[t] = __ldg(p.seq_lens + t);
  __syncthreads();
  if (t < B) {
    const int32_t l = lens[t];
    int rank = 0;
    for (int j = 0; j < B; ++j) {
      const int32_t lj = lens[j];
      rank += (lj > l || (lj == l && j < t)) ? 1 : 0;
    }
    p.order[rank] = t;
  }
}

template <int D>
cudaError_t launch_decode_mma_d(const AttnParams& p, const CUtensorMap& kv_map,
                                cudaStream_t stream) {
  constexpr int SPW = PKV_DECODE_MMA_SPW, MINB = PKV_DECODE_MMA_MINB;
  constexpr size_t SLOT = 2 * kChunk * D * 2;
  const size_t smem = 1024 + kWarps * SPW * SLOT + kWarps * SPW * sizeof(uint64_t) + 16;
  const bool unitq = p.cu_seqlens == nullptr;
  const bool ordered = p.order != nullptr && !unitq && !p.after_prefill && p.num_seqs <= 256;
  const bool early = p.early_pool && !unitq && !ordered && !p.after_prefill && !p.key_start;
  auto kernel = unitq     ? decode_mma_kernel<D, SPW, MINB, true, false, false>
                : ordered ? decode_mma_kernel<D, SPW, MINB, false, true, false>
                : early   ? decode_mma_kernel<D, SPW, MINB, false, false, true>
                          : decode_mma_kernel<D, SPW, MINB, false, false, false>;
  static SmemLimit limit_cu, limit_unit, limit_ordered, limit_early;
  SmemLimit& limit = unitq     ? limit_unit
                     : ordered ? limit_ordered
                     : early   ? limit_early
                               : limit_cu;
  if (cudaError_t e = limit.ensure(reinterpret_cast<const void*>(kernel), (int)smem);
      e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_kv_heads * ((p.decode_max_rows + kRows - 1) / kRows), p.num_parts,
                     p.num_seqs + (p.after_prefill ? 1 : 0));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (ordered) {
    cudaLaunchConfig_t ocfg = cfg;
    ocfg.gridDim = dim3(1);
    ocfg.blockDim = dim3(256);
    ocfg.dynamicSmemBytes = 0;
    if (cudaError_t e = cudaLaunchKernelEx(&ocfg, decode_order_kernel, p); e != cudaSuccess)
      return e;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, kv_map, p);
  if (e != cudaSuccess || p.num_parts < 2) return e;
  // few partitions: a warp per row; many: eight warps split a row's
  cudaLaunchConfig_t mcfg = cfg;
  mcfg.dynamicSmemBytes = 0;
  if (p.num_parts <= 8) {
    mcfg.gridDim = dim3((p.num_heads + 3) / 4, p.num_seqs);
    mcfg.blockDim = dim3(128);
    return cudaLaunchKernelEx(&mcfg, decode_merge_kernel<D, 1>, p);
  }
  mcfg.gridDim = dim3(p.num_heads, p.num_seqs);
  mcfg.blockDim = dim3(256);
  return cudaLaunchKernelEx(&mcfg, decode_merge_kernel<D, 8>, p);
}

}  // namespace

cudaError_t launch_decode_mma(const AttnParams& p, const CUtensorMap& kv_map, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_decode_mma_d<128>(p, kv_map, stream);
  if (p.head_dim == 64) return launch_decode_mma_d<64>(p, kv_map, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
