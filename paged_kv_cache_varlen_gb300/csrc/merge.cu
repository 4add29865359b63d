// merge.cu -- log-sum-exp merge of partial attention results.
//
// Method: page 1 ("从 token 调度到采样输出…", §07): chunked prefill,
// Flash-Decoding and sequence parallelism split attention into pieces and
// renormalise them with log-sum-exp. For a row with partials (o_p, lse_p):
//   M = max_p lse_p, w_p = exp(lse_p - M),
//   o = sum_p w_p o_p / sum_p w_p,  lse = M + ln sum_p w_p.
// A partial with lse = -inf is empty: its o_p never enters a sum (it may
// hold anything, NaN included). A row whose partials are all empty gives
// o = 0, lse = -inf.
//
// HBM-bound: each partial o_p (D fp32) is read once, each output written
// once. One warp per row; lanes hold consecutive float4 slices of D
// (coalesced).
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

// Row geometry: element (p, d) of the partial output of `row` sits at
// o_base + p * o_stride + d; its lse at lse_base + p * lse_stride.
struct RowView {
  const float* o_base;
  const float* lse_base;
  int64_t o_stride;
  int64_t lse_stride;
  int num_parts;
};

// Merge one row with one warp. NV = float4 slices per lane (head_dim <=
// 128 * NV). One pass over the partitions with a running maximum: U
// partitions' lse and outputs are loaded together before any is used, so a
// row costs about ceil(P / U) memory round trips instead of P. An empty
// partition's output is loaded with the others but never enters a sum.
// Writes out_row[0..D) and *out_lse (nullable).
template <int NV, int U>
__device__ __forceinline__ void merge_row(const RowView& v, int D, float* out_row,
                                          float* out_lse) {
  const int lane = threadIdx.x & 31;
  const int nvec = D >> 2;
  float M = -INFINITY, wsum = 0.f;  // log2 domain
  float4 acc[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < v.num_parts; base += U) {
    float l[U];
    float4 o[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int p = base + u;
      l[u] = p < v.num_parts ? v.lse_base[(int64_t)p * v.lse_stride] * kLog2e : -INFINITY;
      const float4* op = reinterpret_cast<const float4*>(v.o_base + (int64_t)p * v.o_stride);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int c = lane + 32 * j;
        o[u][j] = (p < v.num_parts && c < nvec) ? op[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (l[u] == -INFINITY) continue;  // empty (or past the last partition)
      if (l[u] > M) {
        const float c = fast_exp2(M - l[u]);  // 0 while M is -inf
        wsum *= c;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          acc[j].x *= c;
          acc[j].y *= c;
          acc[j].z *= c;
          acc[j].w *= c;
        }
        M = l[u];
      }
      const float w = fast_exp2(l[u] - M);
      wsum += w;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        acc[j].x += w * o[u][j].x;
        acc[j].y += w * o[u][j].y;
        acc[j].z += w * o[u][j].z;
        acc[j].w += w * o[u][j].w;
      }
    }
  }
  const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c = lane + 32 * j;
    if (c < nvec)
      reinterpret_cast<float4*>(out_row)[c] =
          make_float4(acc[j].x * inv, acc[j].y * inv, acc[j].z * inv, acc[j].w * inv);
  }
  if (out_lse && lane == 0) *out_lse = (wsum > 0.f) ? M * kLn2 + logf(wsum) : -INFINITY;
}

// Public dense merge: one warp per row, 4 rows per CTA.
template <int NV>
__global__ void __launch_bounds__(128)
    lse_merge_kernel(float* out, float* out_lse, const float* part_out, const float* part_lse,
                     int num_parts, int64_t num_rows, int D) {
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= num_rows) return;
  RowView v{part_out + row * D, part_lse + row, num_rows * D, num_rows, num_parts};
  merge_row<NV, NV == 1 ? 8 : 4>(v, D, out + row * D, out_lse ? out_lse + row : nullptr);
}

}  // namespace

cudaError_t launch_lse_merge(float* out, float* out_lse, const float* part_out,
                             const float* part_lse, int32_t num_parts, int64_t num_rows,
                             int32_t head_dim, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((num_rows + 3) / 4);
  if (head_dim <= 128)
    lse_merge_kernel<1><<<grid, 128, 0, stream>>>(out, out_lse, part_out, part_lse, num_parts,
                                                  num_rows, head_dim);
  else if (head_dim <= 256)
    lse_merge_kernel<2><<<grid, 128, 0, stream>>>(out, out_lse, part_out, part_lse, num_parts,
                                                  num_rows, head_dim);
  else
    lse_merge_kernel<4><<<grid, 128, 0, stream>>>(out, out_lse, part_out, part_lse, num_parts,
                                                  num_rows, head_dim);
  return cudaGetLastError();
}

}  // namespace pkv
