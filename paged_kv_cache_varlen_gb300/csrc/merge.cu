// merge.cu -- log-sum-exp merge of partial attention results.
//
// Method: page 1 ("从 token 调度到采样输出…", §07): chunked prefill,
// Flash-Decoding and sequence parallelism split attention into pieces and
// renormalise them with log-sum-exp. For a row with partials (o_p, lse_p):
//   M = max_p lse_p, w_p = exp(lse_p - M),
//   o = sum_p w_p o_p / sum_p w_p,  lse = M + ln sum_p w_p.
// A partial with lse = -inf is empty: it is skipped and its o_p never read.
// A row whose partials are all empty gives o = 0, lse = -inf.
//
// HBM-bound: each partial o_p (D fp32) is read once, each output written
// once. Lanes of a warp hold consecutive float4 slices of D (coalesced);
// the warps of a row split the partitions and combine through shared memory.
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

// Merge one row with WPR warps (threads = 32 * WPR). NV = float4 slices per
// lane (head_dim <= 128 * NV). Writes out_row[0..D) and *out_lse (nullable).
template <int WPR, int NV>
__device__ __forceinline__ void merge_row(const RowView& v, int D, float* out_row, float* out_lse,
                                          float* red /* shared, WPR*(D+2) floats or null */) {
  const int lane = threadIdx.x & 31;
  const int warp = (WPR == 1) ? 0 : (threadIdx.x >> 5);
  // max over partitions
  float M = -INFINITY;
  for (int p = warp * 32 + lane; p < v.num_parts; p += WPR * 32)
    M = fmaxf(M, v.lse_base[(int64_t)p * v.lse_stride]);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (WPR > 1) {
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < WPR; ++w) M = fmaxf(M, red[w]);
    __syncthreads();
  }
  const int nvec = D >> 2;
  float4 acc[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int p = warp; p < v.num_parts; p += WPR) {
      const float l = v.lse_base[(int64_t)p * v.lse_stride];
      if (l == -INFINITY) continue;
      const float w = fast_exp2((l - M) * kLog2e);
      wsum += w;
      const float4* op = reinterpret_cast<const float4*>(v.o_base + (int64_t)p * v.o_stride);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int c = lane + 32 * j;
        if (c < nvec) {
          const float4 x = op[c];
          acc[j].x += w * x.x;
          acc[j].y += w * x.y;
          acc[j].z += w * x.z;
          acc[j].w += w * x.w;
        }
      }
    }
  }
  if (WPR > 1) {
    // combine the warps' partial sums: red[w*(D+1) + d], red[w*(D+1) + D] = wsum
    float* mine = red + warp * (D + 1);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = lane + 32 * j;
      if (c < nvec) {
        mine[4 * c] = acc[j].x;
        mine[4 * c + 1] = acc[j].y;
        mine[4 * c + 2] = acc[j].z;
        mine[4 * c + 3] = acc[j].w;
      }
    }
    if (lane == 0) mine[D] = wsum;
    __syncthreads();
    if (warp == 0) {
      wsum = 0.f;
      for (int w = 0; w < WPR; ++w) wsum += red[w * (D + 1) + D];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int c = lane + 32 * j;
        if (c < nvec) {
          float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int w = 0; w < WPR; ++w) {
            const float* r = red + w * (D + 1) + 4 * c;
            s.x += r[0];
            s.y += r[1];
            s.z += r[2];
            s.w += r[3];
          }
          acc[j] = s;
        }
      }
    }
    if (warp != 0) return;
  }
  const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c = lane + 32 * j;
    if (c < nvec)
      reinterpret_cast<float4*>(out_row)[c] =
          make_float4(acc[j].x * inv, acc[j].y * inv, acc[j].z * inv, acc[j].w * inv);
  }
  if (out_lse && lane == 0) *out_lse = (wsum > 0.f) ? M + logf(wsum) : -INFINITY;
}

// Public dense merge: one warp per row, 4 rows per CTA.
template <int NV>
__global__ void __launch_bounds__(128)
    lse_merge_kernel(float* out, float* out_lse, const float* part_out, const float* part_lse,
                     int num_parts, int64_t num_rows, int D) {
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= num_rows) return;
  RowView v{part_out + row * D, part_lse + row, num_rows * D, num_rows, num_parts};
  merge_row<1, NV>(v, D, out + row * D, out_lse ? out_lse + row : nullptr, nullptr);
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
