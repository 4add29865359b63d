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

// Shared-prefix (cascade) merge: one warp per row, 4 rows per CTA, head_dim
// <= 128 (one float4 per lane). The row's request i = row / H belongs to
// the group g with group_starts[g] <= i < group_starts[g + 1] (none when i
// lies outside [group_starts[0], group_starts[G])); its prefix segments are
// slots 1 .. prefix_segment_count(prefix_lens[g], splits), its tail slot 0.
// The group tables (one entry per lane, for up to 31 groups) and the first
// P slots' partials are loaded together, in one memory round trip; slots
// past the request's segments are then treated as empty (they may hold
// anything).
template <int P>
__global__ void __launch_bounds__(128)
    cascade_merge_kernel(float* out, float* out_lse, const float* part_out,
                         const float* part_lse, int64_t num_rows, int H, int D,
                         const int32_t* group_starts, const int32_t* prefix_lens, int num_groups,
                         int splits) {
  griddep_wait();  // the tail and prefix partials are complete
  griddep_launch_dependents();
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= num_rows) return;
  const int lane = threadIdx.x & 31;
  const int32_t i = (int32_t)(row / H);
  const int nvec = D >> 2;
  const int slots = 1 + splits;
  const bool few = num_groups < 32;
  int32_t gs = 0x7fffffff, pl = 0;
  if (few && lane <= num_groups) gs = __ldg(group_starts + lane);
  if (few && lane < num_groups) pl = __ldg(prefix_lens + lane);
  float l[P];
  float4 o[P];
#pragma unroll
  for (int u = 0; u < P; ++u) {
    l[u] = u < slots ? part_lse[(int64_t)u * num_rows + row] * kLog2e : -INFINITY;
    o[u] = (u < slots && lane < nvec)
               ? reinterpret_cast<const float4*>(part_out + ((int64_t)u * num_rows + row) * D)[lane]
               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  int g = -1;
  if (few) {
    // group_starts is non-decreasing: the groups starting at or before i
    // are 0 .. g
    const uint32_t le = __ballot_sync(0xffffffffu, lane <= num_groups && gs <= i);
    const int32_t end = __shfl_sync(0xffffffffu, gs, num_groups);
    g = (le != 0u && i < end) ? 31 - __clz(le) : -1;
    const int32_t Lg = __shfl_sync(0xffffffffu, pl, g < 0 ? 0 : g);
    if (g >= 0) pl = Lg;
  } else if (num_groups > 0 && i >= __ldg(group_starts) && i < __ldg(group_starts + num_groups)) {
    int lo = 0, hi = num_groups;  // group_starts[lo] <= i < group_starts[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(group_starts + mid) <= i)
        lo = mid;
      else
        hi = mid;
    }
    g = lo;
    pl = __ldg(prefix_lens + lo);
  }
  const int segs = (g >= 0 && pl > 0) ? min(splits, prefix_segment_count(pl, splits)) : 0;
  const int used = 1 + segs;  // slots that hold this row's partials
  float M = -INFINITY, wsum = 0.f;  // log2 domain
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](float lu, const float4& ou) {
    if (lu == -INFINITY) return;  // empty
    if (lu > M) {
      const float c = fast_exp2(M - lu);  // 0 while M is -inf
      wsum *= c;
      acc.x *= c;
      acc.y *= c;
      acc.z *= c;
      acc.w *= c;
      M = lu;
    }
    const float w = fast_exp2(lu - M);
    wsum += w;
    acc.x += w * ou.x;
    acc.y += w * ou.y;
    acc.z += w * ou.z;
    acc.w += w * ou.w;
  };
#pragma unroll
  for (int u = 0; u < P; ++u)
    if (u < used) add(l[u], o[u]);
  for (int u = P; u < used; ++u) {  // more segments than one round trip holds
    const float lu = part_lse[(int64_t)u * num_rows + row] * kLog2e;
    const float4 ou =
        lane < nvec
            ? reinterpret_cast<const float4*>(part_out + ((int64_t)u * num_rows + row) * D)[lane]
            : make_float4(0.f, 0.f, 0.f, 0.f);
    add(lu, ou);
  }
  const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
  if (lane < nvec)
    reinterpret_cast<float4*>(out + row * D)[lane] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (out_lse && lane == 0) out_lse[row] = (wsum > 0.f) ? M * kLn2 + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_cascade_merge(float* out, float* out_lse, const float* part_out,
                                 const float* part_lse, int64_t num_rows, int32_t num_heads,
                                 int32_t head_dim, const int32_t* group_starts,
                                 const int32_t* prefix_lens, int32_t num_groups, int32_t splits,
                                 cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((num_rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (head_dim > 128) return cudaErrorInvalidValue;
  return cudaLaunchKernelEx(&cfg, cascade_merge_kernel<8>, out, out_lse, part_out, part_lse,
                            num_rows, (int)num_heads, (int)head_dim, group_starts, prefix_lens,
                            (int)num_groups, (int)splits);
}

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
