// cascade.cu -- preparation for the shared-prefix (cascade) decode: the
// prefix partials start empty (lse = -inf, so the merge ignores the segments
// a group does not have, and requests outside every group keep their tail
// result), and the tail pass gets one query per request (cu_seqlens = 0, 1,
// 2, ...).
#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
    cascade_prepare_kernel(float* part_lse, int64_t n_lse, int32_t* tail_cu, int32_t num_seqs) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_lse) part_lse[i] = -INFINITY;
  if (i <= num_seqs) tail_cu[i] = (int32_t)i;
}

}  // namespace

cudaError_t launch_cascade_prepare(float* part_lse, int64_t n_lse, int32_t* tail_cu,
                                   int32_t num_seqs, cudaStream_t stream) {
  const int64_t n = n_lse > (int64_t)num_seqs + 1 ? n_lse : (int64_t)num_seqs + 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cascade_prepare_kernel, part_lse, n_lse, tail_cu, num_seqs);
}

}  // namespace pkv
