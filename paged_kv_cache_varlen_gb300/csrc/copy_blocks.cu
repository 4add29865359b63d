// copy_blocks.cu -- whole-block copies inside the paged pool: the GPU half of
// copy-on-write (page 2, PagedAttention deep-dive: a shared block gets its own
// copy when a sequence writes into it). The host block manager decides which
// blocks to copy; this kernel moves the bytes.
//
// One CTA per (copy, K|V half, slice of the block): the block's
// block_size * num_kv_heads * head_dim bf16 values of that half are
// contiguous in the pool, so the copy is a straight 16-byte vector stream.
// Copies of one call must be independent (no block both a source and a
// destination), which the block manager's steps guarantee.
#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;  // 16-byte vectors per thread per CTA

__global__ void __launch_bounds__(kThreads)
    copy_blocks_kernel(uint4* pool, const int32_t* src, const int32_t* dst, int32_t num_blocks,
                       int64_t block_vecs, int32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int c = blockIdx.x;
  const int32_t s = __ldg(src + c), d = __ldg(dst + c);
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
      set_status(status, PKV_DEV_BAD_BLOCK);
    return;
  }
  const int64_t half = (int64_t)blockIdx.y * num_blocks * block_vecs;
  const uint4* from = pool + half + (int64_t)s * block_vecs;
  uint4* to = pool + half + (int64_t)d * block_vecs;
  const int64_t base = (int64_t)blockIdx.z * kThreads * kVecPerThread + threadIdx.x;
  uint4 v[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int64_t i = base + (int64_t)k * kThreads;
    if (i < block_vecs) v[k] = __ldg(from + i);
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int64_t i = base + (int64_t)k * kThreads;
    if (i < block_vecs) to[i] = v[k];
  }
}

}  // namespace

cudaError_t launch_copy_blocks(void* pool, const int32_t* src, const int32_t* dst,
                               int32_t num_copies, int32_t num_blocks, int64_t block_vecs,
                               int32_t* status, cudaStream_t stream) {
  const int64_t per_cta = (int64_t)kThreads * kVecPerThread;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_copies, 2u, (unsigned)((block_vecs + per_cta - 1) / per_cta));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, static_cast<uint4*>(pool), src, dst,
                            num_blocks, block_vecs, status);
}

}  // namespace pkv
