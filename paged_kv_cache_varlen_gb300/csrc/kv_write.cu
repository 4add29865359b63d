// kv_write.cu -- scatter the step's new K/V rows into the paged pool.
//
// Method: page 1 ("从 token 调度到采样输出…", §02 Paged Attention): the
// kernel writes each newly produced K/V row to the slot that slot_mapping
// names, slot = physical block * block_size + offset in the block.
//
// Layout: a token's K row for all KV heads, [Hkv][D] bf16, is contiguous in
// k_new and in the pool ([2][NB][BS][Hkv][D]: the slot index s addresses
// Hkv*D contiguous elements at s*Hkv*D in each half), so a token is one
// contiguous copy of Hkv*D*2 bytes per half. One warp copies one (token,
// K-or-V) row with 16-byte vector loads and stores; the whole write is
// HBM-bound (2 * T * Hkv * D * 2 bytes read and written).
#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kWarpsPerCta = 8;

__global__ void __launch_bounds__(kWarpsPerCta * 32)
    kv_write_kernel(KvWriteParams p) {
  griddep_wait();  // the previous step's attention may still read the pool
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (gw >= 2 * (int64_t)p.num_tokens) return;
  const int32_t t = (int32_t)(gw >> 1);
  const int which = (int)(gw & 1);  // 0 = K, 1 = V
  const int64_t s = p.slot_mapping[t];
  if (s == -1) return;
  if (s < 0 || s >= p.num_slots) {
    if (lane == 0 && which == 0) set_status(p.status, PKV_DEV_BAD_SLOT);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(which ? p.v_new : p.k_new) +
                     (int64_t)t * p.row_vecs;
  uint4* dst = reinterpret_cast<uint4*>(p.pool) +
               ((int64_t)which * p.num_slots + s) * p.row_vecs;
  int c = lane;
  for (; c + 96 < p.row_vecs; c += 128) {
    const uint4 a = __ldg(src + c), b = __ldg(src + c + 32), d = __ldg(src + c + 64),
                e = __ldg(src + c + 96);
    dst[c] = a;
    dst[c + 32] = b;
    dst[c + 64] = d;
    dst[c + 96] = e;
  }
  for (; c < p.row_vecs; c += 32) dst[c] = __ldg(src + c);
}

}  // namespace

cudaError_t launch_kv_write(const KvWriteParams& p, cudaStream_t stream) {
  const int64_t warps = 2 * (int64_t)p.num_tokens;
  const int64_t ctas = (warps + kWarpsPerCta - 1) / kWarpsPerCta;
  if (ctas == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_write_kernel, p);
}

}  // namespace pkv
