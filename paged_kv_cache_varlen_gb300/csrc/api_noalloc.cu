// api_noalloc.cu -- pkv_paged_attention_varlen_noalloc: the attention call
// for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory: an inference engine
// whose memory manager has already claimed every byte of the GPU, a server
// that forbids cudaMalloc once it is serving (allocation can block or
// fragment at the worst moment), or a plugin that is handed only its input
// and output buffers. This entry point runs exactly the same kernels as
// pkv_paged_attention_varlen, but takes its split-KV scratch from one
// fixed-size array that lives in the library itself. Nothing here calls
// cudaMalloc, cudaFree or any allocating library routine.
//
// The scratch array is a file-scope __device__ variable. In host code its
// name is only a host-side stand-in, not a device address, so its device
// address is looked up with cudaGetSymbolAddress once per device (by the
// first call on that device, with the device current) and cached.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pkv.h"
#include "launch.h"

namespace {

// 16 MiB per device, shared by every call and held until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; the first call
// on a device looks it up.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_varlen_noalloc(
    float* out, float* out_lse, const void* q, const void* kv_pool, const int32_t* block_table,
    int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q, const int32_t* seq_lens,
    int32_t num_seqs, int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float scale, int32_t partition_size, int32_t* dev_status, void* stream) {
  // Every argument is checked before the scratch is looked up or touched;
  // then the call needs at most the built-in scratch (what
  // pkv_attention_workspace_size gives for these sizes), whose work tickets
  // are cleared on the stream before the kernels run.
  return pkv::attention_with_scratch(out, out_lse, q, kv_pool, block_table, max_blocks_per_seq,
                                     cu_seqlens_q, seq_lens, num_seqs, num_tokens, max_query_len,
                                     max_seq_len, num_heads, num_kv_heads, head_dim, block_size,
                                     num_blocks, scale, partition_size, dev_status, stream,
                                     kNoAllocScratchBytes, noalloc_scratch);
}
