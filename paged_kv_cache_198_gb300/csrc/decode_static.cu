// decode_static.cu -- tvl_paged_attention_decode_noalloc: the decode entry
// point for callers that cannot allocate device memory.
//
// The split-K decode needs scratch memory for its partial (m, l, acc)
// records.  tvl_paged_attention_decode takes that scratch from the caller.
// Some callers have no allocator at the call site: a serving engine that
// handed all device memory to its KV pool up front, a plugin or callback
// interface that passes only input and output pointers, or a thread that must
// not block on the driver's allocation lock.  This entry point serves them
// from one file-scope device array of fixed size, kept by every GPU that
// loads the library until the process exits.
//
// Set-up: on its first call on a device, with that device current, the entry
// point looks up the array's device address (cudaGetSymbolAddress) and
// caches it per device; that first call should therefore come before any
// stream capture.  In host code the array's name is only a host-side stand-in
// and must never be handed to a kernel.
//
// Sharing: every call uses the same array.  The decode writes every partial
// record before the merge reads it, so nothing has to be cleared between
// calls, but calls that overlap on the GPU (different streams, or different
// host threads without ordering) race on the array.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/tvl.h"
#include "kernels.h"

namespace {

// Scratch for the partial records: 4 MiB, enough for the balanced split at
// up to 96 query heads on a 152-SM GPU, or a fixed split with
// S * splits * Hq * 66 * 4 bytes <= 4 MiB.
constexpr size_t kScratchBytes = 4u << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the scratch array (set up once per
// device, with that device current).
tvl_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    tvl::set_last_error(cudaGetErrorString(e));
    return TVL_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    tvl::set_last_error("device ordinal beyond the scratch table");
    return TVL_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char buf[256];
      snprintf(buf, sizeof buf, "cudaGetSymbolAddress(decode scratch): %s",
               cudaGetErrorString(e));
      tvl::set_last_error(buf);
      return TVL_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return TVL_OK;
}

}  // namespace

extern "C" tvl_status tvl_paged_attention_decode_noalloc(
    float* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
    float scale, int partition_size, void* stream) {
  size_t need = 0;
  tvl_status st = tvl_paged_attention_decode_workspace_size(
      num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
      partition_size, &need);
  if (st != TVL_OK) return st;
  if (need > kScratchBytes) {
    char buf[256];
    snprintf(buf, sizeof buf,
             "decode needs %zu bytes of scratch; the built-in scratch holds %zu bytes "
             "(use tvl_paged_attention_decode with a caller workspace)",
             need, kScratchBytes);
    tvl::set_last_error(buf);
    return TVL_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != TVL_OK) return st;
  return tvl_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens,
                                    num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                    num_blocks, max_blocks_per_seq, scale, partition_size,
                                    scratch, kScratchBytes, stream);
}
