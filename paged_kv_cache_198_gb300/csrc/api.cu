// api.cu -- the C ABI of libtvl.so (declared in include/tvl.h): argument
// validation on the host, the per-device status word, error strings and the
// dispatch to the kernels.  Every CUDA return code is checked and mapped to
// TVL_ERR_CUDA with its message [Tiny-vLLM digest, section "Evidence": the
// CUDA API reports errors through return values, which must not be ignored].
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/tvl.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

// Per-device status word (TVL_DEV_* bits and the timeout bit), set by
// kernels with atomicOr and read/cleared by tvl_get_device_status.
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
uint32_t* g_status_ptr[kMaxDevices] = {};

tvl_status fail(tvl_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

tvl_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TVL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of this device's status word (looked up once per device).
tvl_status status_word(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(TVL_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_status_ptr[dev];
  return TVL_OK;
}

tvl_status sm_count(int* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  return TVL_OK;
}

bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

// Shape checks shared by decode and prefill.
tvl_status check_heads(int hq, int hkv, int d) {
  if (hq <= 0 || hkv <= 0) return fail(TVL_ERR_INVALID_ARG, "head counts must be positive");
  if (hq % hkv != 0)
    return fail(TVL_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", hq, hkv);
  if (d != 64) return fail(TVL_ERR_UNSUPPORTED, "head_dim %d (supported: 64)", d);
  if (!supported_group(hq / hkv))
    return fail(TVL_ERR_UNSUPPORTED, "GQA group %d (supported: 1, 2, 4, 8)", hq / hkv);
  return TVL_OK;
}

// Balanced decode: CTAs per KV-head group (one CTA per SM in total); a CTA
// owns up to 8 KV heads (4 for GQA groups of 8).
int balanced_ctas(int sms, int hq, int hkv) {
  const int hmax = hq / hkv >= 8 ? 4 : 8;
  const int hpc = hkv < hmax ? hkv : hmax;
  const int groups = hkv / hpc;
  const int c = sms / groups;
  return c < 1 ? 1 : c;
}

tvl_status decode_sizes(int num_seqs, int hq, int hkv, int d, int mb, int bs, int part,
                        long long* records, int* part_blocks, int* max_splits, int* ctas) {
  if (num_seqs < 0) return fail(TVL_ERR_INVALID_ARG, "num_seqs %d < 0", num_seqs);
  if (mb <= 0) return fail(TVL_ERR_INVALID_ARG, "max_blocks_per_seq %d <= 0", mb);
  if (bs != 16 && bs != 32 && bs != 64 && bs != 128)
    return fail(TVL_ERR_UNSUPPORTED, "block_size %d (decode: 16, 32, 64, 128)", bs);
  if (part < 0 || part % bs != 0)
    return fail(TVL_ERR_INVALID_ARG, "partition_size %d not a non-negative multiple of %d", part,
                bs);
  tvl_status st = check_heads(hq, hkv, d);
  if (st != TVL_OK) return st;
  const int hmax = hq / hkv >= 8 ? 4 : 8;   // KV heads one CTA owns
  if (hkv > hmax && hkv % hmax != 0)
    return fail(TVL_ERR_UNSUPPORTED, "num_kv_heads %d (decode: <= %d or a multiple of %d)", hkv,
                hmax, hmax);
  *part_blocks = part / bs;
  *max_splits = part > 0 ? (mb + *part_blocks - 1) / *part_blocks : 0;
  *ctas = 0;
  if (part == 0) {
    int sms = 0;
    st = sm_count(&sms);
    if (st != TVL_OK) return st;
    *ctas = balanced_ctas(sms, hq, hkv);
  } else if (num_seqs > 65535) {
    return fail(TVL_ERR_UNSUPPORTED, "num_seqs %d > 65535 with a fixed partition", num_seqs);
  }
  *records = tvl::decode_records(num_seqs, mb, *part_blocks, *ctas);
  if (*records * hq > (1LL << 31) - 1)
    return fail(TVL_ERR_UNSUPPORTED, "too many split records (%lld)", *records);
  return TVL_OK;
}

}  // namespace

namespace tvl {
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }
}  // namespace tvl

extern "C" {

const char* tvl_status_string(tvl_status status) {
  switch (status) {
    case TVL_OK: return "ok";
    case TVL_ERR_INVALID_ARG: return "invalid argument";
    case TVL_ERR_UNSUPPORTED: return "unsupported configuration";
    case TVL_ERR_WORKSPACE: return "workspace missing or too small";
    case TVL_ERR_CUDA: return "CUDA error";
    case TVL_ERR_DEVICE_CHECK: return "device-side metadata check failed";
    case TVL_ERR_OUT_OF_BLOCKS: return "block pool exhausted";
  }
  return "unknown status";
}

const char* tvl_last_error(void) { return g_last_error.c_str(); }

int tvl_version(void) { return 100; }

tvl_status tvl_selftest_bounded_wait(void* stream) {
  uint32_t* word = nullptr;
  tvl_status st = status_word(&word);
  if (st != TVL_OK) return st;
  cudaError_t e = tvl::launch_selftest_wait(word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return TVL_OK;
}

tvl_status tvl_get_device_status(void* stream, uint32_t* bits) {
  uint32_t* word = nullptr;
  tvl_status st = status_word(&word);
  if (st != TVL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (host != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyAsync(word, &zero, sizeof zero, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  }
  if (bits) *bits = host;
  if (host != 0) return fail(TVL_ERR_DEVICE_CHECK, "device status bits 0x%x", host);
  return TVL_OK;
}

tvl_status tvl_paged_kv_write(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                              const int32_t* slot_mapping, int num_tokens, int num_kv_heads,
                              int head_dim, int block_size, int num_blocks, void* stream) {
  if (num_tokens < 0) return fail(TVL_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0)
    return fail(TVL_ERR_INVALID_ARG, "num_kv_heads, block_size and num_blocks must be positive");
  if (head_dim != 64) return fail(TVL_ERR_UNSUPPORTED, "head_dim %d (supported: 64)", head_dim);
  if (!k_cache || !v_cache) return fail(TVL_ERR_INVALID_ARG, "null cache pointer");
  if (!aligned16(k_cache) || !aligned16(v_cache))
    return fail(TVL_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  if (num_tokens == 0) return TVL_OK;
  if (!k_new || !v_new || !slot_mapping) return fail(TVL_ERR_INVALID_ARG, "null input pointer");
  if (!aligned16(k_new) || !aligned16(v_new))
    return fail(TVL_ERR_INVALID_ARG, "k_new / v_new must be 16-byte aligned");
  const long long row_bytes = 2LL * num_kv_heads * head_dim;
  if (row_bytes % 16 != 0) return fail(TVL_ERR_UNSUPPORTED, "row of %lld bytes", row_bytes);
  uint32_t* word = nullptr;
  tvl_status st = status_word(&word);
  if (st != TVL_OK) return st;
  tvl::KvWriteArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.row_bytes = static_cast<int>(row_bytes);
  a.num_slots = static_cast<long long>(num_blocks) * block_size;
  a.status = word;
  cudaError_t e = tvl::launch_kv_write(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_write launch");
  return TVL_OK;
}

tvl_status tvl_rope_paged_kv_write(void* q, const void* k_new, const void* v_new, void* k_cache,
                                   void* v_cache, const int32_t* slot_mapping,
                                   const int32_t* positions, int num_tokens, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                   float rope_theta, void* stream) {
  if (num_tokens < 0) return fail(TVL_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0 || num_q_heads < 0)
    return fail(TVL_ERR_INVALID_ARG, "head counts, block_size and num_blocks must be positive");
  if (head_dim != 64) return fail(TVL_ERR_UNSUPPORTED, "head_dim %d (supported: 64)", head_dim);
  if (!(rope_theta > 1.0f) || !std::isfinite(rope_theta))
    return fail(TVL_ERR_INVALID_ARG, "rope_theta must be finite and > 1");
  if (!k_cache || !v_cache) return fail(TVL_ERR_INVALID_ARG, "null cache pointer");
  if (!aligned16(k_cache) || !aligned16(v_cache))
    return fail(TVL_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  if (num_tokens == 0) return TVL_OK;
  if (!k_new || !v_new || !slot_mapping || !positions)
    return fail(TVL_ERR_INVALID_ARG, "null input pointer");
  if (q && num_q_heads == 0) return fail(TVL_ERR_INVALID_ARG, "q given with no query heads");
  if (!aligned16(v_new)) return fail(TVL_ERR_INVALID_ARG, "v_new must be 16-byte aligned");
  uint32_t* word = nullptr;
  tvl_status st = status_word(&word);
  if (st != TVL_OK) return st;
  tvl::RopeKvWriteArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.slot_mapping = slot_mapping;
  a.positions = positions;
  a.num_tokens = num_tokens;
  a.num_q_heads = q ? num_q_heads : 0;
  a.num_kv_heads = num_kv_heads;
  a.num_slots = static_cast<long long>(num_blocks) * block_size;
  a.log2_theta = std::log2(static_cast<double>(rope_theta));
  a.status = word;
  cudaError_t e = tvl::launch_rope_kv_write(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope_kv_write launch");
  return TVL_OK;
}

tvl_status tvl_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst,
                           int n, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           void* stream) {
  if (n < 0) return fail(TVL_ERR_INVALID_ARG, "n %d < 0", n);
  if (num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0)
    return fail(TVL_ERR_INVALID_ARG, "num_kv_heads, block_size and num_blocks must be positive");
  if (head_dim != 64) return fail(TVL_ERR_UNSUPPORTED, "head_dim %d (supported: 64)", head_dim);
  if (n == 0) return TVL_OK;
  if (!k_cache || !v_cache || !src || !dst) return fail(TVL_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_cache) || !aligned16(v_cache))
    return fail(TVL_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  uint32_t* word = nullptr;
  tvl_status st = status_word(&word);
  if (st != TVL_OK) return st;
  tvl::CopyBlocksArgs a;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.src = src;
  a.dst = dst;
  a.n = n;
  a.block_bytes = 2LL * block_size * num_kv_heads * head_dim;
  a.num_blocks = num_blocks;
  a.status = word;
  cudaError_t e = tvl::launch_copy_blocks(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return TVL_OK;
}

tvl_status tvl_paged_attention_decode_workspace_size(int num_seqs, int num_q_heads,
                                                     int num_kv_heads, int head_dim,
                                                     int max_blocks_per_seq, int block_size,
                                                     int partition_size, size_t* bytes) {
  if (!bytes) return fail(TVL_ERR_INVALID_ARG, "null bytes pointer");
  long long records = 0;
  int pb = 0, ms = 0, ctas = 0;
  tvl_status st = decode_sizes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               block_size, partition_size, &records, &pb, &ms, &ctas);
  if (st != TVL_OK) return st;
  *bytes = tvl::decode_workspace_bytes(records, num_q_heads, head_dim,
                                       tvl::decode_prefix_entries(num_seqs, pb));
  return TVL_OK;
}

namespace {

tvl_status decode_impl(float* out, const void* q, const void* k_new, const void* v_new,
                       const void* k_cache, const void* v_cache, const int32_t* block_tables,
                       const int32_t* context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       int max_blocks_per_seq, float scale, int partition_size, void* workspace,
                       size_t workspace_bytes, void* stream) {
  long long records = 0;
  int pb = 0, ms = 0, ctas = 0;
  tvl_status st = decode_sizes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               block_size, partition_size, &records, &pb, &ms, &ctas);
  if (st != TVL_OK) return st;
  if (num_blocks <= 0) return fail(TVL_ERR_INVALID_ARG, "num_blocks %d <= 0", num_blocks);
  if (!std::isfinite(scale)) return fail(TVL_ERR_INVALID_ARG, "scale is not finite");
  if (num_seqs == 0) return TVL_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(TVL_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(TVL_ERR_INVALID_ARG, "out, q, k_cache and v_cache must be 16-byte aligned");
  if ((k_new == nullptr) != (v_new == nullptr))
    return fail(TVL_ERR_INVALID_ARG, "k_new and v_new must both be given");
  if ((k_new && !aligned16(k_new)) || (v_new && !aligned16(v_new)))
    return fail(TVL_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  const long long prefix = tvl::decode_prefix_entries(num_seqs, pb);
  const size_t need = tvl::decode_workspace_bytes(records, num_q_heads, head_dim, prefix);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return fail(TVL_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (!aligned16(workspace)) return fail(TVL_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  }
  uint32_t* word = nullptr;
  st = status_word(&word);
  if (st != TVL_OK) return st;
  tvl::DecodeArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_new = k_new;
  a.v_new = v_new;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.scale = scale;
  a.partition_blocks = pb;
  a.max_splits = ms;
  a.balanced_ctas = ctas;
  a.window_ctas = 0;
  if (pb > 0 && ms > 1) {   // several windows a sequence: one persistent CTA per SM
    int sms = 0;
    st = sm_count(&sms);
    if (st != TVL_OK) return st;
    a.window_ctas = balanced_ctas(sms, num_q_heads, num_kv_heads);
  }
  a.ws = tvl::decode_workspace_carve(workspace, records, num_q_heads, head_dim, prefix);
  a.status = word;
  cudaError_t e = tvl::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return TVL_OK;
}

}  // namespace

tvl_status tvl_paged_attention_decode(float* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int num_blocks, int max_blocks_per_seq, float scale,
                                      int partition_size, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  return decode_impl(out, q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens,
                     num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                     max_blocks_per_seq, scale, partition_size, workspace, workspace_bytes,
                     stream);
}

tvl_status tvl_paged_decode_step(float* out, const void* q, const void* k_new,
                                 const void* v_new, void* k_cache, void* v_cache,
                                 const int32_t* block_tables, const int32_t* context_lens,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, int max_blocks_per_seq,
                                 float scale, int partition_size, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (num_seqs > 0 && (!k_new || !v_new))
    return fail(TVL_ERR_INVALID_ARG, "null k_new / v_new");
  return decode_impl(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                     num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                     max_blocks_per_seq, scale, partition_size, workspace, workspace_bytes,
                     stream);
}

tvl_status tvl_paged_attention_prefill(float* out, const void* q, const int32_t* query_start_loc,
                                       const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens,
                                       int num_seqs, int total_q_tokens, int max_q_len,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, int max_blocks_per_seq,
                                       float scale, void* stream) {
  if (num_seqs < 0 || total_q_tokens < 0 || max_q_len < 0)
    return fail(TVL_ERR_INVALID_ARG, "negative size");
  tvl_status st = check_heads(num_q_heads, num_kv_heads, head_dim);
  if (st != TVL_OK) return st;
  if (num_kv_heads > 255) return fail(TVL_ERR_UNSUPPORTED, "num_kv_heads %d > 255", num_kv_heads);
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
    return fail(TVL_ERR_UNSUPPORTED, "block_size %d (prefill: 16, 32, 64, 128)", block_size);
  if (num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(TVL_ERR_INVALID_ARG, "num_blocks and max_blocks_per_seq must be positive");
  if (!std::isfinite(scale)) return fail(TVL_ERR_INVALID_ARG, "scale is not finite");
  if (num_seqs == 0 || total_q_tokens == 0) return TVL_OK;
  if (max_q_len == 0) return fail(TVL_ERR_INVALID_ARG, "max_q_len 0 with queries present");
  if (num_seqs > 65535) return fail(TVL_ERR_UNSUPPORTED, "num_seqs %d > 65535", num_seqs);
  if (static_cast<long long>(num_seqs) * ((max_q_len + 127) / 128) * num_q_heads > INT_MAX)
    return fail(TVL_ERR_UNSUPPORTED, "num_seqs * ceil(max_q_len / 128) * num_q_heads > 2^31 - 1");
  if (!out || !q || !query_start_loc || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(TVL_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(TVL_ERR_INVALID_ARG, "out, q, k_cache and v_cache must be 16-byte aligned");
  uint32_t* word = nullptr;
  st = status_word(&word);
  if (st != TVL_OK) return st;
  tvl::PrefillArgs a;
  a.out = out;
  a.q = q;
  a.query_start_loc = query_start_loc;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.total_q_tokens = total_q_tokens;
  a.max_q_len = max_q_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.scale = scale;
  a.status = word;
  st = sm_count(&a.num_sms);
  if (st != TVL_OK) return st;
  cudaError_t e = tvl::launch_prefill(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return TVL_OK;
}

}  // extern "C"
