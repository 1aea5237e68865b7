// kernels.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units.  Arguments arrive here already validated.
#pragma once

#include <atomic>

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace tvl {

// Runs a set-up step (e.g. a kernel attribute) once per device: the first
// successful run on a device is remembered, later calls on it return at once.
struct PerDeviceOnce {
  std::atomic<unsigned long long> done{0};   // bit d: device d set up
  template <typename F>
  cudaError_t run(F&& set_up) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = set_up();
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }
};

struct KvWriteArgs {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* slot_mapping;
  int num_tokens;
  int row_bytes;          // Hkv * D * 2, a multiple of 16
  long long num_slots;    // NB * bs
  uint32_t* status;
};
cudaError_t launch_kv_write(const KvWriteArgs& a, cudaStream_t stream);

struct RopeKvWriteArgs {
  void* q;                 // may be null
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* slot_mapping;
  const int32_t* positions;
  int num_tokens, num_q_heads, num_kv_heads;
  long long num_slots;
  double log2_theta;
  uint32_t* status;
};
cudaError_t launch_rope_kv_write(const RopeKvWriteArgs& a, cudaStream_t stream);

struct CopyBlocksArgs {
  void* k_cache;
  void* v_cache;
  const int32_t* src;
  const int32_t* dst;
  int n;
  long long block_bytes;   // bs * Hkv * D * 2
  int num_blocks;
  uint32_t* status;
};
cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream);

// Partial results of the decode (split-K) live in a workspace of `records`
// records; record r, query head h: m (log2 domain running max used),
// l (sum of exp2), acc[D] (unnormalised weighted sum of V).
struct DecodeWorkspace {
  float* m;               // [records, Hq]
  float* l;               // [records, Hq]
  float* acc;             // [records, Hq, D]
  long long* seq_start;   // [S + 1] each sequence's place on the balanced
                          // split's cost line and the line's total (balanced
                          // batches of more than kMergeScanMaxSeqs
                          // sequences), else null
};

// Balanced batches up to this many sequences: every merge CTA scans the
// context lengths itself (before its dependency wait); larger ones read the
// offsets the decode wrote into the workspace.
constexpr int kMergeScanMaxSeqs = 512;

struct DecodeArgs {
  float* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* k_new;      // non-null: write each sequence's new token first (decode step)
  const void* v_new;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  int num_blocks, max_blocks_per_seq;
  float scale;
  int partition_blocks;   // > 0: fixed windows of this many blocks; 0: balanced
  int max_splits;         // fixed mode: ceil(MB / partition_blocks)
  int balanced_ctas;      // balanced mode: CTAs per KV-head group
  int window_ctas;        // fixed mode: CTAs per KV-head group that walk the
                          // windows persistently (0: one CTA per window)
  DecodeWorkspace ws;
  uint32_t* status;
};

// Number of workspace records the decode needs (0 = none).
long long decode_records(int num_seqs, int max_blocks_per_seq, int partition_blocks,
                         int balanced_ctas);
// int64 per-sequence offsets the workspace also holds (0 = none).
long long decode_prefix_entries(int num_seqs, int partition_blocks);
// Byte layout of the workspace for `records` records.
size_t decode_workspace_bytes(long long records, int num_q_heads, int head_dim,
                              long long prefix_entries);
DecodeWorkspace decode_workspace_carve(void* base, long long records, int num_q_heads,
                                       int head_dim, long long prefix_entries);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// One CTA waiting on an mbarrier nothing arrives at (tvl_selftest_bounded_wait).
cudaError_t launch_selftest_wait(uint32_t* status, cudaStream_t stream);

struct PrefillArgs {
  float* out;
  const void* q;
  const int32_t* query_start_loc;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs, total_q_tokens, max_q_len, num_q_heads, num_kv_heads, head_dim;
  int block_size, num_blocks, max_blocks_per_seq;
  float scale;
  uint32_t* status;
  int num_sms;            // the persistent grid's size bound
};
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Sets the calling thread's tvl_last_error() text.
void set_last_error(const char* msg);

}  // namespace tvl
