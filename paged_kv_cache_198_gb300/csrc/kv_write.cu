// kv_write.cu -- the slot-mapped paged KV write.
//
// [tiny-vllm README, curriculum "Paged KV cache"]: each new token's K and V
// rows (Hkv * D bf16 values) are stored at the cache slot the host's block
// allocator chose for it; slot = physical block * bs + offset indexes a row
// of the flat [NB * bs, Hkv * D] view of the cache.
//
// One warp moves one token: its K row and its V row, with 16-byte vector
// loads and stores (a 1 KB row is two 16-byte vectors per lane per tensor).
// The work is a pure copy, bound by HBM bandwidth for large batches and by
// launch latency for small ones.
#include "device.cuh"
#include "kernels.h"

namespace tvl {
namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    kv_write_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                    const int32_t* __restrict__ slot_mapping, int num_tokens, int row_vecs,
                    long long num_slots, uint32_t* status) {
  grid_dependency_wait();        // inputs may come from the preceding kernel
  grid_dependents_launch();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  if (t >= num_tokens) return;
  const long long slot = slot_mapping[t];
  if (slot < 0) return;                      // padding token: nothing to store
  if (slot >= num_slots) {                   // outside the pool: refuse, report
    if (lane == 0) report(status, TVL_DEV_BAD_SLOT);
    return;
  }
  const uint4* ks = k_new + t * row_vecs;
  const uint4* vs = v_new + t * row_vecs;
  uint4* kd = k_cache + slot * row_vecs;
  uint4* vd = v_cache + slot * row_vecs;
  for (int i = lane; i < row_vecs; i += 32) {
    const uint4 kv = __ldcs(ks + i);         // read once: streaming
    const uint4 vv = __ldcs(vs + i);
    kd[i] = kv;
    vd[i] = vv;
  }
}

// One CTA per (pair, cache): block dst of the cache becomes a copy of block
// src, 16-byte vectors.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                       long long block_vecs, int num_blocks, uint32_t* status) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int i = blockIdx.x;
  const int from = src[i];
  const int to = dst[i];
  if (from < 0 || from >= num_blocks || to < 0 || to >= num_blocks) {
    if (threadIdx.x == 0) report(status, TVL_DEV_BAD_BLOCK_ID);
    return;
  }
  uint4* cache = blockIdx.y == 0 ? k_cache : v_cache;
  const uint4* s = cache + from * block_vecs;
  uint4* d = cache + to * block_vecs;
  for (long long v = threadIdx.x; v < block_vecs; v += blockDim.x) d[v] = s[v];
}

// RoPE fused into the paged write [tiny-vllm README, curriculum "RoPE" and
// "Paged KV cache"].  One warp per token; lane i owns the pair
// (x_i, x_{i+D/2}) of every head and rotates it by pos * theta^(-2i/D).
// The angle is formed and reduced modulo 2*pi in double precision (positions
// up to 2^31 keep full accuracy), then sin / cos and the rotation are fp32 and
// the result is rounded to bf16.  q is rotated in place; the rotated K row and
// the V row go to the token's cache slot.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    rope_kv_write_kernel(__nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
                         const uint4* __restrict__ v_new, __nv_bfloat16* __restrict__ k_cache,
                         uint4* __restrict__ v_cache, const int32_t* __restrict__ slot_mapping,
                         const int32_t* __restrict__ positions, int num_tokens, int hq, int hkv,
                         long long num_slots, double log2_theta, uint32_t* status) {
  constexpr int kD = 64, kHalf = 32;
  grid_dependency_wait();
  grid_dependents_launch();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  if (t >= num_tokens) return;
  const long long pos = positions[t];
  const long long slot = slot_mapping[t];
  // angle of pair `lane`, reduced to [-pi, pi] in double precision
  const double inv_freq = exp2(-2.0 * lane / kD * log2_theta);
  const double a = static_cast<double>(pos) * inv_freq;
  const double two_pi = 6.283185307179586476925286766559;
  const double r = fma(-rint(a / two_pi), two_pi, a);
  float sn, cs;
  sincosf(static_cast<float>(r), &sn, &cs);
  auto rotate = [&](const __nv_bfloat16* src, __nv_bfloat16* dst) {
    const float x0 = __bfloat162float(src[lane]);
    const float x1 = __bfloat162float(src[lane + kHalf]);
    const float y0 = fmaf(x0, cs, -x1 * sn);
    const float y1 = fmaf(x1, cs, x0 * sn);
    dst[lane] = __float2bfloat16_rn(y0);
    dst[lane + kHalf] = __float2bfloat16_rn(y1);
  };
  if (q != nullptr) {
    for (int h = 0; h < hq; ++h) {
      __nv_bfloat16* row = q + (t * hq + h) * kD;
      rotate(row, row);
    }
  }
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) report(status, TVL_DEV_BAD_SLOT);
    return;
  }
  for (int h = 0; h < hkv; ++h)
    rotate(k_new + (t * hkv + h) * kD, k_cache + (slot * hkv + h) * kD);
  const int row_vecs = hkv * kD * 2 / 16;
  const uint4* vs = v_new + t * row_vecs;
  uint4* vd = v_cache + slot * row_vecs;
  for (int i = lane; i < row_vecs; i += 32) vd[i] = __ldcs(vs + i);
}

}  // namespace

cudaError_t launch_rope_kv_write(const RopeKvWriteArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int blocks = (a.num_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return launch_pdl(rope_kv_write_kernel, dim3(blocks), dim3(kWarpsPerBlock * 32), 0, stream,
                    static_cast<__nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_new),
                    static_cast<const uint4*>(a.v_new), static_cast<__nv_bfloat16*>(a.k_cache),
                    static_cast<uint4*>(a.v_cache), a.slot_mapping, a.positions, a.num_tokens,
                    a.num_q_heads, a.num_kv_heads, a.num_slots, a.log2_theta, a.status);
}

cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream) {
  if (a.n == 0) return cudaSuccess;
  return launch_pdl(copy_blocks_kernel, dim3(a.n, 2), dim3(256), 0, stream,
                    static_cast<uint4*>(a.k_cache), static_cast<uint4*>(a.v_cache), a.src, a.dst,
                    a.block_bytes / 16, a.num_blocks, a.status);
}

cudaError_t launch_kv_write(const KvWriteArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int blocks = (a.num_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return launch_pdl(kv_write_kernel, dim3(blocks), dim3(kWarpsPerBlock * 32), 0, stream,
                    static_cast<const uint4*>(a.k_new), static_cast<const uint4*>(a.v_new),
                    static_cast<uint4*>(a.k_cache), static_cast<uint4*>(a.v_cache),
                    a.slot_mapping, a.num_tokens, a.row_bytes / 16, a.num_slots, a.status);
}

}  // namespace tvl
