// prefill.cu -- chunked causal prefill over a paged KV cache on the
// Blackwell tensor cores (tcgen05 MMA, TMEM accumulators, TMA gathers).
//
// What it computes [tiny-vllm README, curriculum "Prefill vs decode",
// "Attention", "GQA", "Causal mask", "Online softmax", "Paged Attention";
// nano-vLLM guide ch. 6 "Prefill vs Decode" (prefill is compute-bound),
// ch. 7 "Prefix Caching", ch. 10 "The Optimization Stack" (FlashAttention)]:
// the Lq new query tokens of a sequence are its last Lq positions; row i at
// absolute position p = ctx - Lq + i attends to cached tokens 0..p.
//
// One CTA = one 128-row query tile of one query head.  Warps:
//   0-3  softmax: thread r owns query row r (TMEM lane r); reads S from TMEM,
//        masks, keeps the running maximum (moved lazily: only when a score
//        exceeds it by more than 2^8, which keeps the result exact), writes
//        P = 2^(S*scale*log2e - m) as fp16 into a 128-byte-swizzled K-major
//        shared tile, converts the V tile bf16 -> fp16 in place (exact for
//        |v| >= 2^-14), rescales O in TMEM when the maximum moved, and finally
//        normalises O and stores it;
//   4    producer: TMA loads of the Q tile and, per 128-key tile, one box of
//        bs tokens x 64 dims per physical block (K and V) found through the
//        block table -- the paged gather; blocks past the context are read
//        out of range so TMA fills them with zeros;
//   5    MMA issuer: S = Q K^T (M 128, N 128, bf16 inputs) into one of two
//        TMEM buffers, then O += P V (M 128, N 64, fp16 inputs), fp32
//        accumulation throughout; completion is signalled with
//        tcgen05.commit on mbarriers.
// P and V go through fp16 rather than bf16 so that rounding P costs at most
// 2^-11 relative (bf16 would cost 2^-8) -- the fp32-accumulated result stays
// within 2e-3 of the exact attention even for rows with few keys.
// TMEM: S0 [0,128), S1 [128,256), O [256,320) of a 512-column allocation.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "device.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace tvl {
namespace {

constexpr int kD = 64;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

constexpr uint32_t kTileBytes = kBM * kD * 2;      // 16 KB: 128 rows x 128 B
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = kQOff + kTileBytes;      // 2 stages
constexpr uint32_t kVOff = kKOff + 2 * kTileBytes;  // 2 stages
constexpr uint32_t kPOff = kVOff + 2 * kTileBytes;  // 2 buffers of 2 x 16 KB
constexpr uint32_t kBarOff = kPOff + 4 * kTileBytes;
constexpr uint32_t kSmemUsed = kBarOff + 256;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1 KB

constexpr uint32_t kIdescQK = idesc_f16_f32acc(1, 0, kBM, kBN);   // bf16, K-major B
constexpr uint32_t kIdescPV = idesc_f16_f32acc(0, 1, kBM, kD);    // fp16, MN-major B

struct Barriers {
  uint64_t q_full;
  uint64_t kv_full[2];
  uint64_t kv_empty[2];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(Barriers) <= 256, "barrier area");

struct Params {
  float* out;
  const int32_t* query_start_loc;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs, total_q, hq, hkv, group, bs, num_blocks, max_blocks, n_qtiles;
  float scale_log2;
  uint32_t* status;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t bf16x2_to_half2(uint32_t w) {
  const float2 f = bf16x2_to_float2(w);
  return pack_half2(f.x, f.y);
}

// Bounded wait that records a timeout in the status word and in the CTA's
// abort flag; returns false when the caller must stop.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Barriers* B,
                                              const Params& p) {
  if (mbar_wait(bar, parity)) return true;
  report(p.status, kDevTimeout);
  atomicExch(&B->abort, 1u);
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Barriers* B = reinterpret_cast<Barriers*>(smem + kBarOff);

  const int qtile = p.n_qtiles - 1 - static_cast<int>(blockIdx.x);   // longest tiles first
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  const int g = h / p.group;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- per-tile geometry (identical in every thread)
  const int q0 = p.query_start_loc[s];
  const int lq = p.query_start_loc[s + 1] - q0;
  int ctx = p.context_lens[s];
  const int cap = p.max_blocks * p.bs;
  if (qtile * kBM >= lq) return;                       // no rows here
  if (ctx < lq || ctx > cap || lq < 0) {
    if (threadIdx.x == 0)
      report(p.status, ctx > cap ? TVL_DEV_BAD_CONTEXT_LEN : TVL_DEV_BAD_QUERY_LEN);
    return;
  }
  const int prefix = ctx - lq;
  const int row0 = qtile * kBM;                         // first row of the tile
  const int rows = min(kBM, lq - row0);                 // valid rows
  const int pos_first = prefix + row0;
  const int pos_last = prefix + row0 + rows - 1;
  const int n_kv = pos_last / kBN + 1;                  // KV tiles to visit
  const int nblk = (ctx + p.bs - 1) / p.bs;
  const int boxes = kBN / p.bs;                         // physical blocks per KV tile

  if (threadIdx.x == 0) {
    mbar_init(&B->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->kv_full[i], 1);
      mbar_init(&B->kv_empty[i], 1);
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->s_free[i], 4);
      mbar_init(&B->p_full[i], 4);
      mbar_init(&B->pv_done[i], 1);
    }
    mbar_init(&B->mma_done, 1);
    B->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&B->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B->tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      mbar_arrive_expect_tx(&B->q_full, kTileBytes);
      tma_load_3d(smem + kQOff, &tm_q, 0, h, q0 + row0, &B->q_full);
    }
    const int32_t* table = p.block_tables + static_cast<long long>(s) * p.max_blocks;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      bool ok = true;
      if (j >= 2 && lane == 0) ok = wait_or_abort(&B->kv_empty[st], ((j - 2) >> 1) & 1, B, p);
      if (__shfl_sync(kFull, ok ? 1 : 0, 0) == 0) break;
      if (lane == 0) mbar_arrive_expect_tx(&B->kv_full[st], 2 * kTileBytes);
      __syncwarp();
      for (int b = lane; b < boxes; b += 32) {
        const int lb = j * boxes + b;                   // logical block
        int phys = p.num_blocks;                        // out of range: zero fill
        if (lb < nblk) {
          phys = table[lb];
          if (phys < 0 || phys >= p.num_blocks) {
            report(p.status, TVL_DEV_BAD_BLOCK_ID);
            phys = p.num_blocks;
          }
        }
        const uint32_t off = static_cast<uint32_t>(b * p.bs) * (kD * 2);
        tma_load_4d(smem + kKOff + st * kTileBytes + off, &tm_k, 0, g, 0, phys, &B->kv_full[st]);
        tma_load_4d(smem + kVOff + st * kTileBytes + off, &tm_v, 0, g, 0, phys, &B->kv_full[st]);
      }
    }
    // the loads of the last (up to) two tiles must land before exit
    if (lane == 0) {
      for (int j = (n_kv > 2 ? n_kv - 2 : 0); j < n_kv; ++j)
        if (!mbar_wait(&B->kv_full[j & 1], (j >> 1) & 1)) report(p.status, kDevTimeout);
      if (!mbar_wait(&B->q_full, 0)) report(p.status, kDevTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_addr(smem + kQOff);
      bool ok = wait_or_abort(&B->q_full, 0, B, p);
      int issued_pv = 0;
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {
          const int st = j & 1;
          ok = wait_or_abort(&B->kv_full[st], (j >> 1) & 1, B, p);
          if (ok && j >= 2) ok = wait_or_abort(&B->s_free[st], ((j - 2) >> 1) & 1, B, p);
          if (!ok) break;
          tc_fence_after();
          const uint32_t k_addr = smem_addr(smem + kKOff + st * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            mma_f16_ss(tmem + st * kBN, desc_sw128(q_addr + kk * 32, 16, 1024),
                       desc_sw128(k_addr + kk * 32, 16, 1024), kIdescQK, kk > 0);
          }
          mma_commit(&B->s_full[st]);
        }
        if (j >= 1) {
          const int jp = j - 1;
          const int st = jp & 1;
          ok = wait_or_abort(&B->p_full[st], (jp >> 1) & 1, B, p);
          if (!ok) break;
          tc_fence_after();
          const uint32_t p_addr = smem_addr(smem + kPOff + st * 2 * kTileBytes);
          const uint32_t v_addr = smem_addr(smem + kVOff + st * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            mma_f16_ss(tmem + kTmemO,
                       desc_sw128(p_addr + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16, 1024),
                       desc_sw128(v_addr + kk * 2048, 16, 1024), kIdescPV, (jp > 0 || kk > 0));
          }
          mma_commit(&B->pv_done[st]);
          mma_commit(&B->kv_empty[st]);
          issued_pv = j;
        }
      }
      // every MMA issued must be complete before TMEM is released
      (void)issued_pv;
      mma_commit(&B->mma_done);
      if (!mbar_wait(&B->mma_done, 0)) report(p.status, kDevTimeout);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x;                          // row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int qpos = pos_first + r;
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int sb = j & 1;
      ok = wait_or_abort(&B->s_full[sb], (j >> 1) & 1, B, p);
      if (__any_sync(kFull, !ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + sb * kBN + c * 32, sr[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->s_free[sb]);

      const int key0 = j * kBN;
      const bool masked = (key0 + kBN - 1 > pos_first) || (key0 + kBN > ctx);
      const int limit = min(qpos, ctx - 1) - key0;     // last visible column
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float v = __uint_as_float(sr[c][e]) * p.scale_log2;
          if (masked && (c * 32 + e) > limit) v = -INFINITY;
          sr[c][e] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + kRescaleLog2;
      if (__any_sync(kFull, need)) {
        const float f = need ? ex2(m_used - m_new) : 1.0f;
        if (j > 0) {
          // O *= f needs the previous P.V to have landed in TMEM
          ok = wait_or_abort(&B->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, B, p);
          if (__any_sync(kFull, !ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + kTmemO + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(tmem + lane_off + kTmemO + c * 32, o);
          }
          tmem_st_wait();
        }
        if (need) {
          m_used = m_new;
          l *= f;
        }
      }
      const float mref = m_used == -INFINITY ? 0.f : m_used;
      if (j >= 2) {   // P buffer sb is free once P.V of tile j-2 completed
        ok = wait_or_abort(&B->pv_done[sb], ((j - 2) >> 1) & 1, B, p);
        if (__any_sync(kFull, !ok)) { ok = false; break; }
      }
      uint8_t* pbuf = smem + kPOff + sb * 2 * kTileBytes;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int c = q >> 2, e0 = (q & 3) * 8;
        float pv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          pv[e] = ex2(__uint_as_float(sr[c][e0 + e]) - mref);
          l += pv[e];
        }
        const uint4 w = make_uint4(pack_half2(pv[0], pv[1]), pack_half2(pv[2], pv[3]),
                                   pack_half2(pv[4], pv[5]), pack_half2(pv[6], pv[7]));
        const int region = q >> 3, chunk = q & 7;
        *reinterpret_cast<uint4*>(pbuf + region * kTileBytes + r * 128 +
                                  ((chunk ^ (r & 7)) << 4)) = w;
      }
      // V tile j: bf16 -> fp16 in place; keys past the context become zero
      ok = wait_or_abort(&B->kv_full[sb], (j >> 1) & 1, B, p);
      if (__any_sync(kFull, !ok)) { ok = false; break; }
      uint8_t* vrow = smem + kVOff + sb * kTileBytes + r * 128;
      const bool key_ok = key0 + r < ctx;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int chunk = i ^ (r & 7);
        uint4 w = *reinterpret_cast<const uint4*>(vrow + chunk * 16);
        if (key_ok) {
          w.x = bf16x2_to_half2(w.x);
          w.y = bf16x2_to_half2(w.y);
          w.z = bf16x2_to_half2(w.z);
          w.w = bf16x2_to_half2(w.w);
        } else {
          w = make_uint4(0, 0, 0, 0);
        }
        *reinterpret_cast<uint4*>(vrow + chunk * 16) = w;
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->p_full[sb]);
    }
    if (ok) {
      const int jl = n_kv - 1;
      ok = wait_or_abort(&B->pv_done[jl & 1], (jl >> 1) & 1, B, p);
    }
    if (!__any_sync(kFull, !ok)) {
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld32(tmem + lane_off + kTmemO, o[0]);
      tmem_ld32(tmem + lane_off + kTmemO + 32, o[1]);
      tmem_ld_wait();
      if (r < rows) {
        const float inv = 1.0f / l;
        float4* dst = reinterpret_cast<float4*>(
            p.out + (static_cast<long long>(q0 + row0 + r) * p.hq + h) * kD);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            dst[c * 8 + e / 4] =
                make_float4(__uint_as_float(o[c][e]) * inv, __uint_as_float(o[c][e + 1]) * inv,
                            __uint_as_float(o[c][e + 2]) * inv,
                            __uint_as_float(o[c][e + 3]) * inv);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD),
                                static_cast<cuuint64_t>(a.num_q_heads),
                                static_cast<cuuint64_t>(a.total_q_tokens)};
    const cuuint64_t strides[2] = {kD * 2, static_cast<cuuint64_t>(a.num_q_heads) * kD * 2};
    const cuuint32_t box[3] = {kD, 1, kBM};
    if (!make_map(&tq, a.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD),
                                static_cast<cuuint64_t>(a.num_kv_heads),
                                static_cast<cuuint64_t>(a.block_size),
                                static_cast<cuuint64_t>(a.num_blocks)};
    const cuuint64_t strides[3] = {
        kD * 2, static_cast<cuuint64_t>(a.num_kv_heads) * kD * 2,
        static_cast<cuuint64_t>(a.block_size) * a.num_kv_heads * kD * 2};
    const cuuint32_t box[4] = {kD, 1, static_cast<cuuint32_t>(a.block_size), 1};
    if (!make_map(&tk, a.k_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map(&tv, a.v_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  Params p;
  p.out = a.out;
  p.query_start_loc = a.query_start_loc;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.num_seqs = a.num_seqs;
  p.total_q = a.total_q_tokens;
  p.hq = a.num_q_heads;
  p.hkv = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.bs = a.block_size;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks_per_seq;
  p.n_qtiles = (a.max_q_len + kBM - 1) / kBM;
  p.scale_log2 = a.scale * kLog2e;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_qtiles, a.num_q_heads, a.num_seqs);
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace tvl
