// decode.cu -- PagedAttention decode with online softmax, GQA and split-K.
//
// What it computes [tiny-vllm README, curriculum "Attention", "GQA",
// "Softmax", "Online softmax", "Paged Attention", "Paged Attention CUDA
// kernel"]: for each sequence s and query head h,
//   out[s,h,:] = sum_j softmax_j(scale * q[s,h,:] . K_j) V_j,
// K_j / V_j being token j of KV head h / G, found through the block table
// [nano-vLLM guide ch. 4 "PagedAttention": fixed-size blocks, like pages of
// virtual memory].  Decode is memory-bound [nano-vLLM guide ch. 6 "Prefill vs
// Decode"], so the design streams each cached K/V byte from HBM exactly once.
//
// Work split.  The context of every sequence is cut on physical-block
// boundaries into segments:
//   * balanced mode (partition_size 0): the flattened list of all sequences'
//     blocks is divided evenly over one CTA per SM (per KV-head group), each
//     sequence start counted as one stage's worth of blocks more (it costs a
//     CTA that much), so each CTA streams about the same time's worth of
//     blocks whatever the length mix;
//   * fixed mode (partition_size P): windows of P tokens from position 0,
//     a segment each; with more windows than SMs a persistent grid (one CTA
//     per SM) walks them in equal contiguous ranges, else one CTA each.
// A segment that covers its whole sequence writes the final output; any other
// writes a partial (m, l, acc) record, and merge_kernel combines the records
// of a sequence by log-sum-exp -- the associative form of the online softmax
// (loads of 16 records in flight at once, the batch maximum moving the
// running one; four warps per head when a sequence has many records).
//
// Decode step (tvl_paged_decode_step): the producer of the CTA that streams a
// sequence's last block also writes the step's new token into the cache --
// it loads the new K/V rows when the segment starts and stores them into row
// (ctx - 1) % bs of that block, with a proxy fence, before it issues the
// block's bulk copy -- so the write needs no kernel of its own.
//
// CTA structure.  One producer warp walks the CTA's segments and, per stage
// of 32 tokens (two physical blocks of 16 or one of 32), issues 1-D bulk
// copies (TMA engine) of the blocks' K and V for the CTA's KV heads
// (bs * Hkv * D * 2 contiguous bytes per block when the CTA owns every KV
// head) into a ring of shared-memory stages, with an mbarrier per stage.
// One consumer warp per KV head processes a stage as two 16-token chunks
// whose instruction streams interleave:
//   * q . k with lane = 8 * token_group + dim_chunk: each lane holds 8 dims
//     of the G query heads (fp32, pre-scaled by scale * log2 e) and reads
//     8 dims of 4 tokens per chunk (16-byte shared loads, conflict-free),
//     packed fp32x2 FMAs; the 8-lane partial sums of the 4G (head, token)
//     pairs are reduced with a transposing butterfly (4G/8 values per lane
//     remain; the register order is permuted per lane so no selects are
//     needed);
//   * an online softmax in the exp2 domain, one maximum per 32 tokens, whose
//     running maximum is only moved when a score exceeds it by more than 2^8
//     (exact: the same reference maximum scales numerator and denominator);
//   * p . V with p staged through a per-warp shared buffer as duplicated
//     pairs (p, p), so each fp32x2 FMA takes its operands straight from a
//     16-byte shared load.
// Launch: the kernels use programmatic dependent launch; each waits for its
// predecessor's memory (griddepcontrol.wait) before touching any input, so
// the next kernel's launch and prologue overlap the previous one's tail.
// All waits are bounded; a timeout sets a status bit and the CTA leaves
// after its copies in flight have landed.
#include <cuda_bf16.h>

#include <algorithm>

#include "device.cuh"
#include "kernels.h"

namespace tvl {
namespace {

constexpr int kD = 64;
constexpr uint32_t kRowBytes = kD * 2;   // one head's K or V row of one token
constexpr int kChunk = 16;
constexpr int kStageTokens = 32;
constexpr int kMaxHeadsPerCta = 8;
// KV heads (consumer warps) per CTA: with 9 warps, three share one
// scheduler's register file (<= 168 registers a thread), too few for the
// 8-head groups' q and accumulators; those CTAs take 4 KV heads.
__host__ __device__ constexpr int max_heads_per_cta(int g) { return g >= 8 ? 4 : kMaxHeadsPerCta; }
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kSmemBudget = 224 * 1024;

enum : int { kSegFirst = 1, kSegLast = 2, kTerminate = 4 };

struct StageMeta {
  int seq;
  int valid;    // tokens of this block inside the context
  int flags;
  int record;   // -1: final output, else partial record index
};

struct Params {
  float* out;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const __nv_bfloat16* k_new;     // fused write of each sequence's new token, or null
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_cache_w;       // k_cache / v_cache, writable (fused write only)
  __nv_bfloat16* v_cache_w;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs, hq, hkv, num_blocks, max_blocks;
  int hpc;               // KV heads per CTA == consumer warps
  int stages;
  uint32_t stage_bytes;  // K area + V area + Q area
  float scale_log2;
  int partition_blocks;  // fixed mode when > 0
  int max_splits;
  int balanced_ctas;
  int seg_weight;        // balanced mode: cost of a sequence start, in blocks
  int window_walk;       // fixed mode: a persistent grid walks the windows
  DecodeWorkspace ws;
  uint32_t* status;
};

struct Layout {
  uint32_t barriers, meta, pbuf, sched, total;
};

// Per-warp p buffer: 2 (double buffer) x 2 chunks x 4 token groups x 4G
// (head, token) entries x 2 (duplicated pair).
__host__ __device__ constexpr int kPbufFloats(int g) { return 2 * 2 * 4 * 4 * g * 2; }


__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int stages, uint32_t stage_bytes, int hpc, int g) {
  Layout l;
  uint32_t off = stages * stage_bytes;
  l.barriers = off;
  off += 2 * stages * 8;
  l.meta = align_up(off, 16);
  off = l.meta + stages * sizeof(StageMeta);
  l.pbuf = align_up(off, 16);
  off = l.pbuf + hpc * kPbufFloats(g) * 4;
  l.sched = align_up(off, 16);
  off = l.sched + 64 * 8;
  l.total = off;
  return l;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int load_ctx(const Params& p, int s, int bs) {
  int c = p.context_lens[s];
  const int cap = p.max_blocks * bs;
  if (c < 0 || c > cap) {
    report(p.status, TVL_DEV_BAD_CONTEXT_LEN);
    c = c < 0 ? 0 : cap;
  }
  return c;
}

// Block-wide inclusive scan of one value per thread; every thread gets its
// inclusive prefix and the block total.  All threads must call it.
__device__ void block_scan(long long v, long long& incl, long long& total, long long* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) tmp[lane] = w;
  }
  __syncthreads();
  incl = x + (warp > 0 ? tmp[warp - 1] : 0);
  total = tmp[nw - 1];
  __syncthreads();
}

// The balanced split cuts a cost line into C equal ranges [T*c/C,
// T*(c+1)/C).  On that line every sequence with blocks occupies w + nb
// units: w for its start, then one per block (an empty sequence occupies
// none).  A sequence start costs a CTA about one stage -- a partly filled
// stage at the previous segment's end, the segment's reduction and store,
// the next q -- so w is one stage's worth of blocks, and a CTA that takes
// on sequence starts gets correspondingly fewer blocks.
__host__ __device__ inline long long seq_cost(long long nb, int w) { return nb > 0 ? nb + w : 0; }

// The CTA of the balanced split whose range contains position x of the cost
// line (the largest c with T*c/C <= x).
__host__ __device__ inline long long balanced_cta_of(long long x, long long total, long long ctas) {
  return ((x + 1) * ctas - 1) / total;
}

// Per-CTA schedule written to shared memory by the whole CTA.
struct Schedule {
  int seq0;            // first sequence
  int block0;          // first block inside it
  int seq_end;         // streaming stops at block block_end of sequence
  int block_end;       //   seq_end (seq_end == num_seqs: at the batch's end)
  int cta;             // balanced mode: CTA index inside the KV-head group
};

// ---------------------------------------------------------------- producer

template <int G, int BS>
__device__ void producer(const Params& p, const Schedule& sc, uint8_t* smem, const Layout& L) {
  const int lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.barriers);
  uint64_t* empty = full + p.stages;
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + L.meta);
  const int hg = blockIdx.z;
  const int hpc = p.hpc;
  const bool whole_rows = (hpc == p.hkv);
  constexpr int BPS = BS <= kStageTokens ? kStageTokens / BS : 1;   // blocks per stage
  const uint32_t blk_bytes = BS * hpc * kRowBytes;     // one block, the CTA's heads
  const uint32_t kv_bytes = kStageTokens * hpc * kRowBytes;
  const uint32_t q_bytes = hpc * G * kRowBytes;
  const uint64_t stream_policy = policy_evict_first();
  const uint64_t keep_policy = policy_evict_last();
  const bool fixed = p.partition_blocks > 0;

  long long it = 0;
  bool ok = true;

  // Claims the next stage (waiting until its previous contents were used).
  auto acquire = [&](int& st) -> bool {
    st = static_cast<int>(it % p.stages);
    bool good = true;
    if (it >= p.stages && lane == 0)
      good = mbar_wait(&empty[st], static_cast<uint32_t>(((it / p.stages) - 1) & 1));
    return __shfl_sync(kFull, good ? 1 : 0, 0) != 0;
  };

  int s = sc.seq0;
  long long b = sc.block0;
  bool first_seg = true;
  // A window of 32 sequences: lane i holds the context length of sequence
  // win_base + i and the ids of its first two blocks (those it has), so a
  // segment that starts a sequence issues its first stage without waiting
  // for a table load of its own -- with many short sequences that load was
  // one memory round trip per sequence.
  int win_base = -1000000;
  int win_ctx = 0, win_t0 = 0, win_t1 = 0;
  while (ok && s < p.num_seqs && (s < sc.seq_end || (s == sc.seq_end && b < sc.block_end))) {
    if (s - win_base >= 32 || s < win_base) {
      win_base = s;
      const bool here = s + lane < p.num_seqs;
      win_ctx = here ? load_ctx(p, s + lane, BS) : 0;
      const int32_t* row = p.block_tables + static_cast<long long>(s + lane) * p.max_blocks;
      win_t0 = here && win_ctx > 0 ? row[0] : 0;
      win_t1 = here && win_ctx > BS && BS <= kStageTokens / 2 ? row[1] : 0;
    }
    const int ctx = __shfl_sync(kFull, win_ctx, s - win_base);
    const int wl = s - win_base;                        // this sequence's window lane
    const long long nb = (ctx + BS - 1) / BS;
    if (b >= nb) {
      ++s;
      b = 0;
      continue;
    }
    long long e = (s == sc.seq_end && sc.block_end < nb) ? sc.block_end : nb;
    int record;
    if (fixed) {
      // one segment per window: its record is (sequence, window), or none
      // when the sequence has a single window
      const long long win = b / p.partition_blocks;
      const long long wend = (win + 1) * p.partition_blocks;
      if (wend < e) e = wend;
      record = nb <= p.partition_blocks ? -1
                                        : static_cast<int>(s * static_cast<long long>(p.max_splits) + win);
    } else {
      record = (b == 0 && e == nb) ? -1 : 2 * sc.cta + (first_seg ? 0 : 1);
    }
    const int32_t* table = p.block_tables + static_cast<long long>(s) * p.max_blocks;
    int tbl = 0;
    // Fused write: when this segment holds the sequence's last block, fetch
    // the new token's K/V rows (this CTA's heads) now, so the loads have
    // landed by the time the last block's stage is issued.
    static_assert(kMaxHeadsPerCta * kRowBytes / 16 <= 64, "two 16-byte pieces a lane");
    const int wchunks = hpc * kRowBytes / 16;          // 16-byte pieces per row, <= 64
    uint4 wk[2], wv[2];
    const bool fused_write = p.k_new != nullptr && e == nb;
    if (fused_write) {
      const size_t src = (static_cast<size_t>(s) * p.hkv + hg * hpc) * kD;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int c = lane + 32 * i;
        if (c < wchunks) {
          wk[i] = reinterpret_cast<const uint4*>(p.k_new + src)[c];
          wv[i] = reinterpret_cast<const uint4*>(p.v_new + src)[c];
        }
      }
    }
    if constexpr (BS > kStageTokens) {
      // Blocks larger than a stage: each block is streamed as BS / 32 stages
      // of 32 tokens (the last block only as far as the context reaches).
      constexpr int kSubPerBlock = BS / kStageTokens;
      for (long long blk = b; blk < e && ok; ++blk) {
        const int slot = static_cast<int>((blk - b) & 31);
        if (slot == 0) tbl = (blk + lane < e) ? table[blk + lane] : 0;
        int phys;
        if (blk == 0)
          phys = __shfl_sync(kFull, win_t0, wl);        // from the window
        else
          phys = __shfl_sync(kFull, tbl, slot);
        bool phys_ok = true;
        if (phys < 0 || phys >= p.num_blocks) {
          if (lane == 0) report(p.status, TVL_DEV_BAD_BLOCK_ID);
          phys = 0;
          phys_ok = false;
        }
        const long long tok0 = blk * BS;                // first token of the block
        const int nsub = blk == nb - 1
                             ? static_cast<int>((ctx - tok0 + kStageTokens - 1) / kStageTokens)
                             : kSubPerBlock;
        for (int sub = 0; sub < nsub && ok; ++sub) {
          int st;
          if (!acquire(st)) {
            ok = false;
            break;
          }
          const int t0 = sub * kStageTokens;            // first token of the stage in the block
          const bool first = (blk == b && sub == 0);
          const bool last_stage = (blk == e - 1 && sub == nsub - 1);
          uint8_t* kdst = smem + static_cast<size_t>(st) * p.stage_bytes;
          uint8_t* vdst = kdst + kv_bytes;
          uint8_t* qdst = vdst + kv_bytes;
          if (lane == 0) {
            StageMeta m;
            m.seq = s;
            const long long rem = ctx - tok0 - t0;
            m.valid = static_cast<int>(rem < kStageTokens ? rem : kStageTokens);
            m.flags = (first ? kSegFirst : 0) | (last_stage ? kSegLast : 0);
            m.record = record;
            meta[st] = m;
            mbar_arrive_expect_tx(&full[st], 2 * kv_bytes + (first ? q_bytes : 0));
          }
          if (fused_write && blk == nb - 1 && phys_ok &&
              sub == static_cast<int>((ctx - 1 - tok0) / kStageTokens)) {
            // the new token's rows, stored before this stage's copy reads them
            const size_t row =
                ((static_cast<size_t>(phys) * BS + (ctx - 1 - tok0)) * p.hkv + hg * hpc) * kD;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int c = lane + 32 * i;
              if (c < wchunks) {
                reinterpret_cast<uint4*>(p.k_cache_w + row)[c] = wk[i];
                reinterpret_cast<uint4*>(p.v_cache_w + row)[c] = wv[i];
              }
            }
            asm volatile("fence.proxy.async;" ::: "memory");
            __syncwarp();
            asm volatile("fence.proxy.async;" ::: "memory");
          }
          __syncwarp();
          if (whole_rows) {
            if (lane == 0) {                            // 32 contiguous token rows
              const size_t off = (static_cast<size_t>(phys) * BS + t0) * p.hkv * kD;
              bulk_load(kdst, p.k_cache + off, kv_bytes, &full[st], stream_policy);
              bulk_load(vdst, p.v_cache + off, kv_bytes, &full[st], stream_policy);
            }
          } else {
            const int t = lane;                         // one token row per lane
            const size_t off =
                ((static_cast<size_t>(phys) * BS + t0 + t) * p.hkv + hg * hpc) * kD;
            bulk_load(kdst + t * hpc * kRowBytes, p.k_cache + off, hpc * kRowBytes, &full[st],
                      stream_policy);
            bulk_load(vdst + t * hpc * kRowBytes, p.v_cache + off, hpc * kRowBytes, &full[st],
                      stream_policy);
          }
          if (first && lane == 31) {
            const size_t off = (static_cast<size_t>(s) * p.hq + hg * hpc * G) * kD;
            bulk_load(qdst, p.q + off, q_bytes, &full[st], keep_policy);
          }
          ++it;
        }
      }
    } else
    for (long long blk = b; blk < e && ok; blk += BPS) {
      const int slot = static_cast<int>((blk - b) & 31);   // BPS divides 32
      if (slot == 0) tbl = (blk + lane < e) ? table[blk + lane] : 0;
      const int nstage = (e - blk < BPS) ? static_cast<int>(e - blk) : BPS;
      int phys[BPS];
      bool last_ok = true;                               // stage's last block id valid
#pragma unroll
      for (int i = 0; i < BPS; ++i) {
        if (blk == 0)                                    // the sequence's first stage:
          phys[i] = __shfl_sync(kFull, i == 0 ? win_t0 : win_t1, wl);   // from the window
        else
          phys[i] = __shfl_sync(kFull, tbl, slot + i);
        if (i < nstage && (phys[i] < 0 || phys[i] >= p.num_blocks)) {
          if (lane == 0) report(p.status, TVL_DEV_BAD_BLOCK_ID);
          phys[i] = 0;
          if (i == nstage - 1) last_ok = false;
        }
      }
      int st;
      if (!acquire(st)) {
        ok = false;
        break;
      }
      const bool first = (blk == b);
      const int flags = (first ? kSegFirst : 0) | (blk + nstage >= e ? kSegLast : 0);
      uint8_t* kdst = smem + static_cast<size_t>(st) * p.stage_bytes;
      uint8_t* vdst = kdst + kv_bytes;
      uint8_t* qdst = vdst + kv_bytes;
      if (lane == 0) {
        StageMeta m;
        m.seq = s;
        const long long rem = ctx - blk * BS;
        const long long cap = static_cast<long long>(nstage) * BS;
        m.valid = static_cast<int>(rem < cap ? rem : cap);
        m.flags = flags;
        m.record = record;
        meta[st] = m;
        mbar_arrive_expect_tx(&full[st], 2 * nstage * blk_bytes + (first ? q_bytes : 0));
      }
      if (fused_write && blk + nstage == nb && last_ok) {
        // The new token (position ctx - 1: the last block's row
        // (ctx - 1) % BS) goes into the cache before the block is copied:
        // generic stores, then a proxy fence so that the bulk copy (async
        // proxy) reads them.
        const int last = nstage == 1 ? phys[0] : phys[BPS - 1];
        const size_t row =
            ((static_cast<size_t>(last) * BS + (ctx - 1) % BS) * p.hkv + hg * hpc) * kD;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = lane + 32 * i;
          if (c < wchunks) {
            reinterpret_cast<uint4*>(p.k_cache_w + row)[c] = wk[i];
            reinterpret_cast<uint4*>(p.v_cache_w + row)[c] = wv[i];
          }
        }
        asm volatile("fence.proxy.async;" ::: "memory");
        __syncwarp();
        asm volatile("fence.proxy.async;" ::: "memory");
      }
      __syncwarp();
      if (whole_rows) {
        if (lane < nstage) {
          int mine = phys[0];
          if constexpr (BPS > 1) {
            if (lane == 1) mine = phys[BPS - 1];
          }
          const size_t off = static_cast<size_t>(mine) * BS * p.hkv * kD;
          bulk_load(kdst + lane * blk_bytes, p.k_cache + off, blk_bytes, &full[st],
                    stream_policy);
          bulk_load(vdst + lane * blk_bytes, p.v_cache + off, blk_bytes, &full[st],
                    stream_policy);
        }
      } else {
        for (int t = lane; t < nstage * BS; t += 32) {
          int mine = phys[0];
          if constexpr (BPS > 1) {
            if (t >= BS) mine = phys[BPS - 1];
          }
          const size_t off =
              (static_cast<size_t>(mine) * BS * p.hkv + (t % BS) * p.hkv + hg * hpc) * kD;
          bulk_load(kdst + t * hpc * kRowBytes, p.k_cache + off, hpc * kRowBytes, &full[st],
                    stream_policy);
          bulk_load(vdst + t * hpc * kRowBytes, p.v_cache + off, hpc * kRowBytes, &full[st],
                    stream_policy);
        }
      }
      if (first && lane == 31) {
        const size_t off = (static_cast<size_t>(s) * p.hq + hg * hpc * G) * kD;
        bulk_load(qdst, p.q + off, q_bytes, &full[st], keep_policy);
      }
      ++it;
    }
    first_seg = false;
    b = e;                 // the next window of this sequence, or the next sequence
    if (b >= nb) {
      ++s;
      b = 0;
    }
  }
  // Tell the consumers to stop.
  int st;
  if (ok && acquire(st)) {
    if (lane == 0) {
      meta[st].flags = kTerminate;
      mbar_arrive(&full[st]);
    }
    ++it;
  } else {
    if (lane == 0) report(p.status, kDevTimeout);
  }
  // Copies still in flight must land before the CTA may exit.
  if (lane == 0) {
    for (int i = 0; i < p.stages; ++i) {
      if (it <= i) break;
      const long long last = i + ((it - 1 - i) / p.stages) * p.stages;   // last fill of stage i
      if (!mbar_wait(&full[i], static_cast<uint32_t>((last / p.stages) & 1))) {
        report(p.status, kDevTimeout);
      }
    }
  }
}

// --------------------------------------------------------------- consumers

template <int G>
struct LaneMap {
  // After the butterfly, lane c (0..7) of a token group holds kVals values
  // with logical indices jbase + r, where j = 4 * head + token.
  static constexpr int kVals = G >= 2 ? G / 2 : 1;
  __device__ static int xor_mask(int c) { return G >= 2 ? c * (G / 2) : (c >> 1); }
  __device__ static int jbase(int c) { return G >= 2 ? c * (G / 2) : (c >> 1); }
  // dim-chunk lane c holding head h after the butterfly
  __device__ static int src_c(int h) { return G >= 2 ? h * 8 / G : 0; }
};

template <int G>
__device__ __forceinline__ float reduce_max_head(float x) {
  x = fmaxf(x, __shfl_xor_sync(kFull, x, 8));
  x = fmaxf(x, __shfl_xor_sync(kFull, x, 16));
  if constexpr (G == 4) x = fmaxf(x, __shfl_xor_sync(kFull, x, 1));
  if constexpr (G == 2) {
    x = fmaxf(x, __shfl_xor_sync(kFull, x, 1));
    x = fmaxf(x, __shfl_xor_sync(kFull, x, 2));
  }
  if constexpr (G == 1) {
    x = fmaxf(x, __shfl_xor_sync(kFull, x, 2));
    x = fmaxf(x, __shfl_xor_sync(kFull, x, 4));
  }
  return x;
}

template <int G>
__device__ __forceinline__ float reduce_sum_head(float x) {
  x += __shfl_xor_sync(kFull, x, 8);
  x += __shfl_xor_sync(kFull, x, 16);
  if constexpr (G == 4) x += __shfl_xor_sync(kFull, x, 1);
  if constexpr (G == 2) {
    x += __shfl_xor_sync(kFull, x, 1);
    x += __shfl_xor_sync(kFull, x, 2);
  }
  if constexpr (G == 1) {   // only even dim-chunk lanes carry a (duplicated) value
    x += __shfl_xor_sync(kFull, x, 1);
    x += __shfl_xor_sync(kFull, x, 2);
    x += __shfl_xor_sync(kFull, x, 4);
  }
  return x;
}

template <int G>
struct ConsumerState {
  float2 qf[G][4];    // q of head (hr ^ mh), dims 8c..8c+7, scaled by scale*log2e
  float2 acc[G][4];   // unnormalised output of head h, dims 8c..8c+7 (this lane's tokens)
  float m_used;       // reference maximum of this lane's head
  float l_part;       // this lane's share of the softmax denominator
};

// NCH 16-token chunks of a stage, starting at chunk chunk0 (tokens
// [16 * chunk0, 16 * (chunk0 + NCH)) of the stage; `valid` counts tokens from
// the stage start); kFull: every one of those tokens is inside the context.
template <int G, int NCH, bool kFull>
__device__ __forceinline__ void process_stage(ConsumerState<G>& st, const uint8_t* kbase,
                                              const uint8_t* vbase, int valid, int hpc, int w,
                                              float* pbuf, int chunk0 = 0) {
  using M = LaneMap<G>;
  const int lane = threadIdx.x & 31;
  const int c = lane & 7, tg = lane >> 3;
  const int mi = M::xor_mask(c) & 3;
  constexpr int N = 4 * G;
  constexpr int R = M::kVals;
  const int jb = M::jbase(c);

  // --- scores: part[ch][4*hr + ir] = q(head hr^mh) . k(token ir^mi) over 8 dims
  float part[NCH][N];
#pragma unroll
  for (int ir = 0; ir < 4; ++ir) {
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      const int t = (chunk0 + ch) * kChunk + tg * 4 + (ir ^ mi);
      const uint4 kw =
          *reinterpret_cast<const uint4*>(kbase + (t * hpc + w) * kRowBytes + c * 16);
      const float2 k0 = bf16x2_to_float2(kw.x), k1 = bf16x2_to_float2(kw.y);
      const float2 k2 = bf16x2_to_float2(kw.z), k3 = bf16x2_to_float2(kw.w);
#pragma unroll
      for (int hr = 0; hr < G; ++hr) {
        float2 a = __fmul2_rn(st.qf[hr][0], k0);
        a = __ffma2_rn(st.qf[hr][1], k1, a);
        a = __ffma2_rn(st.qf[hr][2], k2, a);
        a = __ffma2_rn(st.qf[hr][3], k3, a);
        part[ch][4 * hr + ir] = a.x + a.y;
      }
    }
  }
  // --- transposing butterfly over the 8 dim-chunk lanes
  if constexpr (G >= 2) {
#pragma unroll
    for (int k = 0; k < N / 2; ++k)
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        part[ch][k] += __shfl_xor_sync(kFull, part[ch][k + N / 2], 4);
#pragma unroll
    for (int k = 0; k < N / 4; ++k)
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        part[ch][k] += __shfl_xor_sync(kFull, part[ch][k + N / 4], 2);
#pragma unroll
    for (int k = 0; k < N / 8; ++k)
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        part[ch][k] += __shfl_xor_sync(kFull, part[ch][k + N / 8], 1);
  } else {
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      part[ch][0] += __shfl_xor_sync(kFull, part[ch][2], 4);
      part[ch][1] += __shfl_xor_sync(kFull, part[ch][3], 4);
      part[ch][0] += __shfl_xor_sync(kFull, part[ch][1], 2);
      part[ch][0] += __shfl_xor_sync(kFull, part[ch][0], 1);
    }
  }
  if constexpr (!kFull) {
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int t = (chunk0 + ch) * kChunk + tg * 4 + ((jb + r) & 3);
        if (t >= valid) part[ch][r] = -INFINITY;
      }
  }
  // --- online softmax (exp2 domain, lazily moved reference maximum)
  float cm = part[0][0];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
    for (int r = 0; r < R; ++r) cm = fmaxf(cm, part[ch][r]);
  cm = reduce_max_head<G>(cm);
  if (__any_sync(kFull, cm > st.m_used + kRescaleLog2)) {
    const float m_new = fmaxf(st.m_used, cm);
    const float f = ex2(st.m_used - m_new);
    st.m_used = m_new;
    st.l_part *= f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float fh = __shfl_sync(kFull, f, tg * 8 + M::src_c(h));
      const float2 ff = make_float2(fh, fh);
#pragma unroll
      for (int k = 0; k < 4; ++k) st.acc[h][k] = __fmul2_rn(st.acc[h][k], ff);
    }
  }
  // p as duplicated pairs: pbuf[ch][tg][j = 4*head + token][2]
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    float pr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      pr[r] = ex2(part[ch][r] - st.m_used);
      if (G > 1 || (c & 1) == 0) st.l_part += pr[r];
    }
    float* pb = pbuf + ((chunk0 + ch) * 4 + tg) * N * 2 + jb * 2;
    if constexpr (R == 4) {
      reinterpret_cast<float4*>(pb)[0] = make_float4(pr[0], pr[0], pr[1], pr[1]);
      reinterpret_cast<float4*>(pb)[1] = make_float4(pr[2], pr[2], pr[3], pr[3]);
    } else if constexpr (R == 2) {
      *reinterpret_cast<float4*>(pb) = make_float4(pr[0], pr[0], pr[1], pr[1]);
    } else {
      *reinterpret_cast<float2*>(pb) = make_float2(pr[0], pr[0]);
    }
  }
  __syncwarp();
  // --- o += p . V
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const float* pb = pbuf + ((chunk0 + ch) * 4 + tg) * N * 2;
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
      const int t0 = (chunk0 + ch) * kChunk + tg * 4 + i;
      uint4 vw0 = *reinterpret_cast<const uint4*>(vbase + (t0 * hpc + w) * kRowBytes + c * 16);
      uint4 vw1 =
          *reinterpret_cast<const uint4*>(vbase + ((t0 + 1) * hpc + w) * kRowBytes + c * 16);
      if constexpr (!kFull) {   // slots past the context may hold anything
        if (t0 >= valid) vw0 = make_uint4(0, 0, 0, 0);
        if (t0 + 1 >= valid) vw1 = make_uint4(0, 0, 0, 0);
      }
      const float2 a0 = bf16x2_to_float2(vw0.x), a1 = bf16x2_to_float2(vw0.y);
      const float2 a2 = bf16x2_to_float2(vw0.z), a3 = bf16x2_to_float2(vw0.w);
      const float2 b0 = bf16x2_to_float2(vw1.x), b1 = bf16x2_to_float2(vw1.y);
      const float2 b2 = bf16x2_to_float2(vw1.z), b3 = bf16x2_to_float2(vw1.w);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 pp = *reinterpret_cast<const float4*>(pb + (4 * h + i) * 2);
        const float2 p0 = make_float2(pp.x, pp.y), p1 = make_float2(pp.z, pp.w);
        st.acc[h][0] = __ffma2_rn(p0, a0, st.acc[h][0]);
        st.acc[h][1] = __ffma2_rn(p0, a1, st.acc[h][1]);
        st.acc[h][2] = __ffma2_rn(p0, a2, st.acc[h][2]);
        st.acc[h][3] = __ffma2_rn(p0, a3, st.acc[h][3]);
        st.acc[h][0] = __ffma2_rn(p1, b0, st.acc[h][0]);
        st.acc[h][1] = __ffma2_rn(p1, b1, st.acc[h][1]);
        st.acc[h][2] = __ffma2_rn(p1, b2, st.acc[h][2]);
        st.acc[h][3] = __ffma2_rn(p1, b3, st.acc[h][3]);
      }
    }
  }
}

// Ends a segment: the lanes' partial outputs are summed over the four token
// groups and stored, normalised (record < 0) or as a partial record.  The
// sum is a transposing reduction: a lane's 8G values form one flat array
// (index (4h + k) * 2 + component); across the xor-16 pair each lane keeps
// one half and sends the other, across the xor-8 pair one quarter, so token
// group tg ends with the flat indices [2G tg, 2G (tg + 1)) summed -- 6G
// shuffles instead of 16G, and the lanes of one dim chunk hold disjoint
// parts of the output.
template <int G>
__device__ __forceinline__ void finish_segment(ConsumerState<G>& st, const Params& p, int seq,
                                               int record, int hq0) {
  using M = LaneMap<G>;
  const int lane = threadIdx.x & 31;
  const int c = lane & 7, tg = lane >> 3;
  constexpr int V = 8 * G;                      // values a lane holds
  constexpr int Q = V / 4;                      // values a lane keeps
  const float lt = reduce_sum_head<G>(st.l_part);
  float a[V];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      a[(4 * h + k) * 2] = st.acc[h][k].x;
      a[(4 * h + k) * 2 + 1] = st.acc[h][k].y;
    }
  const bool hi2 = (tg & 2) != 0, hi1 = (tg & 1) != 0;
#pragma unroll
  for (int i = 0; i < V / 2; ++i) {
    const float send = hi2 ? a[i] : a[i + V / 2];
    const float keep = hi2 ? a[i + V / 2] : a[i];
    a[i] = keep + __shfl_xor_sync(kFull, send, 16);
  }
#pragma unroll
  for (int i = 0; i < Q; ++i) {
    const float send = hi1 ? a[i] : a[i + Q];
    const float keep = hi1 ? a[i + Q] : a[i];
    a[i] = keep + __shfl_xor_sync(kFull, send, 8);
  }
  // a[i] is flat index Q * tg + i: head (Q tg + i) / 8, dim 8c + (Q tg + i) % 8
  constexpr int HL = Q >= 8 ? Q / 8 : 1;        // heads this lane holds
  constexpr int W = Q >= 8 ? 8 : Q;             // values per held head
#pragma unroll
  for (int j = 0; j < HL; ++j) {
    const int h = (Q * tg) / 8 + j;
    const int d0 = 8 * c + (Q >= 8 ? 0 : (Q * tg) % 8);
    const float lh = __shfl_sync(kFull, lt, tg * 8 + M::src_c(h));
    const float mh = __shfl_sync(kFull, st.m_used, tg * 8 + M::src_c(h));
    const long long row = static_cast<long long>(record < 0 ? seq : record) * p.hq + hq0 + h;
    const float sc = record < 0 ? 1.0f / lh : 1.0f;
    float* dst = (record < 0 ? p.out : p.ws.acc) + row * kD + d0;
    const float* v = a + j * W;
    if constexpr (W == 8) {
      reinterpret_cast<float4*>(dst)[0] = make_float4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
      reinterpret_cast<float4*>(dst)[1] = make_float4(v[4] * sc, v[5] * sc, v[6] * sc, v[7] * sc);
    } else if constexpr (W == 4) {
      reinterpret_cast<float4*>(dst)[0] = make_float4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
    } else {
      reinterpret_cast<float2*>(dst)[0] = make_float2(v[0] * sc, v[1] * sc);
    }
    if (record >= 0 && c == 0 && (Q >= 8 || (Q * tg) % 8 == 0)) {
      p.ws.m[row] = mh;
      p.ws.l[row] = lh;
    }
  }
}

template <int G, int BS>
__device__ void consumer(const Params& p, uint8_t* smem, const Layout& L) {
  using M = LaneMap<G>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = lane & 7;
  const int w = warp;
  const int hpc = p.hpc;
  const int kvh = blockIdx.z * hpc + w;
  const int hq0 = kvh * G;
  const int mh = M::xor_mask(c) >> 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.barriers);
  uint64_t* empty = full + p.stages;
  const StageMeta* meta = reinterpret_cast<const StageMeta*>(smem + L.meta);
  float* pbuf_w = reinterpret_cast<float*>(smem + L.pbuf) + w * kPbufFloats(G);
  const uint32_t kv_bytes = kStageTokens * hpc * kRowBytes;

  ConsumerState<G> st;
  st.m_used = -INFINITY;
  st.l_part = 0.f;
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      st.acc[h][k] = make_float2(0.f, 0.f);
      st.qf[h][k] = make_float2(0.f, 0.f);
    }
  int stage_no = 0;
  for (long long it = 0;; ++it) {
    const int s = static_cast<int>(it % p.stages);
    if (!mbar_wait(&full[s], static_cast<uint32_t>((it / p.stages) & 1))) {
      if (lane == 0) report(p.status, kDevTimeout);
      return;
    }
    const StageMeta md = meta[s];
    if (md.flags & kTerminate) break;
    const uint8_t* kbase = smem + static_cast<size_t>(s) * p.stage_bytes;
    const uint8_t* vbase = kbase + kv_bytes;
    if (md.flags & kSegFirst) {
      const uint8_t* qbase = vbase + kv_bytes;
      st.m_used = -INFINITY;
      st.l_part = 0.f;
#pragma unroll
      for (int hr = 0; hr < G; ++hr) {
        const uint4 qw = *reinterpret_cast<const uint4*>(qbase + (w * G + (hr ^ mh)) * kRowBytes +
                                                         c * 16);
        const float2 sl = make_float2(p.scale_log2, p.scale_log2);
        st.qf[hr][0] = __fmul2_rn(bf16x2_to_float2(qw.x), sl);
        st.qf[hr][1] = __fmul2_rn(bf16x2_to_float2(qw.y), sl);
        st.qf[hr][2] = __fmul2_rn(bf16x2_to_float2(qw.z), sl);
        st.qf[hr][3] = __fmul2_rn(bf16x2_to_float2(qw.w), sl);
#pragma unroll
        for (int k = 0; k < 4; ++k) st.acc[hr][k] = make_float2(0.f, 0.f);
      }
    }
    float* pb = pbuf_w + (stage_no & 1) * (kPbufFloats(G) / 2);
    if (md.valid > kChunk) {
      if constexpr (G <= 4) {     // both chunks at once: twice the independent work
        if (md.valid >= kStageTokens)
          process_stage<G, 2, true>(st, kbase, vbase, md.valid, hpc, w, pb);
        else
          process_stage<G, 2, false>(st, kbase, vbase, md.valid, hpc, w, pb);
      } else {                    // G = 8 would run out of registers: one at a time
        process_stage<G, 1, true>(st, kbase, vbase, md.valid, hpc, w, pb, 0);
        if (md.valid >= kStageTokens)
          process_stage<G, 1, true>(st, kbase, vbase, md.valid, hpc, w, pb, 1);
        else
          process_stage<G, 1, false>(st, kbase, vbase, md.valid, hpc, w, pb, 1);
      }
    } else {
      if (md.valid >= kChunk)
        process_stage<G, 1, true>(st, kbase, vbase, md.valid, hpc, w, pb);
      else
        process_stage<G, 1, false>(st, kbase, vbase, md.valid, hpc, w, pb);
    }
    ++stage_no;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (md.flags & kSegLast) finish_segment<G>(st, p, md.seq, md.record, hq0);
  }
}

// ------------------------------------------------------------------ kernel

// Schedule of a balanced CTA in a batch of more sequences than threads (or
// when the merge wants every sequence's place): kept out of line so that its
// code does not share the kernel body's instruction-cache footprint.
template <int BS>
__device__ __noinline__ void schedule_large(const Params& p, Schedule* sched, long long* tmp,
                                            uint8_t* smem) {
  const int tid = threadIdx.x;
  const int cta = blockIdx.x;
  const int w = p.seg_weight;
  long long total = 0, lo = 0, hi = 0;
  // larger batches: each thread sums the costs of a contiguous slice of
  // the sequences, one block-wide scan gives every slice's place on the
  // cost line and the total, and the threads whose slices hold positions
  // T*c/C and T*(c+1)/C walk them again to find the sequence and block:
  // O(S / threads) work a thread and one scan, whatever the batch size
  const int nthreads = static_cast<int>(blockDim.x);
  const int per = (p.num_seqs + nthreads - 1) / nthreads;
  const int s_lo = min(p.num_seqs, tid * per);
  const int s_hi = min(p.num_seqs, s_lo + per);
  // Slices of more than 8 sequences: the costs are staged in the stage
  // memory (idle until the producer starts) with coalesced loads, since a
  // slice read straight from global memory makes every warp load touch 32
  // cache lines, 8 of them in flight at a time.  Staged costs and in-slice
  // offsets are 32-bit; batches whose figures could exceed that, or that do
  // not fit, read global memory instead.
  int32_t* cst_tab = reinterpret_cast<int32_t*>(smem);
  const uint32_t tab_bytes = align_up(static_cast<uint32_t>(p.num_seqs) * 4u, 8u);
  const bool staged =
      per > 8 &&
      static_cast<long long>(p.num_seqs) * 4 + 8LL * nthreads + 8 <=
          static_cast<long long>(p.stages) * p.stage_bytes &&
      static_cast<long long>(per) * (static_cast<long long>(p.max_blocks) + w) < (1LL << 31);
  if (staged) {
    // 8 coalesced lengths in flight per thread
    for (int i0 = tid; i0 < p.num_seqs; i0 += 8 * nthreads) {
      int c8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * nthreads;
        c8[u] = i < p.num_seqs ? load_ctx(p, i, BS) : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * nthreads;
        if (i < p.num_seqs) cst_tab[i] = static_cast<int32_t>(seq_cost((c8[u] + BS - 1) / BS, w));
      }
    }
    __syncthreads();
  }
  // the slice's costs 8 at a time (from global memory: 8 lengths in
  // flight, one memory round trip per 8 sequences)
  auto costs8 = [&](int s0, long long (&cst)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      cst[u] = s0 + u >= s_hi ? 0
               : staged       ? static_cast<long long>(cst_tab[s0 + u])
                              : seq_cost((load_ctx(p, s0 + u, BS) + BS - 1) / BS, w);
  };
  long long mine = 0;
  for (int s0 = s_lo; s0 < s_hi; s0 += 8) {
    long long cst[8];
    costs8(s0, cst);
#pragma unroll
    for (int u = 0; u < 8; ++u) mine += cst[u];
  }
  long long incl;
  block_scan(mine, incl, total, tmp);
  const long long excl = incl - mine;
  lo = total * cta / p.balanced_ctas;
  hi = total * (cta + 1) / p.balanced_ctas;
  if (tid == 0) {
    sched->seq0 = p.num_seqs;
    sched->block0 = 0;
    sched->seq_end = p.num_seqs;
    sched->block_end = 0;
    sched->cta = cta;
  }
  __syncthreads();
  // position x of the cost line -> (sequence, block), walking this slice
  auto locate = [&](long long x, int& seq, int& blk) {
    long long run = excl;
    for (int s0 = s_lo; s0 < s_hi; s0 += 8) {
      long long cst[8];
      costs8(s0, cst);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (s0 + u < s_hi && x < run + cst[u]) {
          seq = s0 + u;
          blk = static_cast<int>(x - run - w > 0 ? x - run - w : 0);
          return;
        }
        run += cst[u];
      }
    }
  };
  if (lo < total && mine > 0 && excl <= lo && lo < excl + mine)
    locate(lo, sched->seq0, sched->block0);
  if (hi < total && mine > 0 && excl <= hi && hi < excl + mine)
    locate(hi, sched->seq_end, sched->block_end);
  // batches past kMergeScanMaxSeqs: every sequence's place on the cost
  // line (and the total) for the merge, which then scans nothing
  if (p.ws.seq_start != nullptr && cta == 0 && blockIdx.z == 0) {
    if (staged) {
      // each slice's costs become offsets inside the slice (in place,
      // after this thread's own walks); then one coalesced pass adds the
      // slices' places and writes them out
      long long* slice_at = reinterpret_cast<long long*>(smem + tab_bytes);
      slice_at[tid] = excl;
      int32_t run = 0;
      for (int s2 = s_lo; s2 < s_hi; ++s2) {
        const int32_t c2 = cst_tab[s2];
        cst_tab[s2] = run;
        run += c2;
      }
      __syncthreads();
      for (int i = tid; i < p.num_seqs; i += nthreads)
        p.ws.seq_start[i] = slice_at[i / per] + cst_tab[i];
    } else {
      long long run = excl;
      for (int s0 = s_lo; s0 < s_hi; s0 += 8) {
        long long cst[8];
        costs8(s0, cst);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (s0 + u < s_hi) p.ws.seq_start[s0 + u] = run;
          run += cst[u];
        }
      }
    }
    if (tid == 0) p.ws.seq_start[p.num_seqs] = total;
  }
  // the generic writes to the stage memory are ordered before the bulk
  // copies (async proxy) that will fill it
  if (staged) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Fixed windows walked by a persistent grid: the windows of all sequences,
// in (sequence, window) order, are dealt to the C CTAs in equal contiguous
// ranges; a CTA streams its windows one after the other (a segment and a
// record each), so its copies run on across window boundaries instead of a
// CTA starting, filling its ring and draining it for every window.  Out of
// line, like schedule_large.
template <int BS>
__device__ __noinline__ void schedule_windows(const Params& p, Schedule* sched, long long* tmp) {
  const int tid = threadIdx.x;
  const int nthreads = static_cast<int>(blockDim.x);
  const int cta = blockIdx.x;
  const long long P = p.partition_blocks;
  const int per = (p.num_seqs + nthreads - 1) / nthreads;
  const int s_lo = min(p.num_seqs, tid * per);
  const int s_hi = min(p.num_seqs, s_lo + per);
  auto windows = [&](int s) -> long long {
    return ((load_ctx(p, s, BS) + BS - 1) / BS + P - 1) / P;
  };
  long long mine = 0;
  for (int s = s_lo; s < s_hi; ++s) mine += windows(s);
  long long incl, total;
  block_scan(mine, incl, total, tmp);
  const long long excl = incl - mine;
  const long long lo = total * cta / p.balanced_ctas;
  const long long hi = total * (cta + 1) / p.balanced_ctas;
  if (tid == 0) {
    sched->seq0 = p.num_seqs;
    sched->block0 = 0;
    sched->seq_end = p.num_seqs;
    sched->block_end = 0;
    sched->cta = cta;
  }
  __syncthreads();
  // window x of the walk -> (sequence, its first block), walking this slice
  auto locate = [&](long long x, int& seq, int& blk) {
    long long run = excl;
    for (int s = s_lo; s < s_hi; ++s) {
      const long long n = windows(s);
      if (x < run + n) {
        seq = s;
        blk = static_cast<int>((x - run) * P);
        return;
      }
      run += n;
    }
  };
  if (lo < total && mine > 0 && excl <= lo && lo < excl + mine)
    locate(lo, sched->seq0, sched->block0);
  if (hi < total && mine > 0 && excl <= hi && hi < excl + mine)
    locate(hi, sched->seq_end, sched->block_end);
}

template <int G, int BS>
__global__ void __launch_bounds__((max_heads_per_cta(G) + 1) * 32, 1)
    decode_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Layout L = make_layout(p.stages, p.stage_bytes, p.hpc, G);
  Schedule* sched = reinterpret_cast<Schedule*>(smem + L.sched);
  long long* tmp = reinterpret_cast<long long*>(smem + L.sched + 64);
  const int tid = threadIdx.x;

  if (tid == 0) {
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.barriers);
    uint64_t* empty = full + p.stages;
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], p.hpc);
    }
    fence_barrier_init();
  }
  grid_dependency_wait();        // inputs may come from the preceding kernel
  grid_dependents_launch();

  if (p.window_walk) {
    schedule_windows<BS>(p, sched, tmp);
  } else if (p.partition_blocks > 0) {
    // fixed windows: CTA (x = window, y = sequence)
    const int s = blockIdx.y;
    const int win = blockIdx.x;
    const int ctx = load_ctx(p, s, BS);
    const long long nb = (ctx + BS - 1) / BS;
    const long long b0 = static_cast<long long>(win) * p.partition_blocks;
    if (tid == 0) {
      sched->seq0 = s;
      sched->block0 = static_cast<int>(b0);
      sched->seq_end = s;
      sched->block_end = static_cast<int>(b0 < nb ? (nb - b0 < p.partition_blocks ? nb : b0 + p.partition_blocks) : b0);
      sched->cta = win;
    }
    if (nb == 0 && win == 0) {   // empty context: zero output rows
      const long long base = (static_cast<long long>(s) * p.hq + blockIdx.z * p.hpc * G) * kD;
      for (int i = tid; i < p.hpc * G * kD; i += blockDim.x) p.out[base + i] = 0.f;
    }
  } else {
    // balanced: this CTA streams the blocks in range [T*c/C, T*(c+1)/C) of
    // the cost line (see seq_cost); the schedule is where that range's first
    // and last blocks fall.
    if (p.num_seqs <= static_cast<int>(blockDim.x) && p.ws.seq_start == nullptr) {
      const int cta = blockIdx.x;
      const int w = p.seg_weight;
      long long total = 0, lo = 0, hi = 0;
      // a batch of at most one length per thread: one block-wide scan gives
      // the total and every sequence's place on the cost line; the threads
      // of the sequences holding positions T*c/C and T*(c+1)/C record them,
      // and every thread whose sequence has blocks in the CTA's range
      // prefetches those table entries into L1 for the producer
      const int s = tid;
      const long long nb = s < p.num_seqs ? (load_ctx(p, s, BS) + BS - 1) / BS : 0;
      const long long cost = seq_cost(nb, w);
      long long incl;
      block_scan(cost, incl, total, tmp);
      lo = total * cta / p.balanced_ctas;
      hi = total * (cta + 1) / p.balanced_ctas;
      const long long excl = incl - cost;
      if (tid == 0) {
        sched->cta = cta;
        if (lo >= total) {
          sched->seq0 = p.num_seqs;
          sched->block0 = 0;
        }
        if (hi >= total) {
          sched->seq_end = p.num_seqs;
          sched->block_end = 0;
        }
      }
      if (cost > 0 && excl <= lo && lo < excl + cost) {
        sched->seq0 = s;
        sched->block0 = static_cast<int>(lo - excl - w > 0 ? lo - excl - w : 0);
      }
      if (cost > 0 && excl <= hi && hi < excl + cost) {
        sched->seq_end = s;
        sched->block_end = static_cast<int>(hi - excl - w > 0 ? hi - excl - w : 0);
      }
      const long long a = lo > excl + w ? lo : excl + w;            // this sequence's
      const long long b = hi < excl + w + nb ? hi : excl + w + nb;  // blocks in range
      if (a < b) {
        const int32_t* row = p.block_tables + static_cast<long long>(s) * p.max_blocks;
        for (long long x = a - excl - w; x < b - excl - w; x += 32)
          asm volatile("prefetch.global.L1 [%0];" ::"l"(row + x));
        asm volatile("prefetch.global.L1 [%0];" ::"l"(row + (b - excl - w - 1)));
      }
    } else {
      schedule_large<BS>(p, sched, tmp, smem);
    }
  }
  __syncthreads();
  const Schedule sc = *sched;
  if (static_cast<int>(threadIdx.x >> 5) == p.hpc) {
    producer<G, BS>(p, sc, smem, L);
  } else {
    consumer<G, BS>(p, smem, L);
  }
}

// ------------------------------------------------------------------- merge

struct MergeParams {
  float* out;
  const int32_t* context_lens;
  int num_seqs, hq, max_blocks, bs;
  int partition_blocks, max_splits, balanced_ctas, seg_weight;
  DecodeWorkspace ws;
  uint32_t* status;
};

constexpr int kMergeHeads = 4;       // query heads per CTA
constexpr int kMergeMaxParts = 4;    // warps per head when sequences have many records
constexpr int kMergeMaxRecords = 512; // record indices staged per pass
constexpr int kMergeBatch = 16;       // records whose loads are in flight together
constexpr int kMergeWalk = 256;       // split sequences a large-batch merge CTA lists at once

__device__ __forceinline__ int merge_ctx(const MergeParams& p, int s) {
  int c = p.context_lens[s];
  const int cap = p.max_blocks * p.bs;
  return c < 0 ? 0 : (c > cap ? cap : c);
}

// Combines the partial records of one sequence:
//   M = max_r m_r;  out = sum_r 2^(m_r - M) acc_r / sum_r 2^(m_r - M) l_r.
// Small (128 threads, few registers) so that its CTAs fit beside the decode
// CTAs and run their prologue -- the record list, which depends only on the
// context lengths -- while the decode finishes.
__global__ void __launch_bounds__(kMergeHeads * kMergeMaxParts * 32)
    merge_kernel(const MergeParams p) {
  __shared__ long long tmp[32];
  __shared__ int recs[kMergeMaxRecords];
  __shared__ float part_m[kMergeMaxParts][kMergeHeads], part_l[kMergeMaxParts][kMergeHeads];
  __shared__ float part_o[kMergeMaxParts][kMergeHeads][kD];
  const int s = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int parts = static_cast<int>(blockDim.x) / (32 * kMergeHeads);
  const int hw = warp % kMergeHeads, part = warp / kMergeHeads;
  const int h = blockIdx.y * kMergeHeads + hw;
  const long long nb = (merge_ctx(p, s) + p.bs - 1) / p.bs;
  const bool fixed = p.partition_blocks > 0;

  long long n_cand = 0, seq_start = 0, total = 0, c_first = 0;
  if (fixed && nb > 0) {
    if (nb <= p.partition_blocks) return;   // single window: decode wrote the output
    n_cand = (nb + p.partition_blocks - 1) / p.partition_blocks;
  } else {
    if (nb == 0) {   // an empty context: zero rows (no decode CTA owns it in a
                     // balanced batch or a window walk)
      grid_dependency_wait();
      if (h < p.hq && part == 0) {
        float* dst = p.out + (static_cast<long long>(s) * p.hq + h) * kD;
        dst[lane] = 0.f;
        dst[lane + 32] = 0.f;
      }
      return;
    }
    // the same cost line as the decode's split (see seq_cost)
    long long tot_part = 0, pre_part = 0;
    for (int i = tid; i < p.num_seqs; i += blockDim.x) {
      const long long n = seq_cost((merge_ctx(p, i) + p.bs - 1) / p.bs, p.seg_weight);
      tot_part += n;
      if (i < s) pre_part += n;
    }
    long long incl, all;
    block_scan(tot_part, incl, all, tmp);
    total = all;
    block_scan(pre_part, incl, all, tmp);
    seq_start = all;                   // this sequence's place; its blocks follow w later
    const long long C = p.balanced_ctas;
    const long long first = seq_start + p.seg_weight;
    c_first = balanced_cta_of(first, total, C);
    const long long c_last = balanced_cta_of(first + nb - 1, total, C);
    if (c_first == c_last) return;   // one CTA held the whole sequence
    n_cand = c_last - c_first + 1;
  }

  // record index of candidate k, or -1 when that CTA holds none of s
  auto record_of = [&](long long k) -> int {
    if (fixed) return static_cast<int>(static_cast<long long>(s) * p.max_splits + k);
    const long long c = c_first + k;
    const long long lo = total * c / p.balanced_ctas;
    const long long hi = total * (c + 1) / p.balanced_ctas;
    const long long first = seq_start + p.seg_weight;
    const long long a = lo > first ? lo : first;
    const long long b = hi < first + nb ? hi : first + nb;
    if (a >= b) return -1;
    // the CTA's first segment is this sequence when its range starts at or
    // after the sequence's place on the line
    return static_cast<int>(2 * c + (seq_start <= lo ? 0 : 1));
  };

  float mx = -INFINITY, den = 0.f, o0 = 0.f, o1 = 0.f;
  bool waited = false;
  for (long long base = 0; base < n_cand; base += kMergeMaxRecords) {
    const int n = static_cast<int>(n_cand - base < kMergeMaxRecords ? n_cand - base
                                                                     : kMergeMaxRecords);
    if (base > 0) __syncthreads();
    for (int k = tid; k < n; k += blockDim.x) recs[k] = record_of(base + k);
    __syncthreads();
    if (!waited) {
      grid_dependency_wait();      // the decode's records must be complete
      waited = true;
    }
    if (h >= p.hq) continue;
    // this warp's slice of the pass's records
    const int k_lo = n * part / parts, k_hi = n * (part + 1) / parts;
    // 16 records at a time, every load of a batch issued before any is used
    // (a sequence split into 512-token windows has hundreds of records); the
    // batch's maximum moves the running one, as in the online softmax, so
    // one memory round trip serves a batch
    for (int k0 = k_lo; k0 < k_hi; k0 += kMergeBatch) {
      float mv[kMergeBatch], lv[kMergeBatch], a0[kMergeBatch], a1[kMergeBatch];
      bool have[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int r = k0 + u < k_hi ? recs[k0 + u] : -1;
        have[u] = r >= 0;
        mv[u] = -INFINITY;
        lv[u] = a0[u] = a1[u] = 0.f;
        if (have[u]) {
          const long long row = static_cast<long long>(r) * p.hq + h;
          mv[u] = p.ws.m[row];
          lv[u] = p.ws.l[row];
          a0[u] = p.ws.acc[row * kD + lane];
          a1[u] = p.ws.acc[row * kD + lane + 32];
        }
      }
      float mb = mx;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) mb = fmaxf(mb, mv[u]);
      if (mb == -INFINITY) continue;                  // no record in this batch
      const float f = ex2(mx - mb);                   // 0 while mx is -inf
      den *= f;
      o0 *= f;
      o1 *= f;
      mx = mb;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const float wgt = have[u] ? ex2(mv[u] - mx) : 0.f;
        den = fmaf(wgt, lv[u], den);
        o0 = fmaf(wgt, a0[u], o0);
        o1 = fmaf(wgt, a1[u], o1);
      }
    }
  }
  if (parts > 1) {
    // combine the slices of each head:  M = max m_i, sum 2^(m_i - M) (.)_i
    if (lane == 0) {
      part_m[part][hw] = mx;
      part_l[part][hw] = den;
    }
    part_o[part][hw][lane] = o0;
    part_o[part][hw][lane + 32] = o1;
    __syncthreads();
    if (part != 0) return;
    float mm = -INFINITY;
    for (int i = 0; i < parts; ++i) mm = fmaxf(mm, part_m[i][hw]);
    den = o0 = o1 = 0.f;
    for (int i = 0; i < parts; ++i) {
      const float mi = part_m[i][hw];
      const float w = mi == -INFINITY ? 0.f : ex2(mi - mm);
      den = fmaf(w, part_l[i][hw], den);
      o0 = fmaf(w, part_o[i][hw][lane], o0);
      o1 = fmaf(w, part_o[i][hw][lane + 32], o1);
    }
  }
  if (h >= p.hq) return;
  const float inv = 1.0f / den;
  float* dst = p.out + (static_cast<long long>(s) * p.hq + h) * kD;
  dst[lane] = o0 * inv;
  dst[lane + 32] = o1 * inv;
}

// Merge of a large balanced batch (more than kMergeScanMaxSeqs sequences):
// the combination of merge_kernel, but the decode recorded each sequence's
// first flattened block, so nothing scans the lengths.  The grid is two CTAs
// per decode CTA (x) times the head groups (y), 4 warps (one per head); CTA
// x owns sequences x + k gridDim.x.  One thread per sequence finds, in
// parallel, those the decode split over several CTAs and writes the zero rows
// of empty ones; then the CTA merges the split ones.  At most one split
// sequence per decode CTA boundary exists, and the round-robin ownership
// spreads them over the merge CTAs, so the kernel's time does not grow with
// the batch.
__global__ void __launch_bounds__(kMergeHeads * 32)
    merge_walk_kernel(const MergeParams p) {
  __shared__ int recs[kMergeMaxRecords];
  __shared__ int todo[kMergeWalk];
  __shared__ int ntodo;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y * kMergeHeads + warp;
  const long long C = p.balanced_ctas;
  grid_dependency_wait();              // the decode's records and block offsets
  const long long total = p.ws.seq_start[p.num_seqs];
  const long long owned = (p.num_seqs - 1 - static_cast<long long>(blockIdx.x)) / gridDim.x + 1;
  if (tid == 0) ntodo = 0;
  __syncthreads();
  for (long long k = tid; k < owned; k += blockDim.x) {
    const int sq = static_cast<int>(blockIdx.x + k * gridDim.x);
    const long long nb = (merge_ctx(p, sq) + p.bs - 1) / p.bs;
    if (nb == 0) {                     // empty context: zero rows
      for (int hh = 0; hh < kMergeHeads; ++hh) {
        const int hx = blockIdx.y * kMergeHeads + hh;
        if (hx >= p.hq) break;
        float4* dst = reinterpret_cast<float4*>(p.out + (static_cast<long long>(sq) * p.hq + hx) * kD);
        for (int e = 0; e < kD / 4; ++e) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
      const long long first = p.ws.seq_start[sq] + p.seg_weight;   // its first block's place
      if (balanced_cta_of(first, total, C) != balanced_cta_of(first + nb - 1, total, C)) {
        const int slot = atomicAdd(&ntodo, 1);
        if (slot < kMergeWalk) todo[slot] = sq;
      }
    }
  }
  __syncthreads();
  const int listed = ntodo;
  // with more split sequences than the list holds (only with more than
  // kMergeWalk decode CTAs), every owned sequence is visited
  const long long n_seq = listed <= kMergeWalk ? listed : owned;
  for (long long i = 0; i < n_seq; ++i) {
    const int s = listed <= kMergeWalk ? todo[i] : static_cast<int>(blockIdx.x + i * gridDim.x);
    const long long nb = (merge_ctx(p, s) + p.bs - 1) / p.bs;
    if (nb == 0) continue;
    const long long seq_start = p.ws.seq_start[s];
    const long long first = seq_start + p.seg_weight;
    const long long c_first = balanced_cta_of(first, total, C);
    const long long c_last = balanced_cta_of(first + nb - 1, total, C);
    if (c_first == c_last) continue;   // one CTA held the whole sequence
    const long long n_cand = c_last - c_first + 1;
    float mx = -INFINITY, den = 0.f, o0 = 0.f, o1 = 0.f;
    for (long long base = 0; base < n_cand; base += kMergeMaxRecords) {
      const int n = static_cast<int>(n_cand - base < kMergeMaxRecords ? n_cand - base
                                                                       : kMergeMaxRecords);
      __syncthreads();                 // the previous pass (or sequence) has read recs
      for (int k = tid; k < n; k += blockDim.x) {
        // record of candidate CTA c, or -1 when it holds none of s
        const long long c = c_first + base + k;
        const long long lo = total * c / C, hi = total * (c + 1) / C;
        const long long a = lo > first ? lo : first;
        const long long b = hi < first + nb ? hi : first + nb;
        recs[k] = a >= b ? -1 : static_cast<int>(2 * c + (seq_start <= lo ? 0 : 1));
      }
      __syncthreads();
      if (h >= p.hq) continue;
      for (int k0 = 0; k0 < n; k0 += kMergeBatch) {
        float mv[kMergeBatch], lv[kMergeBatch], a0[kMergeBatch], a1[kMergeBatch];
        bool have[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const int r = k0 + u < n ? recs[k0 + u] : -1;
          have[u] = r >= 0;
          mv[u] = -INFINITY;
          lv[u] = a0[u] = a1[u] = 0.f;
          if (have[u]) {
            const long long row = static_cast<long long>(r) * p.hq + h;
            mv[u] = p.ws.m[row];
            lv[u] = p.ws.l[row];
            a0[u] = p.ws.acc[row * kD + lane];
            a1[u] = p.ws.acc[row * kD + lane + 32];
          }
        }
        float mb = mx;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) mb = fmaxf(mb, mv[u]);
        if (mb == -INFINITY) continue;
        const float f = ex2(mx - mb);
        den *= f;
        o0 *= f;
        o1 *= f;
        mx = mb;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const float wgt = have[u] ? ex2(mv[u] - mx) : 0.f;
          den = fmaf(wgt, lv[u], den);
          o0 = fmaf(wgt, a0[u], o0);
          o1 = fmaf(wgt, a1[u], o1);
        }
      }
    }
    if (h >= p.hq) continue;
    const float inv = 1.0f / den;
    float* dst = p.out + (static_cast<long long>(s) * p.hq + h) * kD;
    dst[lane] = o0 * inv;
    dst[lane + 32] = o1 * inv;
  }
}

template <int G, int BS>
cudaError_t launch_t(const Params& prm, dim3 grid, uint32_t smem_bytes, cudaStream_t stream) {
  auto kern = decode_kernel<G, BS>;
  // the shared-memory limit, once per device: the opt-in maximum of a block
  constexpr int kMaxDynSmem = 227 * 1024;
  static PerDeviceOnce once;
  cudaError_t e = once.run([&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
  });
  if (e != cudaSuccess) return e;
  if (smem_bytes > static_cast<uint32_t>(kMaxDynSmem)) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, grid, dim3((prm.hpc + 1) * 32), smem_bytes, stream, prm);
}

}  // namespace

long long decode_prefix_entries(int num_seqs, int partition_blocks) {
  return partition_blocks == 0 && num_seqs > kMergeScanMaxSeqs ? num_seqs + 1LL : 0LL;
}

long long decode_records(int num_seqs, int max_blocks_per_seq, int partition_blocks,
                         int balanced_ctas) {
  if (partition_blocks > 0) {
    const long long splits = (max_blocks_per_seq + partition_blocks - 1) / partition_blocks;
    return splits <= 1 ? 0 : static_cast<long long>(num_seqs) * splits;
  }
  return 2LL * balanced_ctas;
}

// Layout: m [rows], l [rows] (each padded to 256 bytes), acc [rows, D],
// then the per-sequence block offsets (prefix_entries int64) of large
// balanced batches.
size_t decode_workspace_bytes(long long records, int num_q_heads, int head_dim,
                              long long prefix_entries) {
  if (records <= 0) return 0;
  const size_t rows = static_cast<size_t>(records) * num_q_heads;
  const size_t a = (rows * sizeof(float) + 255) / 256 * 256;
  const size_t acc = (rows * head_dim * sizeof(float) + 255) / 256 * 256;
  return 2 * a + acc + static_cast<size_t>(prefix_entries) * sizeof(long long);
}

DecodeWorkspace decode_workspace_carve(void* base, long long records, int num_q_heads,
                                       int head_dim, long long prefix_entries) {
  DecodeWorkspace ws{nullptr, nullptr, nullptr, nullptr};
  if (records <= 0 || base == nullptr) return ws;
  const size_t rows = static_cast<size_t>(records) * num_q_heads;
  const size_t a = (rows * sizeof(float) + 255) / 256 * 256;
  const size_t acc = (rows * head_dim * sizeof(float) + 255) / 256 * 256;
  uint8_t* b = static_cast<uint8_t*>(base);
  ws.m = reinterpret_cast<float*>(b);
  ws.l = reinterpret_cast<float*>(b + a);
  ws.acc = reinterpret_cast<float*>(b + 2 * a);
  if (prefix_entries > 0) ws.seq_start = reinterpret_cast<long long*>(b + 2 * a + acc);
  return ws;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int hmax = max_heads_per_cta(G);
  const int hpc = a.num_kv_heads < hmax ? a.num_kv_heads : hmax;
  const int groups = a.num_kv_heads / hpc;
  const int bs = a.block_size;

  Params prm;
  prm.out = a.out;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.k_cache = static_cast<const __nv_bfloat16*>(a.k_cache);
  prm.v_cache = static_cast<const __nv_bfloat16*>(a.v_cache);
  prm.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  prm.k_cache_w = static_cast<__nv_bfloat16*>(const_cast<void*>(a.k_cache));
  prm.v_cache_w = static_cast<__nv_bfloat16*>(const_cast<void*>(a.v_cache));
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.num_seqs = a.num_seqs;
  prm.hq = a.num_q_heads;
  prm.hkv = a.num_kv_heads;
  prm.num_blocks = a.num_blocks;
  prm.max_blocks = a.max_blocks_per_seq;
  prm.hpc = hpc;
  prm.stage_bytes = align_up(2 * kStageTokens * hpc * kRowBytes + hpc * G * kRowBytes, 128);
  const uint32_t fixed_part = make_layout(0, prm.stage_bytes, hpc, G).total + 2 * 8 * 8 + 16 * 8;
  int stages = static_cast<int>((kSmemBudget - fixed_part) / prm.stage_bytes);
  stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  prm.stages = stages;
  prm.scale_log2 = a.scale * kLog2e;
  prm.partition_blocks = a.partition_blocks;
  prm.max_splits = a.max_splits;
  prm.balanced_ctas = a.balanced_ctas;
  // a sequence start costs about one 32-token stage: 32 / bs blocks, rounded
  prm.seg_weight = a.partition_blocks > 0 ? 0 : (kStageTokens + bs / 2) / bs;
  // more possible windows than persistent CTAs: the CTAs walk the windows
  prm.window_walk = a.partition_blocks > 0 && a.window_ctas > 0 &&
                    static_cast<long long>(a.max_splits) * a.num_seqs > a.window_ctas;
  if (prm.window_walk) prm.balanced_ctas = a.window_ctas;
  prm.ws = a.ws;
  prm.status = a.status;
  const uint32_t smem = make_layout(stages, prm.stage_bytes, hpc, G).total;

  dim3 grid;
  if (prm.window_walk)
    grid = dim3(a.window_ctas, 1, groups);
  else if (a.partition_blocks > 0)
    grid = dim3(a.max_splits, a.num_seqs, groups);
  else
    grid = dim3(a.balanced_ctas, 1, groups);

  cudaError_t e = cudaErrorInvalidValue;
  switch (G * 1000 + bs) {
    case 1016: e = launch_t<1, 16>(prm, grid, smem, stream); break;
    case 1032: e = launch_t<1, 32>(prm, grid, smem, stream); break;
    case 1064: e = launch_t<1, 64>(prm, grid, smem, stream); break;
    case 1128: e = launch_t<1, 128>(prm, grid, smem, stream); break;
    case 2016: e = launch_t<2, 16>(prm, grid, smem, stream); break;
    case 2032: e = launch_t<2, 32>(prm, grid, smem, stream); break;
    case 2064: e = launch_t<2, 64>(prm, grid, smem, stream); break;
    case 2128: e = launch_t<2, 128>(prm, grid, smem, stream); break;
    case 4016: e = launch_t<4, 16>(prm, grid, smem, stream); break;
    case 4032: e = launch_t<4, 32>(prm, grid, smem, stream); break;
    case 4064: e = launch_t<4, 64>(prm, grid, smem, stream); break;
    case 4128: e = launch_t<4, 128>(prm, grid, smem, stream); break;
    case 8016: e = launch_t<8, 16>(prm, grid, smem, stream); break;
    case 8032: e = launch_t<8, 32>(prm, grid, smem, stream); break;
    case 8064: e = launch_t<8, 64>(prm, grid, smem, stream); break;
    case 8128: e = launch_t<8, 128>(prm, grid, smem, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;

  const bool need_merge =
      a.partition_blocks == 0 ||
      (a.max_blocks_per_seq + a.partition_blocks - 1) / a.partition_blocks > 1;
  if (!need_merge) return cudaSuccess;
  MergeParams mp;
  mp.out = a.out;
  mp.context_lens = a.context_lens;
  mp.num_seqs = a.num_seqs;
  mp.hq = a.num_q_heads;
  mp.max_blocks = a.max_blocks_per_seq;
  mp.bs = bs;
  mp.partition_blocks = a.partition_blocks;
  mp.max_splits = a.max_splits;
  mp.balanced_ctas = a.balanced_ctas;
  mp.seg_weight = prm.seg_weight;
  mp.ws = a.ws;
  mp.status = a.status;
  const unsigned hgroups = (a.num_q_heads + kMergeHeads - 1) / kMergeHeads;
  if (a.ws.seq_start != nullptr)        // large balanced batch
    return launch_pdl(merge_walk_kernel,
                      dim3(std::min(a.num_seqs, 2 * a.balanced_ctas), hgroups),
                      dim3(kMergeHeads * 32), 0, stream, mp);
  dim3 mgrid(a.num_seqs, hgroups);
  // many records per sequence (fixed windows over long contexts): four warps
  // per head, each merging a quarter of the records
  const int parts = a.partition_blocks > 0 && a.max_splits > 64 ? kMergeMaxParts : 1;
  return launch_pdl(merge_kernel, mgrid, dim3(kMergeHeads * parts * 32), 0, stream, mp);
}

}  // namespace tvl
