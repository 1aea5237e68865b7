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
// A unit of work is one 128-row query tile of NH query heads of the same GQA
// group (NH = 2 when the group has two or more heads), so each K/V tile
// gathered from the paged cache serves NH heads.  The kernel is persistent:
// one CTA per SM walks its share of the units (longest first, dealt in snake
// order), and the K/V ring, the barriers and TMEM carry on from one unit to
// the next, so a unit's loads and first Q K^T overlap the previous unit's
// last softmax and its output.  Warps:
//   0..4NH-1  softmax, one warpgroup per head: thread r owns query row r
//             (TMEM lane r).  Per 128-key tile it loads its 128 scores into
//             registers and releases S at once, so the next tile's Q K^T
//             overlaps the rest.  It computes P = 2^(S*scale*log2e - m) with
//             packed fp32x2 arithmetic against a reference maximum m set by
//             the first tile; only when a tile's row sum shows that some P
//             nears the fp16 limit does it take the tile's maximum, move m
//             and recompute P from the scores still in registers (O in TMEM
//             is then rescaled; exact, since one reference scales numerator
//             and denominator).  P is stored as fp16 into TMEM once the
//             previous P.V has consumed the buffer.  At a unit's end it
//             normalises O into swizzled staging in shared memory, and each
//             warp's 32 rows leave through four TMA tensor stores;
//   4NH       producer: TMA loads of the Q tiles and, per 128-key tile, one
//             box of bs tokens x 64 dims per physical block (K and V) found
//             through the block table -- the paged gather; blocks past the
//             context are requested out of range, so TMA fills them with 0;
//   4NH+1     MMA issuer: S_h = Q_h K^T (M 128, N 128, bf16, both operands in
//             shared memory) and O_h += P_h V (M 128, N 64, fp16, P read from
//             TMEM, V an MN-major shared operand), fp32 accumulation.  The
//             next tile's S is issued as soon as the softmax has released S,
//             before this tile's P.V (on a unit's last tile, after it).
//             Completion is signalled by tcgen05.commit;
//   4NH+2     V conversion: each V tile bf16 -> fp16 in place (exact for
//             2^-14 <= |v| <= 65504; smaller values keep an absolute error
//             below 2^-25; a larger one becomes infinite, which leaves rows
//             that are not finite, reported as TVL_DEV_NONFINITE; keys past
//             the context become 0);
//   4NH+3     P.V issuer (below).
// P and V go through fp16 rather than bf16 so that rounding P costs at most
// 2^-11 relative (bf16 would cost 2^-8) -- the fp32-accumulated result stays
// within 2e-3 of the exact attention even for rows with few keys.
// TMEM (per head h): S_h 128 columns, O_h 64, P_h 64 (fp16 pairs).
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
constexpr int kStages = 3;
constexpr int kOPitch = kD * 4 + 16;    // bytes per staged output row: 16-byte rows
                                        // land on distinct banks (no conflicts)
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kTileBytes = kBM * kD * 2;      // 16 KB: 128 rows x 128 B

constexpr uint32_t kIdescQK = idesc_f16_f32acc(1, 0, kBM, kBN);   // bf16, K-major B
constexpr uint32_t kIdescPV = idesc_f16_f32acc(0, 1, kBM, kD);    // fp16, MN-major B

template <int NH>
struct Cfg {
  static constexpr int kSoftmaxWarps = 4 * NH;
  static constexpr int kProducerWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;         // issues Q K^T
  static constexpr int kConvWarp = kSoftmaxWarps + 2;        // V conversion
  static constexpr int kPvWarp = kSoftmaxWarps + 3;          // issues P.V
  static constexpr int kThreads = (kSoftmaxWarps + 4) * 32;
  static_assert(kConvWarp + 1 == kPvWarp && kThreads == (kPvWarp + 1) * 32, "warp roles");
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = NH * kTileBytes;
  static constexpr uint32_t kVOff = kKOff + kStages * kTileBytes;
  static constexpr uint32_t kStageOff = kVOff + kStages * kTileBytes;   // output rows
  static constexpr uint32_t kBarOff = kStageOff + NH * kBM * kOPitch;
  static constexpr uint32_t kTabOff = kBarOff + 512;    // item order, lengths, rank keys
  static constexpr uint32_t kSmemBytes = kTabOff + 5 * 4 * kThreads + 1024;   // + alignment slack
  static constexpr uint32_t kTmemCols = NH == 2 ? 512 : 256;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");
  __device__ static uint32_t s_col(int h) { return h * kBN; }
  __device__ static uint32_t o_col(int h) { return NH * kBN + h * kD; }
  __device__ static uint32_t p_col(int h) { return NH * (kBN + kD) + h * (kBN / 2); }
};

// Register split of the two-head kernel: 12 warps launched with 168
// registers each (64512); the producer / MMA / conversion warpgroup drops to
// 72 and the two softmax warpgroups rise to 216, which holds a row's 128
// scores and its 64 packed P together: 2 x 128 x 216 + 128 x 72 = 64512.
// The host checks the launch allocation before the first launch.
constexpr int kRegsSoftmax = 216;
constexpr int kRegsAux = 72;

struct Barriers {
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t v_ready[kStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int4 ustash[8];       // per softmax warp: its unit's rows, first output row, first head
};
static_assert(sizeof(Barriers) <= 512, "barrier area");

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

__device__ __forceinline__ float max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

__device__ __forceinline__ float min3(float a, float b, float c) {
  float y;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
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

// Bounded wait that records a timeout in the status word; returns false
// when the caller must stop (every role then leaves its loop).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const Params& p) {
  if (mbar_wait(bar, parity)) return true;
  report(p.status, kDevTimeout);
  return false;
}

// One work unit: a 128-row query tile of NH query heads of one sequence.
// Every role of the CTA derives the same units in the same order.
struct Unit {
  int s, h0, q0, row0, rows, pos_first, ctx, n_kv;
  bool valid;      // rows to compute and consistent lengths
  bool bad;        // the sequence's lengths are inconsistent (reported, skipped)
  bool bad_ctx;    // the inconsistency is a context past the table's capacity
};

// Index of the k-th unit of CTA c among G: the units in longest-first order
// are dealt to the CTAs row by row, every other row reversed (c, 2G-1-c,
// 2G+c, ...), which evens out the CTAs' totals.  Increases with k.
__device__ __forceinline__ long long unit_index(int k, int c, int G) {
  return static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
}


// Unit u: rank u / pairs in the item order, head group u % pairs.  With
// `tab`, the order and the items' lengths come from shared memory (tab[0..K)
// rank -> item, then K-strided q0, Lq and context per item); without it the
// order is the item order and the lengths are read from global memory.
template <int NH, int K>
__device__ __forceinline__ void unit_info(const Params& p, const int* tab, int u, Unit& x) {
  const int pairs = p.hq / NH;
  const int rank = u / pairs;
  x.h0 = (u - rank * pairs) * NH;
  int item, lq;
  if (tab != nullptr) {
    item = tab[rank];
    x.q0 = tab[K + item];
    lq = tab[2 * K + item];
    x.ctx = tab[3 * K + item];
  } else {
    item = rank;
    const int si = item / p.n_qtiles;
    x.q0 = p.query_start_loc[si];
    lq = p.query_start_loc[si + 1] - x.q0;
    x.ctx = p.context_lens[si];
  }
  x.s = item / p.n_qtiles;
  x.row0 = (p.n_qtiles - 1 - item % p.n_qtiles) * kBM;
  const int cap = p.max_blocks * p.bs;
  const bool rows_here = x.row0 < lq;
  // The whole sequence is skipped (and reported) when its query rows would
  // leave [0, total_q) -- a negative or decreasing query_start_loc entry, or
  // one past total_q_tokens -- when it has more rows than max_q_len's query
  // tiles cover, or when its context cannot hold its chunk or exceeds the
  // block table.  So no unit ever addresses a row outside `out`.
  const bool bad_rows = x.q0 < 0 || lq < 0 ||
                        static_cast<long long>(x.q0) + lq > static_cast<long long>(p.total_q) ||
                        lq > p.n_qtiles * kBM;
  x.bad_ctx = !bad_rows && x.ctx > cap;
  x.bad = bad_rows || (lq > 0 && (x.ctx < lq || x.ctx > cap));
  x.valid = rows_here && !x.bad;
  x.rows = min(kBM, lq - x.row0);
  x.pos_first = x.ctx - lq + x.row0;
  x.n_kv = (x.pos_first + x.rows - 1) / kBN + 1;
}

// The first unit of this CTA at or after index k that has work; k moves to
// it.  With kWarp it is called by whole warps and the fields go through
// lane 0, so that the compiler sees them warp-uniform (fewer registers).
template <int NH, int K, bool kWarp>
__device__ __forceinline__ bool next_valid_unit(const Params& p, const int* tab, int& k, Unit& x) {
  const int n_units = p.num_seqs * p.n_qtiles * (p.hq / NH);
  for (;; ++k) {
    const long long u = unit_index(k, blockIdx.x, gridDim.x);
    if (u >= n_units) return false;
    unit_info<NH, K>(p, tab, static_cast<int>(u), x);
    if (!kWarp) {
      if (x.valid) return true;
      continue;
    }
    if (__shfl_sync(kFull, x.valid ? 1 : 0, 0)) break;
  }
  x.s = __shfl_sync(kFull, x.s, 0);
  x.h0 = __shfl_sync(kFull, x.h0, 0);
  x.q0 = __shfl_sync(kFull, x.q0, 0);
  x.row0 = __shfl_sync(kFull, x.row0, 0);
  x.rows = __shfl_sync(kFull, x.rows, 0);
  x.pos_first = __shfl_sync(kFull, x.pos_first, 0);
  x.ctx = __shfl_sync(kFull, x.ctx, 0);
  x.n_kv = __shfl_sync(kFull, x.n_kv, 0);
  return true;
}

template <int NH>
__global__ void __launch_bounds__(Cfg<NH>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_o, const Params p) {
  using C = Cfg<NH>;
  constexpr int K = C::kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Barriers* B = reinterpret_cast<Barriers*>(smem + C::kBarOff);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);

  grid_dependency_wait();          // inputs may come from the preceding kernel
  grid_dependents_launch();

  // ---- the item order.  Item i is sequence i / n_qtiles, query tile
  // n_qtiles - 1 - i % n_qtiles.  Items with the most key tiles go first
  // (ties in item order), so the long ones are not left for the end.  Every
  // CTA ranks the items the same way from the lengths, one item per thread
  // (beyond that, item order is kept); the ranks are a permutation of the
  // items whatever the lengths hold.
  const int n_units = p.num_seqs * p.n_qtiles * (p.hq / NH);   // < 2^31 (host check)
  const int n_items = p.num_seqs * p.n_qtiles;
  const int* tab = nullptr;
  if (n_items <= K) {
    int* t = reinterpret_cast<int*>(smem + C::kTabOff);
    int* keys = t + 4 * K;
    const int i = threadIdx.x;
    int key = 0;
    if (i < n_items) {
      const int si = i / p.n_qtiles;
      const int qt = p.n_qtiles - 1 - i % p.n_qtiles;
      const int qa = p.query_start_loc[si];
      const int lqi = p.query_start_loc[si + 1] - qa;
      const int ci = p.context_lens[si];
      const int last = ci - lqi + min((qt + 1) * kBM, lqi);   // keys seen
      key = qt * kBM >= lqi ? 0 : (last + kBN - 1) / kBN;
      keys[i] = key;
      t[K + i] = qa;
      t[2 * K + i] = lqi;
      t[3 * K + i] = ci;
    }
    __syncthreads();
    if (i < n_items) {
      int r = 0;
      for (int j = 0; j < n_items; ++j) {
        const int kj = keys[j];
        r += (kj > key || (kj == key && j < i)) ? 1 : 0;
      }
      t[r] = i;
    }
    tab = t;
  }
  auto next_unit = [&](int& k, Unit& x) -> bool {
    return next_valid_unit<NH, K, true>(p, tab, k, x);
  };

  if (threadIdx.x == 0) {
    mbar_init(&B->q_full, 1);
    mbar_init(&B->q_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&B->kv_full[i], 1);
      mbar_init(&B->kv_empty[i], 1);
      mbar_init(&B->v_ready[i], 1);
    }
    for (int i = 0; i < NH; ++i) {
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->s_free[i], 4);
      mbar_init(&B->p_full[i], 4);
      mbar_init(&B->pv_done[i], 1);
    }
    mbar_init(&B->mma_done, 2);           // one commit from each MMA issuer
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&B->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B->tmem_base;

  if (warp >= C::kSoftmaxWarps) {
  if constexpr (NH == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsAux));
  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Per unit: the Q tiles once the previous unit's Q K^T MMAs are done
    // (q_empty), then per 128-key tile one box of bs tokens x 64 dims per
    // physical block (K and V) into the next stage of the ring.
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      prefetch_tensormap(&tm_o);
    }
    const int boxes = kBN / p.bs;                       // physical blocks per KV tile
    int gt = 0;                                         // KV tiles issued
    int nq = 0;                                         // Q loads issued
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit x;
      if (!next_unit(k, x)) break;
      if (lane == 0) {
        if (nq > 0) ok = wait_or_abort(&B->q_empty, (nq - 1) & 1, p);
        if (ok) {
          mbar_arrive_expect_tx(&B->q_full, NH * kTileBytes);
          for (int i = 0; i < NH; ++i)
            tma_load_3d(smem + C::kQOff + i * kTileBytes, &tm_q, 0, x.h0 + i, x.q0 + x.row0,
                        &B->q_full);
        }
      }
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      ++nq;
      const int g = x.h0 / p.group;                     // shared KV head
      const int nblk = (x.ctx + p.bs - 1) / p.bs;
      const int32_t* table = p.block_tables + static_cast<long long>(x.s) * p.max_blocks;
      for (int j = 0; j < x.n_kv; ++j, ++gt) {
        const int st = gt % kStages;
        if (gt >= kStages && lane == 0)
          ok = wait_or_abort(&B->kv_empty[st], ((gt / kStages) - 1) & 1, p);
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&B->kv_full[st], 2 * kTileBytes);
        __syncwarp();
        for (int b = lane; b < boxes; b += 32) {
          const int lb = j * boxes + b;                 // logical block
          int phys = p.num_blocks;                      // out of range: zero fill
          if (lb < nblk) {
            phys = table[lb];
            if (phys < 0 || phys >= p.num_blocks) {
              report(p.status, TVL_DEV_BAD_BLOCK_ID);
              phys = p.num_blocks;
            }
          }
          const uint32_t off = static_cast<uint32_t>(b * p.bs) * (kD * 2);
          tma_load_4d(smem + C::kKOff + st * kTileBytes + off, &tm_k, 0, g, 0, phys,
                      &B->kv_full[st]);
          tma_load_4d(smem + C::kVOff + st * kTileBytes + off, &tm_v, 0, g, 0, phys,
                      &B->kv_full[st]);
        }
      }
    }
    // the loads in flight must land before exit
    if (lane == 0) {
      for (int t = gt > kStages ? gt - kStages : 0; t < gt; ++t)
        if (!mbar_wait(&B->kv_full[t % kStages], (t / kStages) & 1)) report(p.status, kDevTimeout);
      if (nq > 0 && !mbar_wait(&B->q_full, (nq - 1) & 1)) report(p.status, kDevTimeout);
    }
  } else if (warp == C::kMmaWarp || warp == C::kPvWarp) {
    // ------------------------------------------------------- MMA issuers
    // Two threads issue: one the Q K^T MMAs, one the P.V MMAs.  The tensor
    // pipe queues little, so an issuing thread that waits on a barrier
    // idles it; with two, one issues while the other waits.  Both walk one
    // stream of key tiles over all of the CTA's units.
    //   Q K^T: S_h(t) = Q_h K(t)^T once K(t) has landed and the softmax has
    //   taken S_h(t-1) into registers (s_free) -- across unit boundaries too,
    //   so the next unit's first scores are ready when its softmax starts.
    //   After a unit's last Q K^T, q_empty frees the Q buffer.
    //   P.V: O_h += P_h(t) V(t) once P_h(t) is in TMEM (p_full) and V(t) is
    //   fp16 (v_ready); then the stage goes back to the producer (kv_empty:
    //   Q K^T(t) is complete too, the softmax having read S_h(t)).
    if (lane == 0) {
      const bool is_qk = warp == C::kMmaWarp;
      const uint32_t q_addr = smem_addr(smem + C::kQOff);
      int gt = 0;                                       // key tile of the stream
      int st = 0, ph = 0;                               // its stage and phase
      int nq = 0;                                       // units begun
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Unit x;
        if (!next_valid_unit<NH, K, false>(p, tab, k, x)) break;
        for (int j = 0; ok && j < x.n_kv; ++j, ++gt) {
          if (is_qk) {
            ok = wait_or_abort(&B->kv_full[st], ph, p);
            if (ok && j == 0) ok = wait_or_abort(&B->q_full, nq & 1, p);
            const uint32_t k_addr = smem_addr(smem + C::kKOff + st * kTileBytes);
            for (int hh = 0; ok && hh < NH; ++hh) {
              if (gt > 0) ok = wait_or_abort(&B->s_free[hh], (gt - 1) & 1, p);
              if (!ok) break;
              tc_fence_after();
              const uint32_t qa = q_addr + hh * kTileBytes;
#pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk)
                mma_f16_ss(tmem + C::s_col(hh), desc_sw128(qa + kk * 32, 16, 1024),
                           desc_sw128(k_addr + kk * 32, 16, 1024), kIdescQK, kk > 0);
              mma_commit(&B->s_full[hh]);
            }
            if (ok && j + 1 == x.n_kv) mma_commit(&B->q_empty);
          } else {
            ok = wait_or_abort(&B->v_ready[st], ph, p);
            const uint32_t v_addr = smem_addr(smem + C::kVOff + st * kTileBytes);
            for (int hh = 0; ok && hh < NH; ++hh) {
              ok = wait_or_abort(&B->p_full[hh], gt & 1, p);
              if (!ok) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                mma_f16_ts(tmem + C::o_col(hh), tmem + C::p_col(hh) + kk * 8,
                           desc_sw128(v_addr + kk * 2048, 16, 1024), kIdescPV,
                           (j > 0 || kk > 0));
              mma_commit(&B->pv_done[hh]);
            }
            if (ok) mma_commit(&B->kv_empty[st]);
          }
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
        ++nq;
      }
      // every MMA issued must be complete before TMEM is released
      mma_commit(&B->mma_done);
      if (!mbar_wait(&B->mma_done, 0)) report(p.status, kDevTimeout);
    }
  } else {
    // ------------------------------------------------------- V conversion
    // V tile bf16 -> fp16 in place, 16 bytes at a time (the swizzle only
    // permutes 16-byte chunks within a 128-byte row, so a chunk's row is its
    // offset / 128); keys past the context become 0.
    const int t = lane;
    int gt = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit x;
      if (!next_unit(k, x)) break;
      for (int j = 0; j < x.n_kv; ++j, ++gt) {
        const int st = gt % kStages;
        ok = wait_or_abort(&B->kv_full[st], (gt / kStages) & 1, p);
        if (__any_sync(kFull, !ok)) { ok = false; break; }
        uint8_t* vt = smem + C::kVOff + st * kTileBytes;
#pragma unroll 4
        for (int e = t; e < static_cast<int>(kTileBytes / 16); e += 32) {
          uint4 w = *reinterpret_cast<const uint4*>(vt + e * 16);
          if (j * kBN + (e >> 3) < x.ctx) {
            w.x = bf16x2_to_half2(w.x);
            w.y = bf16x2_to_half2(w.y);
            w.z = bf16x2_to_half2(w.z);
            w.w = bf16x2_to_half2(w.w);
          } else {
            w = make_uint4(0, 0, 0, 0);
          }
          *reinterpret_cast<uint4*>(vt + e * 16) = w;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->v_ready[st]);
      }
    }
  }
  } else {
    // ------------------------------------------------------------- softmax
    if constexpr (NH == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    const int hh = warp >> 2;                           // head of this warpgroup
    const int wi = warp & 3;                            // TMEM lane quadrant
    const int r = wi * 32 + lane;                       // row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wi * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + C::s_col(hh);
    const uint32_t o_addr = tmem + lane_off + C::o_col(hh);
    const uint32_t p_addr = tmem + lane_off + C::p_col(hh);
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    int gt = 0;                                         // global key-tile index
    bool ok = true;

    for (int k = 0; ok; ++k) {
      Unit x;
      if (!next_unit(k, x)) break;
      // the unit's place, for the output at its end (cheaper than deriving
      // it again there, and no registers held through the tile loop)
      if (lane == 0) B->ustash[warp] = make_int4(x.rows, x.q0 + x.row0, x.h0, 0);
      __syncwarp();
      const int qpos = x.pos_first + r;
      const int pos_first = x.pos_first;
      const int ctx = x.ctx;
      const int n_kv = x.n_kv;
      float m_used = -INFINITY;                         // reference maximum (log2 units)
      float2 l2 = make_float2(0.f, 0.f);

      for (int j = 0; j < n_kv; ++j, ++gt) {
        const int key0 = j * kBN;
        ok = wait_or_abort(&B->s_full[hh], gt & 1, p);
        if (__any_sync(kFull, !ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[4][32];                             // this row's 128 scores
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(s_addr + cc * 32, sr[cc]);
        tmem_ld_wait();
        // S_h is in registers: the next tile's Q K^T may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->s_free[hh]);

        // Tiles on the causal diagonal or past the context need the mask.
        const bool masked = (key0 + kBN - 1 > pos_first) || (key0 + kBN > ctx);
        const int limit = min(qpos, ctx - 1) - key0;    // last visible column
        // row maximum of the scaled scores of this tile
        auto tile_max = [&]() -> float {
          float mt;
          if (masked) {
            mt = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                float v = __uint_as_float(sr[cc][e]) * p.scale_log2;
                if (cc * 32 + e > limit) v = -INFINITY;
                mt = fmaxf(mt, v);
              }
          } else if (p.scale_log2 >= 0.f) {
            float mx = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int e = 0; e < 32; e += 2)
                mx = max3(mx, __uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]));
            mt = mx * p.scale_log2;
          } else {
            float mn = INFINITY;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int e = 0; e < 32; e += 2)
                mn = min3(mn, __uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]));
            mt = mn * p.scale_log2;
          }
          return mt;
        };
        uint32_t pk[2][32];
        // P = 2^(s * scale * log2e - m) as fp16 pairs; returns the fp32 row sum
        auto make_p = [&](float mref) -> float2 {
          const float2 nm2 = make_float2(-mref, -mref);
          float2 tsum = make_float2(0.f, 0.f);
          if (masked) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float2 v = make_float2(__uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]));
                v = __ffma2_rn(v, sl2, nm2);
                if (cc * 32 + e > limit) v.x = -INFINITY;
                if (cc * 32 + e + 1 > limit) v.y = -INFINITY;
                const float2 pv = make_float2(ex2(v.x), ex2(v.y));
                tsum = __fadd2_rn(tsum, pv);
                pk[cc >> 1][(cc & 1) * 16 + e / 2] = pack_half2(pv.x, pv.y);
              }
          } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float2 v = make_float2(__uint_as_float(sr[cc][e]), __uint_as_float(sr[cc][e + 1]));
                v = __ffma2_rn(v, sl2, nm2);
                const float2 pv = make_float2(ex2(v.x), ex2(v.y));
                tsum = __fadd2_rn(tsum, pv);
                pk[cc >> 1][(cc & 1) * 16 + e / 2] = pack_half2(pv.x, pv.y);
              }
          }
          return tsum;
        };
        float f = 1.f;
        bool move = false;
        float2 tsum;
        if (j == 0) {
          m_used = tile_max();
          tsum = make_p(m_used == -INFINITY ? 0.f : m_used);
        } else {
          // P straight from the reference maximum; only a row sum that shows
          // some P near the fp16 limit (65504) calls for the tile's maximum
          tsum = make_p(m_used == -INFINITY ? 0.f : m_used);
          const float ts = tsum.x + tsum.y;
          move = !(ts <= 60000.f);
          if (__any_sync(kFull, move)) {
            if (move) {
              const float m_new = fmaxf(m_used, tile_max());
              f = ex2(m_used - m_new);
              m_used = m_new;
            }
            tsum = make_p(m_used == -INFINITY ? 0.f : m_used);
          }
        }
        // P_h of the previous tile must have been consumed (and O_h
        // complete) before P_h is overwritten and O_h rescaled.  On a unit's
        // first tile this was awaited at the end of the previous unit.
        if (j > 0) {
          ok = wait_or_abort(&B->pv_done[hh], (gt - 1) & 1, p);
          if (__any_sync(kFull, !ok)) { ok = false; break; }
          tc_fence_after();
          if (__any_sync(kFull, move)) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              uint32_t o[32];
              tmem_ld32(o_addr + cc * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
              tmem_st32(o_addr + cc * 32, o);
            }
          }
        }
        l2.x = fmaf(l2.x, f, tsum.x);
        l2.y = fmaf(l2.y, f, tsum.y);
        tmem_st32(p_addr, pk[0]);
        tmem_st32(p_addr + 32, pk[1]);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->p_full[hh]);
      }
      if (!ok) break;
      // the unit's O_h is complete once its last P.V is; read it out before
      // the next unit's first P.V overwrites it (that P.V waits for this
      // warpgroup's next p_full)
      ok = wait_or_abort(&B->pv_done[hh], (gt - 1) & 1, p);
      if (__any_sync(kFull, !ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld32(o_addr, o[0]);
      tmem_ld32(o_addr + 32, o[1]);
      tmem_ld_wait();
      const int4 us = B->ustash[warp];                  // rows, first output row, first head
      // Each warp stages its 32 rows in shared memory in the tensor-store
      // layout (per head: two 64-column halves of 128 rows x 128 bytes, the
      // 16-byte chunks of row r in 128-byte-swizzled order j ^ (r & 7), which
      // is also free of bank conflicts), and its lane 0 hands them to the
      // TMA engine as 16-row x 32-column tensor stores.  The softmax threads
      // so spend only the staging on the unit's 64 KB of fp32 output.
      const int r0 = wi * 32;                           // the warp's first row
      const int nrows = min(32, us.x - r0);             // rows of it inside the unit
      uint8_t* st_head = smem + C::kStageOff + hh * (kBM * kD * 4);
      if (lane == 0) bulk_wait_read();                  // its last stores have read the rows
      __syncwarp();
      const float inv = 1.0f / (l2.x + l2.y);
      if (lane < nrows) {
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int jc = 0; jc < 8; ++jc)
            *reinterpret_cast<float4*>(st_head + half * (kBM * 128) + r * 128 + ((jc ^ (r & 7)) << 4)) =
                make_float4(__uint_as_float(o[half][4 * jc]) * inv,
                            __uint_as_float(o[half][4 * jc + 1]) * inv,
                            __uint_as_float(o[half][4 * jc + 2]) * inv,
                            __uint_as_float(o[half][4 * jc + 3]) * inv);
        // A row that is not finite: a V value beyond the fp16 range of the
        // P.V product (bf16 holds values past 65504), or non-finite inputs.
        // The sum of the unnormalised row carries any inf or NaN.
        float2 chk[4] = {};
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            chk[(e >> 1) & 3] = __fadd2_rn(chk[(e >> 1) & 3],
                                           make_float2(__uint_as_float(o[cc][e]),
                                                       __uint_as_float(o[cc][e + 1])));
        const float2 c4 = __fadd2_rn(__fadd2_rn(chk[0], chk[1]), __fadd2_rn(chk[2], chk[3]));
        if (!isfinite(c4.x + c4.y) || !isfinite(inv)) report(p.status, TVL_DEV_NONFINITE);
      }
      fence_async_smem();                               // the staging, for the TMA engine
      __syncwarp();
      const int full = nrows >= 32 ? 32 : (nrows >= 16 ? 16 : 0);   // rows in whole 16-row groups
      if (lane == 0 && full > 0) {
        for (int g = 0; g < full; g += 16)
#pragma unroll
          for (int half = 0; half < 2; ++half)
            tma_store_3d(&tm_o, st_head + half * (kBM * 128) + (r0 + g) * 128, half * 32, us.z + hh,
                         us.y + r0 + g);
        bulk_commit();
      }
      if (lane >= full && lane < nrows) {
        // a row outside the whole 16-row groups (a unit shorter than 128
        // rows): straight from registers
        float4* dst = reinterpret_cast<float4*>(
            p.out + (static_cast<long long>(us.y + r) * p.hq + us.z + hh) * kD);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            dst[cc * 8 + e / 4] =
                make_float4(__uint_as_float(o[cc][e]) * inv, __uint_as_float(o[cc][e + 1]) * inv,
                            __uint_as_float(o[cc][e + 2]) * inv, __uint_as_float(o[cc][e + 3]) * inv);
      }
    }
    if (lane == 0) bulk_wait_all();                     // the output stores are complete
    if (threadIdx.x == 0) {
      // units of sequences with inconsistent lengths were skipped: say so
      for (int k = 0;; ++k) {
        const long long u = unit_index(k, c, G);
        if (u >= n_units) break;
        Unit x;
        unit_info<NH, K>(p, tab, static_cast<int>(u), x);
        if (x.bad) report(p.status, x.bad_ctx ? TVL_DEV_BAD_CONTEXT_LEN : TVL_DEV_BAD_QUERY_LEN);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
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
              const cuuint64_t* strides, const cuuint32_t* box,
              CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, type, rank, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int NH>
cudaError_t launch_nh(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& to, const Params& p, int num_seqs, int num_sms,
                      cudaStream_t stream) {
  using C = Cfg<NH>;
  // once per device: the shared-memory limit, and the check that the
  // register split fits the registers the block is launched with
  static PerDeviceOnce once;
  cudaError_t e = once.run([] {
    cudaError_t r = cudaFuncSetAttribute(prefill_kernel<NH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (r != cudaSuccess || NH != 2) return r;
    cudaFuncAttributes fa;
    r = cudaFuncGetAttributes(&fa, prefill_kernel<NH>);
    if (r != cudaSuccess) return r;
    if (fa.numRegs * C::kThreads < 2 * 128 * kRegsSoftmax + 128 * kRegsAux) {
      set_last_error("prefill kernel register allocation smaller than its register split");
      return cudaErrorInvalidConfiguration;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (at most one per unit), each walking its units
  const long long units = static_cast<long long>(num_seqs) * p.n_qtiles * (p.hq / NH);
  dim3 grid(static_cast<unsigned>(units < num_sms ? units : num_sms));
  // A plain launch, not a programmatic-dependent one: the units are dealt to
  // the CTAs up front, so the CTAs should start together.  Launched early
  // behind a kernel that is still draining, they started over that kernel's
  // tail and the last to start set the end (chunked prefill after the paged
  // write: 176 us per step against 157 us).
  prefill_kernel<NH><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to;
  {
    // the fp32 output [Tq, Hq, D]: 16-row x 32-column tiles of one head
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD),
                                static_cast<cuuint64_t>(a.num_q_heads),
                                static_cast<cuuint64_t>(a.total_q_tokens)};
    const cuuint64_t strides[2] = {kD * 4, static_cast<cuuint64_t>(a.num_q_heads) * kD * 4};
    const cuuint32_t box[3] = {32, 1, 16};
    if (!make_map(&to, a.out, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return cudaErrorInvalidValue;
  }
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
  if (p.group >= 2) return launch_nh<2>(tq, tk, tv, to, p, a.num_seqs, a.num_sms, stream);
  return launch_nh<1>(tq, tk, tv, to, p, a.num_seqs, a.num_sms, stream);
}

}  // namespace tvl
