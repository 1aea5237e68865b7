/*
 * tvl.h -- C ABI of libtvl.so, a GB300 (sm_103a) implementation of the paged
 * attention hot path: the slot-mapped paged KV-cache write, PagedAttention
 * decode (single pass or split-K with a log-sum-exp merge), the two fused
 * into one decode-step call, and chunked causal prefill over a cached
 * prefix; around them the rotary embedding fused into the write, block
 * copies for copy-on-write, and a host block allocator.
 *
 * Sources of the method (web pages on tiny-vLLM and nano-vLLM):
 *   [tiny-vllm README]  "tiny-vllm" README, Korean translation: feature list
 *                       ("KV cache", "online softmax, FlashAttention style",
 *                       "PagedAttention") and the curriculum entries
 *                       "Attention", "GQA", "Softmax", "Causal mask",
 *                       "Prefill vs decode", "Online softmax",
 *                       "Paged Attention", "Paged KV cache",
 *                       "Paged Attention CUDA kernel".
 *   [Tiny-vLLM digest]  "Tiny-vLLM: C++와 CUDA로 만드는 고성능 LLM 추론 엔진",
 *                       section "Core Mechanics" (bf16, every op a CUDA
 *                       kernel, KV cache, online softmax, PagedAttention, GQA,
 *                       causal mask) and section "Evidence" (CUDA return codes
 *                       must be checked).
 *   [nano-vLLM guide]   "LLM 추론(Inference)이 실제로 어떻게 작동하는지에 대한 11장
 *                       분량의 인터랙티브 가이드", chapter 4 "PagedAttention" (the
 *                       KV cache as virtual memory made of fixed-size blocks),
 *                       chapter 6 "Prefill vs Decode", chapter 7 "Prefix
 *                       Caching", chapter 10 "The Optimization Stack".
 *
 * Common conventions
 * ------------------
 * Shapes: S = num_seqs, Hq = num_q_heads, Hkv = num_kv_heads, G = Hq / Hkv,
 *   D = head_dim, bs = block_size, NB = num_blocks (physical blocks in the
 *   pool), MB = max_blocks_per_seq (columns of block_tables).
 * Element types: q, K and V are bfloat16 (passed as void*, 2 bytes each);
 *   attention outputs are float32; all metadata is int32.
 * Cache layout: k_cache and v_cache are each a contiguous bf16 array
 *   [NB, bs, Hkv, D].  Token slot `x = block * bs + offset` is row x of the
 *   flat view [NB * bs, Hkv * D]; one physical block is one contiguous run of
 *   bs * Hkv * D * 2 bytes.
 * Block table: block_tables is int32 [S, MB], row-major.  Logical token j of
 *   sequence s lives in physical block block_tables[s * MB + j / bs], at
 *   offset j % bs.  Entries at or beyond ceil(context_lens[s] / bs) are never
 *   read.  Two rows may name the same physical block (shared prefixes).
 * GQA: query head h reads KV head h / G.
 * Scores: s_j = scale * sum_d q[d] * k_j[d], accumulated in float32.
 * Pointers: every pointer except `stream` and a zero-size workspace is a
 *   device pointer, owned by the caller, and must be 16-byte aligned.  The
 *   library allocates no device memory and frees nothing.
 * Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream).  A non-OK return means nothing was launched.
 * Errors: arguments are validated on the host before any launch.  Kernels
 *   never trap: an out-of-range block id, slot or context length found on the
 *   device is replaced by a safe value, the work it touches is undefined, and
 *   a bit is set in a per-device status word read by tvl_get_device_status().
 * Threads: calls are thread-safe; tvl_last_error() is per thread.
 */
#ifndef TVL_H
#define TVL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TVL_OK = 0,
  TVL_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or shape     */
  TVL_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim 128)  */
  TVL_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required     */
  TVL_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed              */
  TVL_ERR_DEVICE_CHECK = 5,  /* a kernel found bad metadata (status word set)  */
  TVL_ERR_OUT_OF_BLOCKS = 6  /* allocator: the block pool cannot cover a call  */
} tvl_status;

/* Bits of the device status word (tvl_get_device_status). */
#define TVL_DEV_BAD_SLOT        0x1  /* slot_mapping entry >= NB * bs            */
#define TVL_DEV_BAD_BLOCK_ID    0x2  /* block table entry outside [0, NB)        */
#define TVL_DEV_BAD_CONTEXT_LEN 0x4  /* context length < 0 or > MB * bs          */
#define TVL_DEV_BAD_QUERY_LEN   0x8  /* prefill: query rows outside [0, Tq),
                                        more than max_q_len, or more than the
                                        context length                          */
#define TVL_DEV_TIMEOUT         0x10 /* a kernel's bounded wait gave up (~1 s);
                                        its CTA left after its copies landed    */
#define TVL_DEV_NONFINITE       0x20 /* prefill: an output row is not finite --
                                        a V value with |v| > 65504 (beyond the
                                        fp16 range its P.V uses) or non-finite
                                        inputs                                  */

/*
 * Paged KV write [tiny-vllm README, curriculum "Paged KV cache" and "Why KV
 * cache exists"]: for every t in [0, T) with slot_mapping[t] >= 0,
 *   k_cache row slot_mapping[t] <- k_new[t]   and   v_cache row <- v_new[t],
 * where a row is Hkv * D bf16 values.  Rows with a negative slot are skipped.
 * The copy is bit-exact.  Slots must be distinct (duplicates: which writer
 * wins is unspecified).  A slot >= NB * bs is skipped and sets
 * TVL_DEV_BAD_SLOT.
 *   k_new, v_new : bf16 [T, Hkv, D]   (device, read)
 *   k_cache, v_cache : bf16 [NB, bs, Hkv, D] (device, written in place)
 *   slot_mapping : int32 [T]          (device, read)
 * T == 0 is valid and launches nothing.  Supported: D in {64};
 * Hkv * D * 2 a multiple of 16 bytes.
 */
tvl_status tvl_paged_kv_write(const void* k_new, const void* v_new,
                              void* k_cache, void* v_cache,
                              const int32_t* slot_mapping, int num_tokens,
                              int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, void* stream);

/*
 * Rotary position embedding fused into the paged KV write [tiny-vllm README,
 * curriculum "RoPE" and "Paged KV cache"; Tiny-vLLM digest, "Core
 * Mechanics"]: for every token t, each head vector of q[t] (in place, when q
 * is not NULL) and of k_new[t] has its pairs (x_i, x_{i+D/2}), i < D/2,
 * rotated by the angle a = positions[t] * rope_theta^(-2i/D):
 *   x_i <- x_i cos a - x_{i+D/2} sin a,  x_{i+D/2} <- x_{i+D/2} cos a + x_i sin a,
 * rounded to bf16 (the angle is reduced in double precision, the rotation is
 * fp32).  Then, for slot_mapping[t] >= 0, the rotated K row and the V row are
 * stored at that slot exactly as tvl_paged_kv_write does (negative slots:
 * q is still rotated, nothing is stored).  k_new and v_new are not modified.
 *   q        : bf16 [T, Hq, D] or NULL (device, rotated in place)
 *   positions: int32 [T], absolute token positions >= 0 (device)
 * Each result is within one bf16 ulp of the double-precision definition plus
 * the fp32 rounding of the rotation, at most 2^-21 * (|x_i| + |x_{i+D/2}|)
 * (visible only where the two products cancel).  Supported: D == 64.
 */
tvl_status tvl_rope_paged_kv_write(void* q, const void* k_new, const void* v_new,
                                   void* k_cache, void* v_cache,
                                   const int32_t* slot_mapping,
                                   const int32_t* positions, int num_tokens,
                                   int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, int num_blocks,
                                   float rope_theta, void* stream);

/*
 * Workspace needed by tvl_paged_attention_decode for these sizes, written to
 * *bytes.  The arguments mean what they mean in the decode call and are
 * validated the same way.  With partition_size == 0 the answer depends on the
 * current device's SM count.  A zero answer means the call needs no
 * workspace.
 */
tvl_status tvl_paged_attention_decode_workspace_size(
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int max_blocks_per_seq, int block_size, int partition_size,
    size_t* bytes);

/*
 * PagedAttention decode [tiny-vllm README, curriculum "Attention", "GQA",
 * "Softmax", "Online softmax", "Paged Attention", "Paged Attention CUDA
 * kernel"; nano-vLLM guide ch. 4 "PagedAttention", ch. 6 "Prefill vs Decode"]:
 * one query token per sequence attends to all context_lens[s] cached tokens
 * of that sequence (the token written by this step's tvl_paged_kv_write is
 * included; no mask):
 *   out[s, h, :] = sum_j softmax_j(s_j) * V_j,   j in [0, context_lens[s]),
 * with K_j, V_j gathered through the block table from KV head h / G.
 * context_lens[s] == 0 gives a zero output row.
 *   out          : float32 [S, Hq, D]  (device, written)
 *   q            : bf16 [S, Hq, D]     (device, read)
 *   block_tables : int32 [S, MB]; context_lens : int32 [S] (device, read)
 * partition_size selects how the context is split (all splits are merged
 * exactly by log-sum-exp, the associative form of the online softmax):
 *   0   the library balances the blocks over one CTA per SM, each sequence
 *       start counted as one 32-token stage more (its fixed cost); a
 *       sequence may be cut anywhere on a block boundary.
 *   >0  fixed windows [p * P, (p + 1) * P) of P tokens from position 0 (the
 *       last one partial); P must be a multiple of block_size.  P >= MB * bs
 *       is a single pass per sequence and needs no workspace.  With more
 *       windows than SMs, one CTA per SM walks them in equal contiguous
 *       ranges; the results are the same either way.
 * workspace: device memory of at least the size reported by
 *   tvl_paged_attention_decode_workspace_size (may be NULL when that is 0);
 *   its contents on entry are ignored and on exit unspecified.
 * Supported: D == 64, G in {1, 2, 4, 8}, bs in {16, 32, 64, 128}, Hkv <= 8 or a
 * multiple of 8 (for G == 8: Hkv <= 4 or a multiple of 4).
 */
tvl_status tvl_paged_attention_decode(
    float* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, int max_blocks_per_seq, float scale, int partition_size,
    void* workspace, size_t workspace_bytes, void* stream);

/*
 * One decode step in a single call [tiny-vllm README, curriculum "Why KV
 * cache exists", "Paged KV cache", "Paged Attention"; nano-vLLM guide ch. 4
 * "PagedAttention", ch. 5 "The Scheduler" (each step appends one token per
 * running sequence and attends over its cache)]: for every sequence s with
 * context_lens[s] >= 1, the new token's K and V rows (k_new[s], v_new[s],
 * bf16 [S, Hkv, D], device, read) are written into the cache at position
 * context_lens[s] - 1, i.e. slot block_tables[s][(ctx - 1) / bs] * bs +
 * (ctx - 1) % bs -- the slot a slot_mapping of this step holds -- and then
 * the decode of tvl_paged_attention_decode runs over the updated cache.
 * Same results as tvl_paged_kv_write with that slot_mapping followed by
 * tvl_paged_attention_decode (the cache bit for bit, the output to the same
 * bits), with one kernel boundary less: the CTA that streams a sequence's
 * last block writes the row before it copies the block.
 * All other arguments, layouts, the workspace and the errors are those of
 * tvl_paged_attention_decode; k_new and v_new must be 16-byte aligned.  A
 * sequence with context_lens[s] == 0 writes nothing.  A block-table entry
 * that is out of range is reported (TVL_DEV_BAD_BLOCK_ID) and its row is not
 * written.
 */
tvl_status tvl_paged_decode_step(
    float* out, const void* q, const void* k_new, const void* v_new,
    void* k_cache, void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int num_blocks,
    int max_blocks_per_seq, float scale, int partition_size, void* workspace,
    size_t workspace_bytes, void* stream);

/*
 * Chunked causal prefill over a cached prefix [tiny-vllm README, curriculum
 * "Prefill vs decode", "Attention", "GQA", "Causal mask", "Online softmax",
 * "Paged Attention"; nano-vLLM guide ch. 6 "Prefill vs Decode", ch. 7
 * "Prefix Caching", ch. 10 "The Optimization Stack" (FlashAttention)]:
 * sequence s owns query tokens [query_start_loc[s], query_start_loc[s+1]),
 * Lq = their count, which are the LAST Lq tokens of its context_lens[s]
 * tokens; their K/V must already be in the paged cache (tvl_paged_kv_write).
 * Query row i sits at absolute position p = context_lens[s] - Lq + i and
 * attends to cached tokens 0..p inclusive (causal):
 *   out[t, h, :] = sum_{j<=p} softmax_j(s_j) * V_j.
 *   out  : float32 [Tq, Hq, D]; q : bf16 [Tq, Hq, D]        (device)
 *   query_start_loc : int32 [S + 1], non-decreasing, [0] = 0, [S] = Tq
 *   block_tables : int32 [S, MB]; context_lens : int32 [S]  (device)
 * max_q_len must be >= every Lq (it sets the number of 128-row query tiles
 * per sequence).  On the device, a sequence whose rows would leave [0, Tq)
 * (query_start_loc[s] < 0, a decreasing entry, or query_start_loc[s+1] > Tq),
 * whose Lq exceeds max_q_len rounded up to 128, or whose Lq exceeds
 * context_lens[s] is reported (TVL_DEV_BAD_QUERY_LEN), as is a context
 * longer than MB * bs (TVL_DEV_BAD_CONTEXT_LEN); such a sequence's rows are
 * left unwritten and nothing outside `out` is touched.
 * Precision: P and V enter the P.V product as fp16 (P rounded to 2^-11
 * relative, exact where the sum is taken in fp32).  V values must lie within
 * the fp16 range, |v| <= 65504 (bf16 can hold more): a larger one makes
 * the output rows of the query tiles whose key range holds it inf or NaN,
 * and any output row that is not finite sets TVL_DEV_NONFINITE.  V values
 * below 2^-14 in magnitude keep an absolute error under 2^-25.
 * Supported: D == 64, G in {1, 2, 4, 8}, bs in {16, 32, 64, 128}, Hkv <= 255,
 * num_seqs <= 65535 and num_seqs * ceil(max_q_len / 128) * Hq < 2^31
 * (else TVL_ERR_UNSUPPORTED).  The call launches one kernel (at most one
 * block per SM) and allocates nothing.
 */
tvl_status tvl_paged_attention_prefill(
    float* out, const void* q, const int32_t* query_start_loc,
    const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int total_q_tokens,
    int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, float scale,
    void* stream);

/*
 * Decode without a caller workspace.  No counterpart on the source pages: it
 * exists for callers that cannot allocate device memory where they decode --
 * an engine that gave all device memory to its KV pool up front, a plugin or
 * callback interface that hands over only input and output pointers, or a
 * thread that must not block on the driver's allocation lock.
 * Same arguments, layouts and results as tvl_paged_attention_decode, minus
 * the workspace: the split-K partial records go to one built-in device array
 * of 4 MiB (held by every GPU that loads the library until exit).  A call
 * that needs more scratch than that returns TVL_ERR_WORKSPACE and launches
 * nothing.  The call allocates and frees nothing.
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address once; make that first call before any stream
 * capture.  Calls share the array: nothing needs clearing between calls, but
 * calls that overlap on the GPU race on it.
 */
tvl_status tvl_paged_attention_decode_noalloc(
    float* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, int max_blocks_per_seq, float scale, int partition_size,
    void* stream);

/*
 * Block copy [nano-vLLM guide ch. 7 "Prefix Caching": sequences that share a
 * prefix share its blocks until one of them writes into a shared block]:
 * for i in [0, n), physical block dst[i] of both caches becomes a copy of
 * block src[i] (bs * Hkv * D bf16 values each), bit-exact.  The pairs must
 * not overlap (no block is both a source and a destination).  Ids outside
 * [0, NB) are skipped and set TVL_DEV_BAD_BLOCK_ID.
 *   k_cache, v_cache : bf16 [NB, bs, Hkv, D] (device, in place)
 *   src, dst         : int32 [n] (device)
 */
tvl_status tvl_copy_blocks(void* k_cache, void* v_cache, const int32_t* src,
                           const int32_t* dst, int n, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks,
                           void* stream);

/*
 * Host block allocator: the CPU control plane that hands out the physical
 * blocks and slots the kernels read [nano-vLLM guide ch. 2 (control plane vs
 * data plane), ch. 4 "PagedAttention" (block allocator, no fragmentation
 * beyond the last block of a sequence), ch. 5 "The Scheduler" (continuous
 * batching), ch. 7 "Prefix Caching" (shared prefix blocks)].  Host memory
 * only; calls on one allocator are serialised internally.  Every call is
 * all-or-nothing.
 */
typedef struct tvl_allocator tvl_allocator;

typedef struct {
  int num_blocks;        /* pool size                                        */
  int free_blocks;       /* blocks with no owner                             */
  int live_sequences;
  int shared_blocks;     /* blocks owned by more than one sequence           */
  long long tokens;      /* sum of the live sequences' lengths               */
  long long slack_slots; /* sum over sequences of unused slots in own blocks */
} tvl_allocator_stats_t;

/* A pool of num_blocks blocks of block_size tokens; *out owns it. */
tvl_status tvl_allocator_create(int num_blocks, int block_size,
                                tvl_allocator** out);
void tvl_allocator_destroy(tvl_allocator* allocator);
/* A new empty sequence; its id goes to *seq (ids of freed sequences are
 * reused). */
tvl_status tvl_allocator_new_sequence(tvl_allocator* allocator, int* seq);
/* A new sequence that shares every block (and the length) of `parent`. */
tvl_status tvl_allocator_fork(tvl_allocator* allocator, int parent, int* child);
/* Reserves the next num_tokens positions of `seq` and writes their cache
 * slots (block * bs + offset) to slots[0..num_tokens).  New blocks are taken
 * from the pool; if the sequence's last block is shared and partly filled it
 * is first replaced by a private copy, and the (old, new) pair is queued for
 * tvl_allocator_take_copies -- run those copies (tvl_copy_blocks) before
 * writing to the returned slots.  TVL_ERR_OUT_OF_BLOCKS if the pool cannot
 * cover the call (nothing changes). */
tvl_status tvl_allocator_append(tvl_allocator* allocator, int seq,
                                int num_tokens, int32_t* slots);
/* Releases the sequence's hold on its blocks and retires its id. */
tvl_status tvl_allocator_free_sequence(tvl_allocator* allocator, int seq);
tvl_status tvl_allocator_context_len(tvl_allocator* allocator, int seq,
                                     long long* len);
/* Row i of block_tables [n, max_blocks_per_seq] (host, -1 padded) and
 * context_lens[i] describe sequence seqs[i]: the arguments of the decode and
 * prefill calls for that batch. */
tvl_status tvl_allocator_build_tables(tvl_allocator* allocator,
                                      const int* seqs, int n,
                                      int max_blocks_per_seq,
                                      int32_t* block_tables,
                                      int32_t* context_lens);
/* Moves the queued copy-on-write pairs into src/dst (host, `capacity`
 * entries) and their number into *count.  If capacity is too small nothing is
 * moved, *count holds the number needed and TVL_ERR_INVALID_ARG is
 * returned. */
tvl_status tvl_allocator_take_copies(tvl_allocator* allocator, int32_t* src,
                                     int32_t* dst, int capacity, int* count);
tvl_status tvl_allocator_stats(tvl_allocator* allocator,
                               tvl_allocator_stats_t* stats);

/* Static description of a status code. */
const char* tvl_status_string(tvl_status status);

/* Detail of the last non-OK return on the calling thread ("" if none). */
const char* tvl_last_error(void);

/*
 * Reads and clears the current device's status word (TVL_DEV_* bits).  The
 * read is ordered after all prior work on `stream` and synchronises it.
 * Returns TVL_OK when the word was zero, TVL_ERR_DEVICE_CHECK when a bit was
 * set (the bits go to *bits if bits != NULL), TVL_ERR_CUDA on a CUDA error.
 */
tvl_status tvl_get_device_status(void* stream, uint32_t* bits);

/*
 * Self-test of the kernels' bounded waits (no counterpart on the pages).  It
 * launches one CTA that waits, with the same bounded mbarrier wait the
 * kernels use, on a barrier nothing arrives at: after the wait's limit (about
 * one second) it gives up and sets TVL_DEV_TIMEOUT in the status word, and
 * the context stays usable.  Asynchronous on `stream`; tests use it to check
 * that a wait that is never satisfied cannot hang the GPU.
 */
tvl_status tvl_selftest_bounded_wait(void* stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int tvl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TVL_H */
