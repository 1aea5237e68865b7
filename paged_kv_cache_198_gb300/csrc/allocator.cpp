// allocator.cpp -- host block allocator: the control plane that decides
// which physical block and slot every token of every sequence occupies.
//
// [nano-vLLM guide ch. 2: the CPU control plane drives the GPU data plane;
// ch. 4 "PagedAttention": the KV cache as virtual memory made of fixed-size
// blocks, handed out by a block allocator so that memory is not lost to
// fragmentation; ch. 5 "The Scheduler": continuous batching, sequences join
// and leave the batch every step; ch. 7 "Prefix Caching": sequences share
// the blocks of a common prefix.]
//
// Blocks are reference counted.  fork() lets a new sequence share all of
// another's blocks; the first append that would write into a shared,
// partially filled block gives the writer a private copy (copy-on-write) and
// queues a (source, destination) pair that the caller executes on the device
// with tvl_copy_blocks before the write.  Every call is all-or-nothing: when
// the pool cannot cover it, nothing changes and TVL_ERR_OUT_OF_BLOCKS is
// returned.  Calls on one allocator are serialised by a mutex.
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/tvl.h"
#include "kernels.h"

struct tvl_allocator {
  std::mutex mu;
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> free_blocks;          // stack of free physical blocks
  std::vector<int32_t> refcount;             // per physical block
  struct Seq {
    bool live = false;
    long long tokens = 0;
    std::vector<int32_t> blocks;
  };
  std::vector<Seq> seqs;
  std::vector<int> free_ids;
  std::vector<int32_t> copy_src, copy_dst;   // pending copy-on-write pairs

  int32_t take_block() {
    const int32_t b = free_blocks.back();
    free_blocks.pop_back();
    refcount[b] = 1;
    return b;
  }
  void release_block(int32_t b) {
    if (--refcount[b] == 0) free_blocks.push_back(b);
  }
  Seq* seq(int id) {
    if (id < 0 || id >= static_cast<int>(seqs.size()) || !seqs[id].live) return nullptr;
    return &seqs[id];
  }
  int new_id() {
    int id;
    if (!free_ids.empty()) {
      id = free_ids.back();
      free_ids.pop_back();
    } else {
      id = static_cast<int>(seqs.size());
      seqs.emplace_back();
    }
    seqs[id] = Seq();
    seqs[id].live = true;
    return id;
  }
};

namespace {

tvl_status bad(const char* msg) {
  tvl::set_last_error(msg);
  return TVL_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

tvl_status tvl_allocator_create(int num_blocks, int block_size, tvl_allocator** out) {
  if (!out) return bad("null output pointer");
  if (num_blocks <= 0 || block_size <= 0) return bad("num_blocks and block_size must be > 0");
  auto* a = new tvl_allocator();
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->refcount.assign(num_blocks, 0);
  a->free_blocks.reserve(num_blocks);
  for (int b = num_blocks - 1; b >= 0; --b) a->free_blocks.push_back(b);   // hands out 0, 1, ...
  *out = a;
  return TVL_OK;
}

void tvl_allocator_destroy(tvl_allocator* a) { delete a; }

tvl_status tvl_allocator_new_sequence(tvl_allocator* a, int* seq) {
  if (!a || !seq) return bad("null argument");
  std::lock_guard<std::mutex> lock(a->mu);
  *seq = a->new_id();
  return TVL_OK;
}

tvl_status tvl_allocator_fork(tvl_allocator* a, int parent, int* child) {
  if (!a || !child) return bad("null argument");
  std::lock_guard<std::mutex> lock(a->mu);
  if (!a->seq(parent)) return bad("no such sequence");
  const int id = a->new_id();
  tvl_allocator::Seq& p = a->seqs[parent];   // re-fetch: new_id may grow the vector
  a->seqs[id].tokens = p.tokens;
  a->seqs[id].blocks = p.blocks;
  for (int32_t b : p.blocks) ++a->refcount[b];
  *child = id;
  return TVL_OK;
}

tvl_status tvl_allocator_append(tvl_allocator* a, int seq, int num_tokens, int32_t* slots) {
  if (!a) return bad("null allocator");
  if (num_tokens < 0) return bad("num_tokens < 0");
  if (num_tokens > 0 && !slots) return bad("null slots");
  std::lock_guard<std::mutex> lock(a->mu);
  tvl_allocator::Seq* s = a->seq(seq);
  if (!s) return bad("no such sequence");
  const long long bs = a->block_size;
  const long long before = static_cast<long long>(s->blocks.size());
  const long long after = (s->tokens + num_tokens + bs - 1) / bs;
  const bool partial = s->tokens % bs != 0;
  const bool cow = num_tokens > 0 && partial && a->refcount[s->blocks.back()] > 1;
  const long long need = (after - before) + (cow ? 1 : 0);
  if (need > static_cast<long long>(a->free_blocks.size())) {
    tvl::set_last_error("block pool exhausted");
    return TVL_ERR_OUT_OF_BLOCKS;
  }
  if (cow) {
    const int32_t old = s->blocks.back();
    const int32_t fresh = a->take_block();
    a->copy_src.push_back(old);
    a->copy_dst.push_back(fresh);
    a->release_block(old);
    s->blocks.back() = fresh;
  }
  for (int i = 0; i < num_tokens; ++i) {
    const long long pos = s->tokens + i;
    if (pos % bs == 0) s->blocks.push_back(a->take_block());
    slots[i] = static_cast<int32_t>(s->blocks[pos / bs] * bs + pos % bs);
  }
  s->tokens += num_tokens;
  return TVL_OK;
}

tvl_status tvl_allocator_free_sequence(tvl_allocator* a, int seq) {
  if (!a) return bad("null allocator");
  std::lock_guard<std::mutex> lock(a->mu);
  tvl_allocator::Seq* s = a->seq(seq);
  if (!s) return bad("no such sequence");
  for (int32_t b : s->blocks) a->release_block(b);
  *s = tvl_allocator::Seq();
  a->free_ids.push_back(seq);
  return TVL_OK;
}

tvl_status tvl_allocator_context_len(tvl_allocator* a, int seq, long long* len) {
  if (!a || !len) return bad("null argument");
  std::lock_guard<std::mutex> lock(a->mu);
  tvl_allocator::Seq* s = a->seq(seq);
  if (!s) return bad("no such sequence");
  *len = s->tokens;
  return TVL_OK;
}

tvl_status tvl_allocator_build_tables(tvl_allocator* a, const int* seqs, int n,
                                      int max_blocks_per_seq, int32_t* block_tables,
                                      int32_t* context_lens) {
  if (!a || (n > 0 && (!seqs || !block_tables || !context_lens))) return bad("null argument");
  if (n < 0 || max_blocks_per_seq <= 0) return bad("bad size");
  std::lock_guard<std::mutex> lock(a->mu);
  for (int i = 0; i < n; ++i) {
    tvl_allocator::Seq* s = a->seq(seqs[i]);
    if (!s) return bad("no such sequence");
    if (static_cast<long long>(s->blocks.size()) > max_blocks_per_seq)
      return bad("sequence longer than max_blocks_per_seq blocks");
    if (s->tokens > INT32_MAX) return bad("sequence too long");
  }
  for (int i = 0; i < n; ++i) {
    const tvl_allocator::Seq& s = a->seqs[seqs[i]];
    int32_t* row = block_tables + static_cast<long long>(i) * max_blocks_per_seq;
    const int nb = static_cast<int>(s.blocks.size());
    for (int b = 0; b < max_blocks_per_seq; ++b) row[b] = b < nb ? s.blocks[b] : -1;
    context_lens[i] = static_cast<int32_t>(s.tokens);
  }
  return TVL_OK;
}

tvl_status tvl_allocator_take_copies(tvl_allocator* a, int32_t* src, int32_t* dst,
                                     int capacity, int* count) {
  if (!a || !count) return bad("null argument");
  std::lock_guard<std::mutex> lock(a->mu);
  const int n = static_cast<int>(a->copy_src.size());
  *count = n;
  if (n == 0) return TVL_OK;
  if (!src || !dst || capacity < n) {
    tvl::set_last_error("copy list larger than the capacity given");
    return TVL_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; ++i) {
    src[i] = a->copy_src[i];
    dst[i] = a->copy_dst[i];
  }
  a->copy_src.clear();
  a->copy_dst.clear();
  return TVL_OK;
}

tvl_status tvl_allocator_stats(tvl_allocator* a, tvl_allocator_stats_t* st) {
  if (!a || !st) return bad("null argument");
  std::lock_guard<std::mutex> lock(a->mu);
  st->num_blocks = a->num_blocks;
  st->free_blocks = static_cast<int>(a->free_blocks.size());
  st->live_sequences = 0;
  st->tokens = 0;
  st->shared_blocks = 0;
  st->slack_slots = 0;
  for (const auto& s : a->seqs) {
    if (!s.live) continue;
    ++st->live_sequences;
    st->tokens += s.tokens;
    st->slack_slots += static_cast<long long>(s.blocks.size()) * a->block_size - s.tokens;
  }
  for (int b = 0; b < a->num_blocks; ++b)
    if (a->refcount[b] > 1) ++st->shared_blocks;
  return TVL_OK;
}

}  // extern "C"
