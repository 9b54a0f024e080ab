// pkv_blocks.cpp -- host-side block manager: the pre-allocated block pool's free list,
// per-block reference counts, and per-sequence page tables.
//
// "Efficient AI Lecture 13: LLM Deployment Techniques", section "PagedAttention / How it
// works": split each sequence's cache into logical blocks, allocate physical blocks on
// demand, store them non-contiguously, translate through a block table; shared prompt
// prefixes can reuse physical blocks (parallel sampling, beam search).  "Lesson 4", 4.2:
// a global pre-allocated block pool with dynamic allocation and release.
//
// Sharing works by reference counts: fork() gives a child sequence the parent's blocks
// (each count + 1).  Appending to a sequence whose last block is shared and partly
// filled first copies that block (copy on write): the manager takes a fresh block,
// reports the (source, destination) pair for pkv_copy_blocks, and moves its own reference.
// Full shared blocks are never written again, so they stay shared.
//
// Sliding window ("LLM/MLLM inference optimisation", 2.3: keep only the most recent window
// of the cache): release_before() gives back the blocks wholly behind a window; their
// table entries become -1 while positions keep counting, so the memory a sequence holds
// stays bounded by its window.
#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "pagedkv.h"

struct pkv_block_manager {
  struct Seq {
    bool live = false;
    int32_t len = 0;       // tokens in the cache (positions, released ones included)
    int32_t released = 0;  // leading blocks given back by release_before (entries -1)
    std::vector<int32_t> blocks;
  };
  int64_t num_blocks = 0;
  int max_seqs = 0;
  int max_blocks_per_seq = 0;
  std::vector<int32_t> refcount;
  std::vector<int32_t> free_blocks;  // a stack; allocation pops from the back
  std::vector<Seq> seqs;
  std::vector<int> free_seqs;
  int live = 0;
  mutable std::mutex mu;
};

namespace {

constexpr int kBlock = PKV_BLOCK_SIZE;

bool seq_ok(const pkv_block_manager* m, int s) {
  return s >= 0 && s < m->max_seqs && m->seqs[size_t(s)].live;
}

int32_t take_block(pkv_block_manager* m) {
  const int32_t b = m->free_blocks.back();
  m->free_blocks.pop_back();
  m->refcount[size_t(b)] = 1;
  return b;
}

void drop_block(pkv_block_manager* m, int32_t b) {
  if (b < 0) return;  // released entry
  if (--m->refcount[size_t(b)] == 0) m->free_blocks.push_back(b);
}

}  // namespace

extern "C" {

PKV_API pkv_status pkv_block_manager_create(int64_t num_blocks, int max_seqs, int max_blocks_per_seq,
                                            pkv_block_manager** out) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks < 1 || num_blocks > INT32_MAX || max_seqs < 1 || max_blocks_per_seq < 1)
    return PKV_ERR_INVALID_ARG;
  auto* m = new (std::nothrow) pkv_block_manager;
  if (!m) return PKV_ERR_CAPACITY;
  try {
    m->num_blocks = num_blocks;
    m->max_seqs = max_seqs;
    m->max_blocks_per_seq = max_blocks_per_seq;
    m->refcount.assign(size_t(num_blocks), 0);
    m->free_blocks.resize(size_t(num_blocks));
    // Pop order 0, 1, 2, ...: the stack holds the ids in reverse.
    for (int64_t i = 0; i < num_blocks; ++i) m->free_blocks[size_t(i)] = int32_t(num_blocks - 1 - i);
    m->seqs.resize(size_t(max_seqs));
    m->free_seqs.resize(size_t(max_seqs));
    for (int i = 0; i < max_seqs; ++i) m->free_seqs[size_t(i)] = max_seqs - 1 - i;
  } catch (...) {
    delete m;
    return PKV_ERR_CAPACITY;
  }
  *out = m;
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_destroy(pkv_block_manager* m) {
  delete m;
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_add_sequence(pkv_block_manager* m, int* seq) {
  if (!m || !seq) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (m->free_seqs.empty()) return PKV_ERR_CAPACITY;
  const int s = m->free_seqs.back();
  m->free_seqs.pop_back();
  auto& q = m->seqs[size_t(s)];
  q.live = true;
  q.len = 0;
  q.released = 0;
  q.blocks.clear();
  ++m->live;
  *seq = s;
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_fork(pkv_block_manager* m, int parent, int* child) {
  if (!m || !child) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (!seq_ok(m, parent)) return PKV_ERR_INVALID_ARG;
  if (m->free_seqs.empty()) return PKV_ERR_CAPACITY;
  const int c = m->free_seqs.back();
  m->free_seqs.pop_back();
  const auto& p = m->seqs[size_t(parent)];
  auto& q = m->seqs[size_t(c)];
  q.live = true;
  q.len = p.len;
  q.released = p.released;
  q.blocks = p.blocks;
  for (int32_t b : q.blocks)
    if (b >= 0) ++m->refcount[size_t(b)];
  ++m->live;
  *child = c;
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_free_sequence(pkv_block_manager* m, int seq) {
  if (!m) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (!seq_ok(m, seq)) return PKV_ERR_INVALID_ARG;
  auto& q = m->seqs[size_t(seq)];
  for (int32_t b : q.blocks) drop_block(m, b);
  q.blocks.clear();
  q.len = 0;
  q.released = 0;
  q.live = false;
  m->free_seqs.push_back(seq);
  --m->live;
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_append(pkv_block_manager* m, const int* seqs,
                                            const int* num_new_tokens, int n,
                                            int32_t* slot_mapping, int32_t* copy_pairs,
                                            int max_copies, int* num_copies) {
  if (!m || n < 0 || (n > 0 && (!seqs || !num_new_tokens || !slot_mapping)) || !num_copies)
    return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  *num_copies = 0;
  // Validate and count what the call needs before changing anything.
  int64_t need_blocks = 0;
  int need_copies = 0;
  for (int i = 0; i < n; ++i) {
    const int s = seqs[i];
    if (!seq_ok(m, s) || num_new_tokens[i] < 0) return PKV_ERR_INVALID_ARG;
    for (int k = 0; k < i; ++k)
      if (seqs[k] == s) return PKV_ERR_INVALID_ARG;  // one entry per sequence
    const auto& q = m->seqs[size_t(s)];
    const int64_t len = q.len, add = num_new_tokens[i];
    if (add == 0) continue;
    const int64_t blocks_after = (len + add + kBlock - 1) / kBlock;
    if (blocks_after > m->max_blocks_per_seq) return PKV_ERR_CAPACITY;
    need_blocks += blocks_after - int64_t(q.blocks.size());
    if (len % kBlock != 0 && m->refcount[size_t(q.blocks.back())] > 1) {
      ++need_blocks;  // copy of the shared partial last block
      ++need_copies;
    }
  }
  if (need_blocks > int64_t(m->free_blocks.size())) return PKV_ERR_CAPACITY;
  if (need_copies > 0 && (!copy_pairs || max_copies < need_copies)) return PKV_ERR_INVALID_ARG;

  int64_t out = 0;
  int copies = 0;
  for (int i = 0; i < n; ++i) {
    auto& q = m->seqs[size_t(seqs[i])];
    for (int k = 0; k < num_new_tokens[i]; ++k) {
      const int32_t pos = q.len;
      const int32_t j = pos / kBlock, off = pos % kBlock;
      if (off == 0) {
        q.blocks.push_back(take_block(m));
      } else if (m->refcount[size_t(q.blocks[size_t(j)])] > 1) {
        const int32_t src = q.blocks[size_t(j)];
        const int32_t dst = take_block(m);
        drop_block(m, src);
        q.blocks[size_t(j)] = dst;
        copy_pairs[2 * copies] = src;
        copy_pairs[2 * copies + 1] = dst;
        ++copies;
      }
      slot_mapping[out++] = q.blocks[size_t(j)] * kBlock + off;
      ++q.len;
    }
  }
  *num_copies = copies;
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_truncate(pkv_block_manager* m, int seq, int num_tokens) {
  if (!m) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (!seq_ok(m, seq)) return PKV_ERR_INVALID_ARG;
  auto& q = m->seqs[size_t(seq)];
  if (num_tokens < 0 || num_tokens > q.len || num_tokens < q.released * kBlock)
    return PKV_ERR_INVALID_ARG;
  const size_t keep = size_t((num_tokens + kBlock - 1) / kBlock);
  while (q.blocks.size() > keep) {
    drop_block(m, q.blocks.back());
    q.blocks.pop_back();
  }
  q.len = num_tokens;
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_release_before(pkv_block_manager* m, int seq, int token) {
  if (!m) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (!seq_ok(m, seq)) return PKV_ERR_INVALID_ARG;
  auto& q = m->seqs[size_t(seq)];
  if (token < 0 || token > q.len) return PKV_ERR_INVALID_ARG;
  const int32_t upto = token / kBlock;  // blocks 0 .. upto-1 hold only tokens before `token`
  for (int32_t j = q.released; j < upto; ++j) {
    drop_block(m, q.blocks[size_t(j)]);
    q.blocks[size_t(j)] = -1;
  }
  if (upto > q.released) q.released = upto;
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_tables(const pkv_block_manager* m, const int* seqs, int n,
                                            int32_t* block_tables, int32_t* context_lens) {
  if (!m || n < 0 || (n > 0 && (!seqs || !block_tables || !context_lens))) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  for (int i = 0; i < n; ++i)
    if (!seq_ok(m, seqs[i])) return PKV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const auto& q = m->seqs[size_t(seqs[i])];
    int32_t* row = block_tables + int64_t(i) * m->max_blocks_per_seq;
    std::fill(row, row + m->max_blocks_per_seq, -1);
    std::copy(q.blocks.begin(), q.blocks.end(), row);
    context_lens[i] = q.len;
  }
  return PKV_OK;
}

PKV_API pkv_status pkv_block_manager_stats(const pkv_block_manager* m, int64_t* free_blocks,
                                           int* live_seqs) {
  if (!m) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(m->mu);
  if (free_blocks) *free_blocks = int64_t(m->free_blocks.size());
  if (live_seqs) *live_seqs = m->live;
  return PKV_OK;
}

PKV_API int32_t pkv_block_manager_refcount(const pkv_block_manager* m, int32_t block) {
  if (!m || block < 0 || int64_t(block) >= m->num_blocks) return -1;
  std::lock_guard<std::mutex> lock(m->mu);
  return m->refcount[size_t(block)];
}

}  // extern "C"
