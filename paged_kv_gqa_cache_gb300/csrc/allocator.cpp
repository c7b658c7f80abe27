// Host-side block allocator and per-sequence block tables (page "Модуль 12:
// Финальный проект: мини-движок инференса", task 12.1, qwen_serve/paged.py:
// BlockAllocator and SequenceCache), the bookkeeping that produces the block
// tables, slot mappings and lengths the attention kernels consume.
//
// What follows the page:
//   - fixed 16-token blocks, a reference count per block, a first-in
//     first-out free list (a new pool hands out 0, 1, 2, ...; a released block
//     joins the back);
//   - fork shares every block of the source sequence by reference, and the
//     first write into a shared, partly filled block copies it (allocate a
//     fresh block, copy, release the old one; task 12.1's copy-on-write
//     rule and its worked example);
//   - adopting a prefix retains full blocks and sets the length to their
//     tokens, so later writes never land in them;
//   - reserve/commit: room first, length moves only after the KV is written.
// What differs, on purpose:
//   - allocation is all or nothing (the page's loop could hand out part of a
//     request before failing, leaving blocks with no owner);
//   - the block copy itself runs on the GPU (pa_kv_block_copy): here the
//     copy is only recorded as a (src, dst) pair for the caller to enqueue;
//   - retain of a free block is refused (it would leave a referenced block in
//     the free list).
// Prefix hashing and eviction (the page's prefix cache) are not part of this
// library; a caller that keeps such a cache passes the shared blocks to
// pa_sequence_adopt_prefix.
#include <deque>
#include <vector>

#include "pagedattn.h"

struct pa_allocator {
  std::vector<int32_t> refcount;
  std::deque<int32_t> free_list;
  int64_t n_allocated = 0;
  int64_t n_cow = 0;
  std::vector<int32_t> copies;  // recorded (src, dst) pairs, flattened
  int32_t used = 0;             // blocks with refcount > 0
  int32_t shared = 0;           // blocks with refcount > 1
};

struct pa_sequence {
  pa_allocator *alloc = nullptr;
  std::vector<int32_t> blocks;
  int32_t length = 0;    // committed tokens
  int32_t reserved = 0;  // tokens reserved after them, not yet committed
};

namespace {

constexpr int32_t kBlockTokens = PA_BLOCK_SIZE;

bool in_pool(const pa_allocator *a, int32_t b) { return b >= 0 && b < (int32_t)a->refcount.size(); }

void ref_up(pa_allocator *a, int32_t b) {
  int32_t &r = a->refcount[b];
  if (r == 0) ++a->used;
  if (r == 1) ++a->shared;
  ++r;
}

void ref_down(pa_allocator *a, int32_t b) {
  int32_t &r = a->refcount[b];
  --r;
  if (r == 1) --a->shared;
  if (r == 0) {
    --a->used;
    a->free_list.push_back(b);
  }
}

int32_t take_free(pa_allocator *a) {
  const int32_t b = a->free_list.front();
  a->free_list.pop_front();
  ref_up(a, b);
  ++a->n_allocated;
  return b;
}

int32_t blocks_for(int64_t tokens) { return (int32_t)((tokens + kBlockTokens - 1) / kBlockTokens); }

}  // namespace

extern "C" {

pa_status pa_allocator_create(int32_t num_blocks, pa_allocator **out) {
  if (!out) return PA_ERR_NULL;
  *out = nullptr;
  if (num_blocks < 1) return PA_ERR_SHAPE;
  pa_allocator *a = new pa_allocator;
  a->refcount.assign((size_t)num_blocks, 0);
  for (int32_t b = 0; b < num_blocks; ++b) a->free_list.push_back(b);
  *out = a;
  return PA_OK;
}

void pa_allocator_destroy(pa_allocator *alloc) { delete alloc; }

pa_status pa_allocator_allocate(pa_allocator *alloc, int32_t n, int32_t *out) {
  if (!alloc) return PA_ERR_NULL;
  if (n < 0) return PA_ERR_SHAPE;
  if (n == 0) return PA_OK;
  if (!out) return PA_ERR_NULL;
  if ((size_t)n > alloc->free_list.size()) return PA_ERR_NO_BLOCKS;
  for (int32_t i = 0; i < n; ++i) out[i] = take_free(alloc);
  return PA_OK;
}

pa_status pa_allocator_retain(pa_allocator *alloc, int32_t block) {
  if (!alloc) return PA_ERR_NULL;
  if (!in_pool(alloc, block)) return PA_ERR_RANGE;
  if (alloc->refcount[block] == 0) return PA_ERR_STATE;
  ref_up(alloc, block);
  return PA_OK;
}

pa_status pa_allocator_release(pa_allocator *alloc, int32_t block) {
  if (!alloc) return PA_ERR_NULL;
  if (!in_pool(alloc, block)) return PA_ERR_RANGE;
  if (alloc->refcount[block] <= 0) return PA_ERR_STATE;
  ref_down(alloc, block);
  return PA_OK;
}

int32_t pa_allocator_refcount(const pa_allocator *alloc, int32_t block) {
  if (!alloc || !in_pool(alloc, block)) return -1;
  return alloc->refcount[block];
}

pa_status pa_allocator_stats_get(const pa_allocator *alloc, pa_allocator_stats *out) {
  if (!alloc || !out) return PA_ERR_NULL;
  out->total = (int32_t)alloc->refcount.size();
  out->free = (int32_t)alloc->free_list.size();
  out->used = alloc->used;
  out->shared = alloc->shared;
  out->n_allocated = alloc->n_allocated;
  out->n_cow = alloc->n_cow;
  return PA_OK;
}

pa_status pa_allocator_take_copies(pa_allocator *alloc, int32_t *pairs, int32_t capacity, int32_t *num) {
  if (!alloc || !num) return PA_ERR_NULL;
  const int32_t n = (int32_t)(alloc->copies.size() / 2);
  *num = n;
  if (n == 0) return PA_OK;
  if (capacity < n) return PA_ERR_SHAPE;
  if (!pairs) return PA_ERR_NULL;
  for (size_t i = 0; i < alloc->copies.size(); ++i) pairs[i] = alloc->copies[i];
  alloc->copies.clear();
  return PA_OK;
}

pa_status pa_sequence_create(pa_allocator *alloc, pa_sequence **out) {
  if (!alloc || !out) return PA_ERR_NULL;
  pa_sequence *s = new pa_sequence;
  s->alloc = alloc;
  *out = s;
  return PA_OK;
}

pa_status pa_sequence_release(pa_sequence *seq) {
  if (!seq) return PA_ERR_NULL;
  for (int32_t b : seq->blocks) ref_down(seq->alloc, b);
  seq->blocks.clear();
  seq->length = 0;
  seq->reserved = 0;
  return PA_OK;
}

void pa_sequence_destroy(pa_sequence *seq) {
  if (!seq) return;
  pa_sequence_release(seq);
  delete seq;
}

pa_status pa_sequence_reserve(pa_sequence *seq, int32_t n, int64_t *slots) {
  if (!seq) return PA_ERR_NULL;
  if (n < 0) return PA_ERR_SHAPE;
  if (n == 0) return PA_OK;
  pa_allocator *a = seq->alloc;
  const int64_t pos = (int64_t)seq->length + seq->reserved;  // first position to write
  if (pos + n > (int64_t)INT32_MAX) return PA_ERR_SHAPE;
  const int32_t have = (int32_t)seq->blocks.size();
  const int32_t need = blocks_for(pos + n);
  // the block holding position pos is written into; if it is shared with
  // another sequence (and partly filled, else pos would open a new block)
  // this sequence must first get a copy of its own
  const int32_t bi = (int32_t)(pos / kBlockTokens);
  const bool cow = bi < have && a->refcount[seq->blocks[bi]] > 1;
  const int32_t fresh = (need > have ? need - have : 0) + (cow ? 1 : 0);
  if ((size_t)fresh > a->free_list.size()) return PA_ERR_NO_BLOCKS;
  if (cow) {
    const int32_t src = seq->blocks[bi];
    const int32_t dst = take_free(a);
    a->copies.push_back(src);
    a->copies.push_back(dst);
    ref_down(a, src);
    seq->blocks[bi] = dst;
    ++a->n_cow;
  }
  for (int32_t i = have; i < need; ++i) seq->blocks.push_back(take_free(a));
  if (slots) {
    for (int32_t i = 0; i < n; ++i) {
      const int64_t p = pos + i;
      slots[i] = (int64_t)seq->blocks[(size_t)(p / kBlockTokens)] * kBlockTokens + p % kBlockTokens;
    }
  }
  seq->reserved += n;
  return PA_OK;
}

pa_status pa_sequence_commit(pa_sequence *seq, int32_t n) {
  if (!seq) return PA_ERR_NULL;
  if (n < 0) return PA_ERR_SHAPE;
  if (n > seq->reserved) return PA_ERR_STATE;
  seq->length += n;
  seq->reserved -= n;
  return PA_OK;
}

pa_status pa_sequence_adopt_prefix(pa_sequence *seq, const int32_t *blocks, int32_t n) {
  if (!seq) return PA_ERR_NULL;
  if (n < 0) return PA_ERR_SHAPE;
  if (!seq->blocks.empty() || seq->length != 0 || seq->reserved != 0) return PA_ERR_STATE;
  if (n == 0) return PA_OK;
  if (!blocks) return PA_ERR_NULL;
  if ((int64_t)n * kBlockTokens > (int64_t)INT32_MAX) return PA_ERR_SHAPE;
  for (int32_t i = 0; i < n; ++i) {  // every check before any change
    if (!in_pool(seq->alloc, blocks[i])) return PA_ERR_RANGE;
    if (seq->alloc->refcount[blocks[i]] == 0) return PA_ERR_STATE;
  }
  for (int32_t i = 0; i < n; ++i) {
    ref_up(seq->alloc, blocks[i]);
    seq->blocks.push_back(blocks[i]);
  }
  seq->length = n * kBlockTokens;
  return PA_OK;
}

pa_status pa_sequence_fork(pa_sequence *seq, const pa_sequence *other) {
  if (!seq || !other) return PA_ERR_NULL;
  if (seq == other || seq->alloc != other->alloc) return PA_ERR_STATE;
  if (!seq->blocks.empty() || seq->length != 0 || seq->reserved != 0) return PA_ERR_STATE;
  if (other->reserved != 0) return PA_ERR_STATE;
  for (int32_t b : other->blocks) {
    ref_up(seq->alloc, b);
    seq->blocks.push_back(b);
  }
  seq->length = other->length;
  return PA_OK;
}

int32_t pa_sequence_length(const pa_sequence *seq) { return seq ? seq->length : -1; }

int32_t pa_sequence_reserved(const pa_sequence *seq) { return seq ? seq->reserved : -1; }

int32_t pa_sequence_num_blocks(const pa_sequence *seq) { return seq ? (int32_t)seq->blocks.size() : -1; }

pa_status pa_sequence_blocks(const pa_sequence *seq, int32_t *out, int32_t capacity) {
  if (!seq) return PA_ERR_NULL;
  const int32_t n = (int32_t)seq->blocks.size();
  if (n == 0) return PA_OK;
  if (capacity < n) return PA_ERR_SHAPE;
  if (!out) return PA_ERR_NULL;
  for (int32_t i = 0; i < n; ++i) out[i] = seq->blocks[i];
  return PA_OK;
}

pa_status pa_build_step_tables(const pa_sequence *const *seqs, int32_t num_seqs, int32_t max_blocks,
                               int32_t *block_tables, int32_t *chunk_starts, int32_t *chunk_lens,
                               int32_t *context_lens) {
  if (num_seqs < 0 || max_blocks < 1) return PA_ERR_SHAPE;
  if (num_seqs == 0) return PA_OK;
  if (!seqs || !block_tables) return PA_ERR_NULL;
  for (int32_t i = 0; i < num_seqs; ++i) {
    if (!seqs[i]) return PA_ERR_NULL;
    if ((int32_t)seqs[i]->blocks.size() > max_blocks) return PA_ERR_SHAPE;
  }
  for (int32_t i = 0; i < num_seqs; ++i) {
    const pa_sequence *s = seqs[i];
    int32_t *row = block_tables + (int64_t)i * max_blocks;
    const int32_t n = (int32_t)s->blocks.size();
    for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < n ? s->blocks[j] : -1;
    if (chunk_starts) chunk_starts[i] = s->length;
    if (chunk_lens) chunk_lens[i] = s->reserved;
    if (context_lens) context_lens[i] = s->length + s->reserved;
  }
  return PA_OK;
}

}  // extern "C"
