// Host block allocator for the paged KV cache.
//
// "How LLM Inference Serving Works" (dev.to): section "PagedAttention:
// Virtual Memory for the KV Cache" (fixed-size physical blocks, a per-request
// block table, blocks taken on demand), "Sharing comes for free" (reference
// counts, copy-on-write), "Putting It Together: The Life of a Request in
// vLLM" (a new block only when the current one fills; counts drop at the
// end), "When memory runs out anyway" (running out of blocks is reported so
// the caller can preempt).  Behaviour is specified in include/pa.h.
//
// Every entry point validates first and mutates only after it knows the call
// will succeed, so a failed call leaves the allocator unchanged.

#include <algorithm>
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pa.h"

namespace {

struct Sequence {
  std::vector<int32_t> table;  // logical block -> physical block
  int64_t len = 0;             // tokens held
};

}  // namespace

struct pa_alloc {
  int num_blocks = 0;
  int block_size = 0;
  std::deque<int32_t> free_fifo;  // head = next block handed out
  std::vector<int32_t> refs;      // per physical block
  std::unordered_map<int, Sequence> seqs;

  Sequence* find(int id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
  const Sequence* find(int id) const {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }

  // 1 if the next append to `s` takes a block from the free list: either the
  // token opens a new block, or it lands in a shared, partly filled block.
  int blocks_for_next_append(const Sequence& s) const {
    if (s.len % block_size == 0) return 1;
    return refs[s.table.back()] > 1 ? 1 : 0;
  }

  int32_t take() {
    int32_t b = free_fifo.front();
    free_fifo.pop_front();
    refs[b] = 1;
    return b;
  }

  // Appends one token; the caller has checked a free block exists if needed.
  int64_t append(Sequence& s, int32_t* cow_src, int32_t* cow_dst) {
    int32_t src = -1, dst = -1;
    const int64_t pos = s.len;
    if (pos % block_size == 0) {
      s.table.push_back(take());
    } else if (refs[s.table.back()] > 1) {
      src = s.table.back();
      dst = take();
      refs[src] -= 1;
      s.table.back() = dst;
    }
    s.len = pos + 1;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return static_cast<int64_t>(s.table[pos / block_size]) * block_size + pos % block_size;
  }
};

extern "C" {

pa_status pa_alloc_create(int num_blocks, int block_size, const int32_t* initial_free_order,
                          pa_alloc** out) {
  if (!out) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  std::vector<int32_t> order(num_blocks);
  if (initial_free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
      const int32_t b = initial_free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) return PA_ERR_INVALID_ARG;
      seen[b] = 1;
      order[i] = b;
    }
  } else {
    for (int i = 0; i < num_blocks; ++i) order[i] = i;
  }
  pa_alloc* a = new (std::nothrow) pa_alloc();
  if (!a) return PA_ERR_INVALID_ARG;
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->free_fifo.assign(order.begin(), order.end());
  a->refs.assign(num_blocks, 0);
  *out = a;
  return PA_OK;
}

void pa_alloc_destroy(pa_alloc* a) { delete a; }

pa_status pa_alloc_add_seq(pa_alloc* a, int seq_id) {
  if (!a || a->find(seq_id)) return PA_ERR_INVALID_ARG;
  a->seqs.emplace(seq_id, Sequence{});
  return PA_OK;
}

pa_status pa_alloc_append_slot(pa_alloc* a, int seq_id, int64_t* slot_out, int32_t* cow_src,
                               int32_t* cow_dst) {
  if (!a || !slot_out) return PA_ERR_INVALID_ARG;
  Sequence* s = a->find(seq_id);
  if (!s) return PA_ERR_INVALID_ARG;
  if (a->blocks_for_next_append(*s) > static_cast<int>(a->free_fifo.size()))
    return PA_ERR_OUT_OF_BLOCKS;
  *slot_out = a->append(*s, cow_src, cow_dst);
  return PA_OK;
}

pa_status pa_alloc_append_slots(pa_alloc* a, const int* seq_ids, int n, int64_t* slots_out,
                                int32_t* cow_src, int32_t* cow_dst) {
  if (!a || n < 0 || (n > 0 && (!seq_ids || !slots_out))) return PA_ERR_INVALID_ARG;
  std::unordered_set<int> distinct;
  std::vector<Sequence*> ptrs(n);
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    if (!distinct.insert(seq_ids[i]).second) return PA_ERR_INVALID_ARG;
    ptrs[i] = a->find(seq_ids[i]);
    if (!ptrs[i]) return PA_ERR_INVALID_ARG;
    need += a->blocks_for_next_append(*ptrs[i]);
  }
  if (need > static_cast<int64_t>(a->free_fifo.size())) return PA_ERR_OUT_OF_BLOCKS;
  for (int i = 0; i < n; ++i)
    slots_out[i] = a->append(*ptrs[i], cow_src ? cow_src + i : nullptr,
                             cow_dst ? cow_dst + i : nullptr);
  return PA_OK;
}

pa_status pa_alloc_reserve(pa_alloc* a, int seq_id, int num_tokens, int32_t* cow_src,
                           int32_t* cow_dst) {
  if (!a || num_tokens < 0) return PA_ERR_INVALID_ARG;
  Sequence* s = a->find(seq_id);
  if (!s) return PA_ERR_INVALID_ARG;
  if (cow_src) *cow_src = -1;
  if (cow_dst) *cow_dst = -1;
  if (num_tokens == 0) return PA_OK;
  const int64_t bs = a->block_size;
  const int64_t have = (s->len + bs - 1) / bs;
  const int64_t want = (s->len + num_tokens + bs - 1) / bs;
  const int64_t cow = (s->len % bs != 0 && a->refs[s->table.back()] > 1) ? 1 : 0;
  if (want - have + cow > static_cast<int64_t>(a->free_fifo.size())) return PA_ERR_OUT_OF_BLOCKS;
  a->append(*s, cow_src, cow_dst);
  for (int i = 1; i < num_tokens; ++i) a->append(*s, nullptr, nullptr);
  return PA_OK;
}

pa_status pa_alloc_fork(pa_alloc* a, int parent_id, int child_id) {
  if (!a) return PA_ERR_INVALID_ARG;
  const Sequence* p = a->find(parent_id);
  if (!p || a->find(child_id)) return PA_ERR_INVALID_ARG;
  Sequence c = *p;
  for (int32_t b : c.table) a->refs[b] += 1;
  a->seqs.emplace(child_id, std::move(c));
  return PA_OK;
}

pa_status pa_alloc_free_seq(pa_alloc* a, int seq_id) {
  if (!a) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PA_ERR_INVALID_ARG;
  for (int32_t b : it->second.table) {
    if (--a->refs[b] == 0) a->free_fifo.push_back(b);
  }
  a->seqs.erase(it);
  return PA_OK;
}

pa_status pa_alloc_block_table(const pa_alloc* a, int seq_id, int32_t* out, int cap, int* n_out) {
  if (!a || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
  const Sequence* s = a->find(seq_id);
  if (!s) return PA_ERR_INVALID_ARG;
  const int n = static_cast<int>(s->table.size());
  std::copy(s->table.begin(), s->table.begin() + std::min(n, cap), out);
  *n_out = n;
  return PA_OK;
}

pa_status pa_alloc_block_tables(const pa_alloc* a, const int* seq_ids, int n, int32_t* out,
                                int max_blocks, int32_t* ctx_out) {
  if (!a || n < 0 || max_blocks < 0) return PA_ERR_INVALID_ARG;
  if (n > 0 && (!seq_ids || (max_blocks > 0 && !out))) return PA_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const Sequence* s = a->find(seq_ids[i]);
    if (!s || static_cast<int64_t>(s->table.size()) > max_blocks) return PA_ERR_INVALID_ARG;
    if (ctx_out && s->len > INT32_MAX) return PA_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; ++i) {
    const Sequence* s = a->find(seq_ids[i]);
    int32_t* row = out + static_cast<int64_t>(i) * max_blocks;
    std::fill(row, row + max_blocks, -1);
    std::copy(s->table.begin(), s->table.end(), row);
    if (ctx_out) ctx_out[i] = static_cast<int32_t>(s->len);
  }
  return PA_OK;
}

int64_t pa_alloc_seq_len(const pa_alloc* a, int seq_id) {
  if (!a) return -1;
  const Sequence* s = a->find(seq_id);
  return s ? s->len : -1;
}

int pa_alloc_refcount(const pa_alloc* a, int block) {
  if (!a || block < 0 || block >= a->num_blocks) return -1;
  return a->refs[block];
}

int pa_alloc_num_free(const pa_alloc* a) { return a ? static_cast<int>(a->free_fifo.size()) : -1; }

int pa_alloc_num_blocks(const pa_alloc* a) { return a ? a->num_blocks : -1; }

pa_status pa_alloc_free_list(const pa_alloc* a, int32_t* out, int cap, int* n_out) {
  if (!a || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
  const int n = static_cast<int>(a->free_fifo.size());
  std::copy(a->free_fifo.begin(), a->free_fifo.begin() + std::min(n, cap), out);
  *n_out = n;
  return PA_OK;
}

int pa_alloc_tail_waste(const pa_alloc* a, int seq_id) {
  if (!a) return -1;
  const Sequence* s = a->find(seq_id);
  if (!s) return -1;
  return static_cast<int>(static_cast<int64_t>(s->table.size()) * a->block_size - s->len);
}

}  // extern "C"
