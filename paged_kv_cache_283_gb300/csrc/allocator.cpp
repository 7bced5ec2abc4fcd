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
//
// Automatic prefix caching (optional, section "Prefix Caching and Chunked
// Prefill"): every full block of a prompt is named by a chained hash of its
// tokens and of all tokens before it (with an optional per-request salt mixed
// into the first block); a table maps names to physical blocks, so a new
// prompt reuses the blocks of the longest cached prefix.  A named block whose
// reference count drops to zero is not freed but kept, cached-but-evictable,
// in least-recently-used order, and is evicted (its name dropped) only when
// a block is needed and the free list is empty.

#include <algorithm>
#include <array>
#include <cstdint>
#include <cstring>
#include <deque>
#include <list>
#include <new>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pa.h"
#include "sha256.h"

namespace {

using Digest = std::array<uint8_t, 32>;

struct DigestHash {
  size_t operator()(const Digest& d) const {
    size_t v;
    std::memcpy(&v, d.data(), sizeof(v));
    return v;
  }
};

// Name of the first block's parent: 32 zero bytes, or SHA-256 of the salt.
Digest root_digest(const void* salt, int salt_len) {
  Digest d{};
  if (salt && salt_len > 0) {
    pa::Sha256 h;
    h.update(salt, static_cast<size_t>(salt_len));
    h.final(d.data());
  }
  return d;
}

// SHA-256(parent || tokens as little-endian int32).
Digest block_digest(const Digest& parent, const int32_t* tokens, int n) {
  pa::Sha256 h;
  h.update(parent.data(), parent.size());
  for (int i = 0; i < n; ++i) {
    const uint32_t t = static_cast<uint32_t>(tokens[i]);
    const uint8_t b[4] = {static_cast<uint8_t>(t), static_cast<uint8_t>(t >> 8),
                          static_cast<uint8_t>(t >> 16), static_cast<uint8_t>(t >> 24)};
    h.update(b, 4);
  }
  Digest d;
  h.final(d.data());
  return d;
}

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
  // prefix cache (empty unless enabled)
  bool prefix_cache = false;
  std::unordered_map<Digest, int32_t, DigestHash> by_digest;
  std::vector<Digest> digest_of;  // per block, valid where named[b]
  std::vector<char> named;
  std::list<int32_t> evictable;  // unreferenced named blocks, least recent first
  std::vector<std::list<int32_t>::iterator> lru_pos;

  int64_t available() const {
    return static_cast<int64_t>(free_fifo.size()) + static_cast<int64_t>(evictable.size());
  }

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

  // A fresh block: the free list first, else the least recently used cached
  // block, whose name is dropped.  The caller has checked available() > 0.
  int32_t take() {
    int32_t b;
    if (!free_fifo.empty()) {
      b = free_fifo.front();
      free_fifo.pop_front();
    } else {
      b = evictable.front();
      evictable.pop_front();
      by_digest.erase(digest_of[b]);
      named[b] = 0;
    }
    refs[b] = 1;
    return b;
  }

  // One reference fewer; an unreferenced block is freed, or kept cached if named.
  void release(int32_t b) {
    if (--refs[b] != 0) return;
    if (prefix_cache && named[b]) {
      evictable.push_back(b);
      lru_pos[b] = std::prev(evictable.end());
    } else {
      free_fifo.push_back(b);
    }
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
  if (a->blocks_for_next_append(*s) > a->available()) return PA_ERR_OUT_OF_BLOCKS;
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
  if (need > a->available()) return PA_ERR_OUT_OF_BLOCKS;
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
  if (want - have + cow > a->available()) return PA_ERR_OUT_OF_BLOCKS;
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
  for (int32_t b : it->second.table) a->release(b);
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

extern "C" {

pa_status pa_alloc_enable_prefix_cache(pa_alloc* a) {
  if (!a || !a->seqs.empty()) return PA_ERR_INVALID_ARG;
  if (a->prefix_cache) return PA_OK;
  a->prefix_cache = true;
  a->digest_of.assign(a->num_blocks, Digest{});
  a->named.assign(a->num_blocks, 0);
  a->lru_pos.assign(a->num_blocks, a->evictable.end());
  return PA_OK;
}

pa_status pa_alloc_add_seq_prompt(pa_alloc* a, int seq_id, const int32_t* tokens, int num_tokens,
                                  const void* salt, int salt_len, int* cached_tokens) {
  if (!a || !a->prefix_cache || num_tokens < 0 || salt_len < 0 || (num_tokens > 0 && !tokens) ||
      (salt_len > 0 && !salt) || a->find(seq_id))
    return PA_ERR_INVALID_ARG;
  const int bs = a->block_size;
  const int full = num_tokens / bs;
  std::vector<Digest> names(full);
  Digest parent = root_digest(salt, salt_len);
  for (int i = 0; i < full; ++i) {
    names[i] = block_digest(parent, tokens + static_cast<int64_t>(i) * bs, bs);
    parent = names[i];
  }
  // longest cached prefix
  int hits = 0, hits_unreferenced = 0;
  for (; hits < full; ++hits) {
    auto it = a->by_digest.find(names[hits]);
    if (it == a->by_digest.end()) break;
    if (a->refs[it->second] == 0) ++hits_unreferenced;
  }
  const int64_t need = (static_cast<int64_t>(num_tokens) + bs - 1) / bs - hits;
  if (need > a->available() - hits_unreferenced) return PA_ERR_OUT_OF_BLOCKS;
  Sequence s;
  for (int i = 0; i < hits; ++i) {
    const int32_t b = a->by_digest[names[i]];
    if (a->refs[b] == 0) {
      a->evictable.erase(a->lru_pos[b]);
      a->lru_pos[b] = a->evictable.end();
    }
    a->refs[b] += 1;
    s.table.push_back(b);
  }
  s.len = static_cast<int64_t>(hits) * bs;
  for (int64_t t = s.len; t < num_tokens; ++t) a->append(s, nullptr, nullptr);
  // name the prompt's new full blocks (a name already in use keeps its block)
  for (int i = hits; i < full; ++i) {
    const int32_t b = s.table[i];
    if (a->by_digest.count(names[i])) continue;
    a->by_digest.emplace(names[i], b);
    a->digest_of[b] = names[i];
    a->named[b] = 1;
  }
  a->seqs.emplace(seq_id, std::move(s));
  if (cached_tokens) *cached_tokens = hits * bs;
  return PA_OK;
}

int pa_alloc_num_evictable(const pa_alloc* a) {
  return a ? static_cast<int>(a->evictable.size()) : -1;
}

pa_status pa_alloc_evictable_list(const pa_alloc* a, int32_t* out, int cap, int* n_out) {
  if (!a || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
  int i = 0;
  for (int32_t b : a->evictable) {
    if (i < cap) out[i] = b;
    ++i;
  }
  *n_out = i;
  return PA_OK;
}

pa_status pa_prefix_root_hash(const void* salt, int salt_len, uint8_t* out) {
  if (!out || salt_len < 0 || (salt_len > 0 && !salt)) return PA_ERR_INVALID_ARG;
  const Digest d = root_digest(salt, salt_len);
  std::memcpy(out, d.data(), 32);
  return PA_OK;
}

pa_status pa_prefix_block_hash(const uint8_t* parent, const int32_t* tokens, int num_tokens,
                               uint8_t* out) {
  if (!parent || !out || num_tokens < 0 || (num_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
  Digest p;
  std::memcpy(p.data(), parent, 32);
  const Digest d = block_digest(p, tokens, num_tokens);
  std::memcpy(out, d.data(), 32);
  return PA_OK;
}

}  // extern "C"
