// Choice of the split-K partition size for a decode batch (host only).
//
// Split-K ("PagedAttention" decode over long contexts, merged by
// log-sum-exp) trades parallelism against per-CTA cost: small partitions
// give many CTAs and a short tail, large ones fewer CTAs with less start-up
// and merge work.  Which wins depends on the batch, so the size is chosen per
// batch by a model of the launch: the CTAs of the grid (KV head fastest, then
// sequence, then partition) go, in that order, to the first free CTA slot of
// the GPU (slots = SMs x CTAs per SM of the kernel), and the launch takes as
// long as its busiest slot.  A CTA costs
//   kTokenUs * tokens  (its K/V at one slot's share of the bandwidth)
//   + kCtaUs           (start-up: tables, q, the first copies; the epilogue)
//   + kMergeUs         (a sequence with several partitions: publishing and
//                       merging the partial results)
// and a batch whose sequences need more than 16 partitions merges in a second
// launch (kApartUs).  The constants were fitted to pa_decode_step timings of
// the Llama-3.1-8B-shaped batch-64 and 32-layer batch-256 steps on a GB300
// (bf16 cache), once for each dispatch order: grid order at partition 384 ..
// 1536, longest first (pa_splitk_order) at 768 .. 2048 (refitted to 7 µs a
// CTA once 1280 and 1792 were candidates: batch 64 measured 47.3-47.6 µs at
// 1280, 47.9-48.3 at 1536, 51.0 at 1792, 53.2-53.4 at 1024 and 2048, and the
// model now picks 1280 there).  The 1-byte kernels are issue-bound:
// a CTA that runs with fewer neighbours on its SM does not get much faster,
// which the grid-order model (fixed CTA durations) gets right only once the
// batch has a CTA for every slot without splitting; with fewer (sequence, KV
// head) units than slots they take 512-token partitions in grid order, the
// measured best there.  Longest first, the model's choice matched the
// measured best for them too (batch 64: 1024; 32 layers: 2048).

#include <stdint.h>

#include <algorithm>
#include <functional>
#include <queue>
#include <vector>

#include "../../include/pa.h"

namespace {

// Costs (µs) fitted per dispatch order: grid order, and longest first.
struct Costs {
  double token_bf16;  // per token and KV head, head_dim 128, bf16 cache
  double token_1byte;
  double cta;
  double merge;
};
constexpr Costs kGridCosts = {0.025, 0.019, 4.0, 2.0};
constexpr Costs kOrderedCosts = {0.022, 0.0167, 7.0, 3.0};
constexpr double kApartUs = 3.0;
constexpr int kMergeInKernelParts = 16;  // as pa_decode_step
constexpr int kCandidates[] = {256, 384, 512, 640, 768, 1024, 1280, 1536, 1792, 2048, 4096};

// CTAs per SM of the split-K kernels (their __launch_bounds__ minimum).
int ctas_per_sm(int group, int kv_kind) {
  if (kv_kind == 0) return group <= 4 ? 3 : 1;
  return group <= 4 ? 4 : 3;
}

// Tokens of item (b, z) of a split into `part`-token partitions.
int item_tokens(int n, int z, int part) { return std::max(0, std::min(part, n - z * part)); }

double makespan(const int32_t* ctx, int num_seqs, int hkv, int part, int slots, double token_us,
                bool ordered) {
  const Costs& k = ordered ? kOrderedCosts : kGridCosts;
  int maxp = 1;
  for (int b = 0; b < num_seqs; ++b) maxp = std::max(maxp, (std::max(ctx[b], 0) + part - 1) / part);
  const bool apart = maxp > kMergeInKernelParts;
  // CTA durations in dispatch order: the grid's (partition slowest), or
  // longest first (the order pa_splitk_order gives)
  std::vector<double> items;
  for (int z = 0; z < maxp; ++z) {
    for (int b = 0; b < num_seqs; ++b) {
      const int n = std::max(ctx[b], 0);
      const int np = (n + part - 1) / part;
      if (z >= std::max(np, 1)) continue;
      items.push_back(token_us * item_tokens(n, z, part) + k.cta +
                      ((np > 1 && !apart) ? k.merge : 0.0));
    }
  }
  if (ordered) std::stable_sort(items.begin(), items.end(), std::greater<double>());
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int s = 0; s < slots; ++s) free_at.push(0.0);
  for (const double d : items) {
    for (int h = 0; h < hkv; ++h) {
      const double t = free_at.top();
      free_at.pop();
      free_at.push(t + d);
    }
  }
  double end = 0.0;
  while (!free_at.empty()) {
    end = std::max(end, free_at.top());
    free_at.pop();
  }
  return end + (apart ? kApartUs : 0.0);
}

}  // namespace

extern "C" int pa_splitk_partition_size(const int32_t* context_lens, int num_seqs,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int kv_kind, int num_sms, int ordered) {
  if (!context_lens || num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || head_dim <= 0 || kv_kind < 0 || kv_kind > 2 ||
      num_sms <= 0)
    return 0;
  const int group = num_q_heads / num_kv_heads;
  const int slots = num_sms * ctas_per_sm(group, kv_kind);
  const Costs& k = ordered ? kOrderedCosts : kGridCosts;
  const double token_us = (kv_kind == 0 ? k.token_bf16 : k.token_1byte) * head_dim / 128.0;
  int max_ctx = 0;
  for (int b = 0; b < num_seqs; ++b) max_ctx = std::max(max_ctx, context_lens[b]);
  if (!ordered && kv_kind != 0 && static_cast<int64_t>(num_seqs) * num_kv_heads < slots &&
      (static_cast<int64_t>(max_ctx) + 511) / 512 <= 65535)
    return 512;
  int best = 0;
  double best_t = 0.0;
  for (int part : kCandidates) {
    if ((static_cast<int64_t>(max_ctx) + part - 1) / part > 65535) continue;  // grid z
    const double t =
        makespan(context_lens, num_seqs, num_kv_heads, part, slots, token_us, ordered != 0);
    // ties go to the larger partition: fewer CTAs, less workspace
    if (best == 0 || t <= best_t + 1e-9) {
      best = part;
      best_t = t;
    }
    if (part >= max_ctx) break;  // larger sizes give the same single partitions
  }
  return best;
}

// Longest-first work order for a split-K launch: a permutation of the items
// [0, num_seqs * max_partitions) (item = part * num_seqs + b) sorted by the
// tokens each covers, most first, ties in item order; items past a sequence's
// end (0 tokens) come last.  The block scheduler hands CTAs out in this order,
// so the long ones start first and the short ones fill the tail.
extern "C" int pa_splitk_order(const int32_t* context_lens, int num_seqs, int partition_size,
                               int max_partitions, int32_t* order_out) {
  if (!context_lens || !order_out || num_seqs <= 0 || partition_size <= 0 ||
      max_partitions <= 0 || static_cast<int64_t>(num_seqs) * max_partitions > 65535)
    return -1;
  const int n_items = num_seqs * max_partitions;
  std::vector<std::pair<int, int>> key(n_items);  // (-tokens, item)
  for (int item = 0; item < n_items; ++item) {
    const int b = item % num_seqs, z = item / num_seqs;
    key[item] = {-item_tokens(std::max(context_lens[b], 0), z, partition_size), item};
  }
  std::sort(key.begin(), key.end());
  for (int i = 0; i < n_items; ++i) order_out[i] = key[i].second;
  return n_items;
}
