// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Arguments of the decode kernels (plain and split-K).  Pointers are device
// pointers, already validated on the host.
struct DecodeParams {
  __nv_bfloat16* out;  // pa_decode: [B, Hq, D]
  float* ws_o;         // split-K: [B, Hq, max_partitions, D]
  float* ws_m;         // split-K: [B, Hq, max_partitions]
  float* ws_l;         // split-K: [B, Hq, max_partitions]
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int8_t* k8;        // int8 cache: codes [NB, Hkv, bs, D] (null for a bf16 cache)
  const int8_t* v8;
  const float* k_scales;   // int8 / fp8 cache: one scale per (block, head, token)
  const float* v_scales;
  int fp8;                 // 1-byte cache: codes are FP8 (E4M3), not INT8
  const int32_t* block_tables;
  const int32_t* context_lens;
  unsigned* err;
  int max_blocks_per_seq;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int max_partitions;    // split-K only
  int partition_blocks;  // split-K only: blocks per partition
  float scale_log2;      // scale * log2(e): scores are kept in base-2 units
  // Fused decode step (pa_decode_step*), null when off.  The pools above are
  // then written as well (the CTA reading each new token's position writes
  // that token's K and V rows first).
  const __nv_bfloat16* new_key;    // [B, Hkv, D]: each sequence's new token
  const __nv_bfloat16* new_value;
  const int64_t* slot_mapping;     // [B]: the slot of position context_lens[b] - 1, or < 0
  unsigned* counters;              // split-K: [B, Hkv] arrivals; the last CTA merges
  // split-K, optional: the order in which the (sequence, partition) items run,
  // a permutation of [0, B * max_partitions) (item = part * B + b); null: grid order
  const int32_t* order;
  // Tables, lengths, order and pools are not written by the preceding kernel:
  // they may be read before waiting for it (programmatic dependent launch).
  int early_read;
  // split-K: partitions below first_partition are not computed here (a
  // shared prefix's prefix_blocks blocks, computed by launch_prefix_partials,
  // which also checks that every sequence holds them); the others hold
  // partition_blocks blocks each from block prefix_blocks on.
  int first_partition;
  int prefix_blocks;
};

struct ReduceParams {
  __nv_bfloat16* out;
  const float* ws_o;
  const float* ws_m;
  const float* ws_l;
  const int32_t* context_lens;
  unsigned* err;
  int num_seqs;
  int num_q_heads;
  int max_partitions;
  int partition_size;
};

struct CacheWriteParams {
  const __nv_bfloat16* key;
  const __nv_bfloat16* value;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  const int64_t* slot_mapping;
  unsigned* err;
  int num_tokens;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int64_t num_slots;  // num_blocks * block_size
  int8_t* k8;         // int8 / fp8 cache (null for bf16): codes [NB, Hkv, bs, D]
  int8_t* v8;
  float* k_scales;    // [NB, Hkv, bs]
  float* v_scales;
  int fp8;            // codes are FP8 (E4M3), not INT8
};

// Pools of up to kCopyMaxLayers layers go to one copy_blocks launch.
constexpr int kCopyMaxLayers = 64;

struct CopyBlocksParams {
  void* k_caches[kCopyMaxLayers];
  void* v_caches[kCopyMaxLayers];
  const int64_t* block_mapping;  // [num_pairs, 2]: (src, dst)
  unsigned* err;
  int64_t block_bytes;  // Hkv * bs * D * 2
  int64_t num_blocks;
};

// Shapes with a compiled decode kernel.
bool decode_shape_supported(int head_dim, int group, int block_size);

cudaError_t launch_decode(const DecodeParams& p, int head_dim, int group, bool split,
                          cudaStream_t stream);
cudaError_t launch_splitk_reduce(const ReduceParams& p, int head_dim, cudaStream_t stream);
// prefill.cu: the split-K partials of a decode batch's queries over a shared
// prefix, partitions [0, splits) of split_blocks blocks each (head_dim 128);
// sets PA_DEVERR_PREFIX for a sequence not holding the prefix's blocks or not
// going past them.
cudaError_t launch_prefix_partials(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int num_blocks, float scale,
                                   int split_blocks, int splits, float* ws_o, float* ws_m,
                                   float* ws_l, int max_partitions, unsigned* err,
                                   cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const CacheWriteParams& p, cudaStream_t stream);
cudaError_t launch_reshape_and_cache_int8(const CacheWriteParams& p, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyBlocksParams& p, int num_pairs, int num_layers,
                               cudaStream_t stream);

// Address of the current device's error word (device memory), or nullptr.
unsigned* device_error_word();

// Records e as the calling thread's last CUDA error (pa_last_cuda_error) and
// returns PA_ERR_CUDA.
pa_status cuda_fail(cudaError_t e);

}  // namespace pa
