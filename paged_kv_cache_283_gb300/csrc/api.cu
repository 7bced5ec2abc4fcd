// C ABI of libpa.so: argument checks, the per-device error word, and the
// hand-off to the kernel launchers.  Semantics are specified in include/pa.h.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>

#include "../../include/pa.h"
#include "internal.h"

namespace pa {

namespace {

// Error word written by the kernels (PA_DEVERR_* bits); one per device.
__device__ unsigned g_error_word;

thread_local std::string t_last_cuda_error;

constexpr int kMaxDevices = 64;
std::atomic<unsigned*> g_error_word_ptr[kMaxDevices];

}  // namespace

pa_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = cudaGetErrorString(e);
  return PA_ERR_CUDA;
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool ok_ptr(const void* p, uintptr_t align) { return p != nullptr && aligned(p, align); }

}  // namespace

unsigned* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned* ptr = g_error_word_ptr[dev].load(std::memory_order_acquire);
  if (ptr) return ptr;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess) return nullptr;
  ptr = static_cast<unsigned*>(addr);
  g_error_word_ptr[dev].store(ptr, std::memory_order_release);
  return ptr;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK:
      return "ok";
    case PA_ERR_INVALID_ARG:
      return "invalid argument";
    case PA_ERR_UNSUPPORTED_SHAPE:
      return "unsupported shape (no compiled kernel for this head_dim / group / block_size)";
    case PA_ERR_OUT_OF_BLOCKS:
      return "out of KV blocks";
    case PA_ERR_CUDA:
      return "CUDA error";
  }
  return "unknown status";
}

const char* pa_last_cuda_error(void) { return t_last_cuda_error.c_str(); }

pa_status pa_get_device_error(unsigned* bits) {
  if (!bits) return PA_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpyFromSymbol(bits, g_error_word, sizeof(unsigned));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_clear_device_error(void) {
  const unsigned zero = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_decode_supported(int num_q_heads, int num_kv_heads, int head_dim, int block_size) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  return decode_shape_supported(head_dim, num_q_heads / num_kv_heads, block_size)
             ? PA_OK
             : PA_ERR_UNSUPPORTED_SHAPE;
}

pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, pa_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 != 0 ||
      block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!ok_ptr(key, 16) || !ok_ptr(value, 16) || !ok_ptr(k_cache, 16) || !ok_ptr(v_cache, 16) ||
      !ok_ptr(slot_mapping, 8))
    return PA_ERR_INVALID_ARG;
  CacheWriteParams p;
  p.key = static_cast<const __nv_bfloat16*>(key);
  p.value = static_cast<const __nv_bfloat16*>(value);
  p.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  p.slot_mapping = slot_mapping;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  p.num_tokens = num_tokens;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_slots = static_cast<int64_t>(num_blocks) * block_size;
  cudaError_t e = launch_reshape_and_cache(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                         const int64_t* block_mapping, int num_pairs, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_stream_t stream) {
  if (num_layers < 0 || num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 8 != 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_layers == 0 || num_pairs == 0) return PA_OK;
  if (num_pairs > 0x7fffffff / 2 || !k_caches || !v_caches || !ok_ptr(block_mapping, 8))
    return PA_ERR_INVALID_ARG;
  for (int l = 0; l < num_layers; ++l)
    if (!ok_ptr(k_caches[l], 16) || !ok_ptr(v_caches[l], 16)) return PA_ERR_INVALID_ARG;
  CopyBlocksParams p{};
  p.block_mapping = block_mapping;
  p.block_bytes = static_cast<int64_t>(num_kv_heads) * block_size * head_dim * 2;
  p.num_blocks = num_blocks;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  for (int l0 = 0; l0 < num_layers; l0 += kCopyMaxLayers) {
    const int n = num_layers - l0 < kCopyMaxLayers ? num_layers - l0 : kCopyMaxLayers;
    for (int l = 0; l < n; ++l) {
      p.k_caches[l] = k_caches[l0 + l];
      p.v_caches[l] = v_caches[l0 + l];
    }
    cudaError_t e = launch_copy_blocks(p, num_pairs, n, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PA_OK;
}

}  // extern "C"

namespace {

pa_status cache_write_1byte(const void* key, const void* value, void* k_cache, void* v_cache,
                            float* k_scales, float* v_scales, const int64_t* slot_mapping,
                            int num_tokens, int num_kv_heads, int head_dim, int block_size,
                            int num_blocks, int fp8, pa_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!ok_ptr(key, 16) || !ok_ptr(value, 16) || !ok_ptr(k_cache, 16) || !ok_ptr(v_cache, 16) ||
      !ok_ptr(k_scales, 16) || !ok_ptr(v_scales, 16) || !ok_ptr(slot_mapping, 8))
    return PA_ERR_INVALID_ARG;
  CacheWriteParams p{};
  p.key = static_cast<const __nv_bfloat16*>(key);
  p.value = static_cast<const __nv_bfloat16*>(value);
  p.k8 = static_cast<int8_t*>(k_cache);
  p.v8 = static_cast<int8_t*>(v_cache);
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.fp8 = fp8;
  p.slot_mapping = slot_mapping;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  p.num_tokens = num_tokens;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_slots = static_cast<int64_t>(num_blocks) * block_size;
  cudaError_t e = launch_reshape_and_cache_int8(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

pa_status pa_reshape_and_cache_int8(const void* key, const void* value, int8_t* k_cache,
                                    int8_t* v_cache, float* k_scales, float* v_scales,
                                    const int64_t* slot_mapping, int num_tokens,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, pa_stream_t stream) {
  return cache_write_1byte(key, value, k_cache, v_cache, k_scales, v_scales, slot_mapping,
                           num_tokens, num_kv_heads, head_dim, block_size, num_blocks, 0, stream);
}

pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, uint8_t* k_cache,
                                   uint8_t* v_cache, float* k_scales, float* v_scales,
                                   const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                   int head_dim, int block_size, int num_blocks,
                                   pa_stream_t stream) {
  return cache_write_1byte(key, value, k_cache, v_cache, k_scales, v_scales, slot_mapping,
                           num_tokens, num_kv_heads, head_dim, block_size, num_blocks, 1, stream);
}


namespace {

// Checks shared by pa_decode and pa_decode_splitk.
pa_status check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            float scale) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || !(scale == scale))
    return PA_ERR_INVALID_ARG;
  pa_status s = pa_decode_supported(num_q_heads, num_kv_heads, head_dim, block_size);
  if (s != PA_OK) return s;
  if (num_seqs > 65535) return PA_ERR_UNSUPPORTED_SHAPE;  // grid y
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7fffffff)
    return PA_ERR_UNSUPPORTED_SHAPE;
  if (num_seqs == 0) return PA_OK;
  if (!ok_ptr(q, 16) || !ok_ptr(k_cache, 16) || !ok_ptr(v_cache, 16) || !ok_ptr(block_tables, 4) ||
      !ok_ptr(context_lens, 4))
    return PA_ERR_INVALID_ARG;
  return PA_OK;
}

DecodeParams make_decode_params(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int num_seqs, int num_q_heads,
                                int num_kv_heads, int num_blocks, float scale) {
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  return p;
}

}  // namespace

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                    int head_dim, int block_size, int num_blocks, float scale,
                    pa_stream_t stream) {
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale);
  if (s != PA_OK || num_seqs == 0) return s;
  if (!ok_ptr(out, 16)) return PA_ERR_INVALID_ARG;
  DecodeParams p = make_decode_params(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                      context_lens, num_seqs, num_q_heads, num_kv_heads,
                                      num_blocks, scale);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.max_partitions = 1;
  p.partition_blocks = max_blocks_per_seq;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, false,
                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t pa_splitk_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_context_len,
                                 int partition_size) {
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
      partition_size <= 0)
    return 0;
  const size_t parts = (static_cast<size_t>(max_context_len) + partition_size - 1) / partition_size;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * (parts ? parts : 1);
  return rows * head_dim * sizeof(float) + 2 * rows * sizeof(float);
}

pa_status pa_decode_splitk(float* ws_out, float* ws_m, float* ws_l, int max_partitions,
                           const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           float scale, int partition_size, pa_stream_t stream) {
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale);
  if (s != PA_OK) return s;
  if (max_partitions <= 0 || max_partitions > 65535 || partition_size <= 0 ||
      partition_size % block_size != 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!ok_ptr(ws_out, 16) || !ok_ptr(ws_m, 4) || !ok_ptr(ws_l, 4)) return PA_ERR_INVALID_ARG;
  DecodeParams p = make_decode_params(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                      context_lens, num_seqs, num_q_heads, num_kv_heads,
                                      num_blocks, scale);
  p.ws_o = ws_out;
  p.ws_m = ws_m;
  p.ws_l = ws_l;
  p.max_partitions = max_partitions;
  p.partition_blocks = partition_size / block_size;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, true,
                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_splitk_reduce(void* out, const float* ws_out, const float* ws_m, const float* ws_l,
                           int max_partitions, const int32_t* context_lens, int num_seqs,
                           int num_q_heads, int head_dim, int partition_size,
                           pa_stream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || max_partitions <= 0 || partition_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED_SHAPE;
  if (num_seqs > 65535) return PA_ERR_UNSUPPORTED_SHAPE;  // grid y
  if (num_seqs == 0) return PA_OK;
  if (!ok_ptr(out, 16) || !ok_ptr(ws_out, 16) || !ok_ptr(ws_m, 4) || !ok_ptr(ws_l, 4) ||
      !ok_ptr(context_lens, 4))
    return PA_ERR_INVALID_ARG;
  ReduceParams p{};
  p.out = static_cast<__nv_bfloat16*>(out);
  p.ws_o = ws_out;
  p.ws_m = ws_m;
  p.ws_l = ws_l;
  p.context_lens = context_lens;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.max_partitions = max_partitions;
  p.partition_size = partition_size;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  cudaError_t e = launch_splitk_reduce(p, head_dim, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

pa_status decode_1byte(void* out, const void* q, const void* k_cache, const void* v_cache,
                       const float* k_scales, const float* v_scales, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, float scale, int fp8, pa_stream_t stream) {
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale);
  if (s != PA_OK || num_seqs == 0) return s;
  if (!ok_ptr(out, 16) || !ok_ptr(k_scales, 16) || !ok_ptr(v_scales, 16))
    return PA_ERR_INVALID_ARG;
  DecodeParams p = make_decode_params(q, nullptr, nullptr, block_tables, max_blocks_per_seq,
                                      context_lens, num_seqs, num_q_heads, num_kv_heads,
                                      num_blocks, scale);
  p.k8 = static_cast<const int8_t*>(k_cache);
  p.v8 = static_cast<const int8_t*>(v_cache);
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.fp8 = fp8;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.max_partitions = 1;
  p.partition_blocks = max_blocks_per_seq;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, false,
                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status decode_splitk_1byte(float* ws_out, float* ws_m, float* ws_l, int max_partitions,
                              const void* q, const void* k_cache, const void* v_cache,
                              const float* k_scales, const float* v_scales,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, int num_seqs, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks,
                              float scale, int partition_size, int fp8, pa_stream_t stream) {
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale);
  if (s != PA_OK) return s;
  if (max_partitions <= 0 || max_partitions > 65535 || partition_size <= 0 ||
      partition_size % block_size != 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!ok_ptr(ws_out, 16) || !ok_ptr(ws_m, 4) || !ok_ptr(ws_l, 4) || !ok_ptr(k_scales, 16) ||
      !ok_ptr(v_scales, 16))
    return PA_ERR_INVALID_ARG;
  DecodeParams p = make_decode_params(q, nullptr, nullptr, block_tables, max_blocks_per_seq,
                                      context_lens, num_seqs, num_q_heads, num_kv_heads,
                                      num_blocks, scale);
  p.k8 = static_cast<const int8_t*>(k_cache);
  p.v8 = static_cast<const int8_t*>(v_cache);
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.fp8 = fp8;
  p.ws_o = ws_out;
  p.ws_m = ws_m;
  p.ws_l = ws_l;
  p.max_partitions = max_partitions;
  p.partition_blocks = partition_size / block_size;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, true,
                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

pa_status pa_decode_int8(void* out, const void* q, const int8_t* k_cache, const int8_t* v_cache,
                         const float* k_scales, const float* v_scales,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         float scale, pa_stream_t stream) {
  return decode_1byte(out, q, k_cache, v_cache, k_scales, v_scales, block_tables,
                      max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, scale, 0, stream);
}

pa_status pa_decode_splitk_int8(float* ws_out, float* ws_m, float* ws_l, int max_partitions,
                                const void* q, const int8_t* k_cache, const int8_t* v_cache,
                                const float* k_scales, const float* v_scales,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int num_seqs, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                float scale, int partition_size, pa_stream_t stream) {
  return decode_splitk_1byte(ws_out, ws_m, ws_l, max_partitions, q, k_cache, v_cache, k_scales,
                             v_scales, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                             partition_size, 0, stream);
}

pa_status pa_decode_fp8(void* out, const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                        const float* k_scales, const float* v_scales, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        int num_blocks, float scale, pa_stream_t stream) {
  return decode_1byte(out, q, k_cache, v_cache, k_scales, v_scales, block_tables,
                      max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, scale, 1, stream);
}

pa_status pa_decode_splitk_fp8(float* ws_out, float* ws_m, float* ws_l, int max_partitions,
                               const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                               const float* k_scales, const float* v_scales,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               float scale, int partition_size, pa_stream_t stream) {
  return decode_splitk_1byte(ws_out, ws_m, ws_l, max_partitions, q, k_cache, v_cache, k_scales,
                             v_scales, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                             partition_size, 1, stream);
}

}  // extern "C"

namespace {

// pa_decode_step*: the cache write of each sequence's new token and its
// attention in one launch (kv: 0 bf16, 1 INT8, 2 FP8).
pa_status decode_step_impl(void* out, const void* q, const void* key, const void* value,
                           const int64_t* slot_mapping, void* k_cache, void* v_cache,
                           float* k_scales, float* v_scales, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, float scale, int partition_size, float* ws_out,
                           float* ws_m, float* ws_l, unsigned* counters, int max_partitions,
                           const int32_t* order, int flags, int kv, pa_stream_t stream) {
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale);
  if (s != PA_OK) return s;
  const bool write = key != nullptr || value != nullptr || slot_mapping != nullptr;
  const bool split = partition_size != 0;
  if (partition_size < 0 || (split && (partition_size % block_size != 0 || max_partitions <= 0 ||
                                       max_partitions > 65535)))
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!ok_ptr(out, 16)) return PA_ERR_INVALID_ARG;
  if (write && (!ok_ptr(key, 16) || !ok_ptr(value, 16) || !ok_ptr(slot_mapping, 8)))
    return PA_ERR_INVALID_ARG;
  if (split && (!ok_ptr(ws_out, 16) || !ok_ptr(ws_m, 4) || !ok_ptr(ws_l, 4) ||
                !ok_ptr(counters, 4)))
    return PA_ERR_INVALID_ARG;
  if (kv != 0 && (!ok_ptr(k_scales, 16) || !ok_ptr(v_scales, 16))) return PA_ERR_INVALID_ARG;
  if ((flags & ~PA_STEP_EARLY_READ) != 0) return PA_ERR_INVALID_ARG;
  if (order != nullptr) {
    if (!split || !ok_ptr(order, 4)) return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_seqs) * max_partitions > 65535)
      return PA_ERR_UNSUPPORTED_SHAPE;  // the ordered grid's y extent
  }
  DecodeParams p = make_decode_params(q, kv ? nullptr : k_cache, kv ? nullptr : v_cache,
                                      block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                      num_q_heads, num_kv_heads, num_blocks, scale);
  if (kv != 0) {
    p.k8 = static_cast<const int8_t*>(k_cache);
    p.v8 = static_cast<const int8_t*>(v_cache);
    p.k_scales = k_scales;
    p.v_scales = v_scales;
    p.fp8 = kv == 2;
  }
  p.out = static_cast<__nv_bfloat16*>(out);
  p.early_read = (flags & PA_STEP_EARLY_READ) != 0;
  if (write) {
    p.new_key = static_cast<const __nv_bfloat16*>(key);
    p.new_value = static_cast<const __nv_bfloat16*>(value);
    p.slot_mapping = slot_mapping;
  }
  // Up to kMergeInKernelParts partitions per sequence are merged by the last
  // CTA of each (sequence, KV head); beyond that one CTA's merge would sit on
  // the critical path of the launch's tail, and the merge runs as its own
  // launch (pa_splitk_reduce's kernel) over all SMs instead.
  constexpr int kMergeInKernelParts = 16;
  const bool merge_apart = split && max_partitions > kMergeInKernelParts;
  if (split) {
    p.ws_o = ws_out;
    p.ws_m = ws_m;
    p.ws_l = ws_l;
    p.counters = merge_apart ? nullptr : counters;
    p.order = order;
    p.max_partitions = max_partitions;
    p.partition_blocks = partition_size / block_size;
  } else {
    p.max_partitions = 1;
    p.partition_blocks = max_blocks_per_seq;
  }
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, split, st);
  if (e == cudaSuccess && merge_apart) {
    ReduceParams r{};
    r.out = p.out;
    r.ws_o = ws_out;
    r.ws_m = ws_m;
    r.ws_l = ws_l;
    r.context_lens = context_lens;
    r.err = p.err;
    r.num_seqs = num_seqs;
    r.num_q_heads = num_q_heads;
    r.max_partitions = max_partitions;
    r.partition_size = partition_size;
    e = launch_splitk_reduce(r, head_dim, st);
  }
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

// Shared-prefix decode step: the prefix's partitions by the tensor-core
// prefill kernel (all queries of the batch against the shared keys), the
// rest by the fused split-K decode (with the cache write), which overlaps the
// first and merges every sequence's partitions in its last CTA.
pa_status pa_decode_step_shared_prefix(void* out, const void* q, const void* key,
                                       const void* value, const int64_t* slot_mapping,
                                       void* k_cache, void* v_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int num_blocks, float scale,
                                       int prefix_len, int prefix_split, int partition_size,
                                       float* ws_out, float* ws_m, float* ws_l,
                                       unsigned* counters, int max_partitions,
                                       const int32_t* order, pa_stream_t stream) {
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale);
  if (s != PA_OK) return s;
  // the prefix launch (the prefill kernel) takes row maxima of unscaled
  // scores: a positive scale only, as pa_prefill
  if (!(scale > 0.f) || prefix_split <= 0 ||
      prefix_split % block_size != 0 || prefix_len <= 0 ||
      prefix_len % prefix_split != 0 || prefix_len / block_size > max_blocks_per_seq ||
      partition_size <= 0 || partition_size % block_size != 0 ||
      max_partitions <= prefix_len / prefix_split || max_partitions > 65535)
    return PA_ERR_INVALID_ARG;
  if (!pa_prefill_supported(head_dim, num_q_heads / num_kv_heads, block_size) ||
      num_seqs > 65535)
    return PA_ERR_UNSUPPORTED_SHAPE;
  if (num_seqs == 0) return PA_OK;
  const bool write = key != nullptr || value != nullptr || slot_mapping != nullptr;
  if (!ok_ptr(out, 16) || !ok_ptr(ws_out, 16) || !ok_ptr(ws_m, 4) || !ok_ptr(ws_l, 4) ||
      !ok_ptr(counters, 4))
    return PA_ERR_INVALID_ARG;
  if (write && (!ok_ptr(key, 16) || !ok_ptr(value, 16) || !ok_ptr(slot_mapping, 8)))
    return PA_ERR_INVALID_ARG;
  const int splits = prefix_len / prefix_split;
  if (order != nullptr) {
    if (!ok_ptr(order, 4)) return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_seqs) * (max_partitions - splits) > 65535)
      return PA_ERR_UNSUPPORTED_SHAPE;
  }
  unsigned* err = device_error_word();
  if (!err) return cuda_fail(cudaGetLastError());
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_prefix_partials(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                         context_lens, num_seqs, num_q_heads, num_kv_heads,
                                         num_blocks, scale, prefix_split / block_size, splits,
                                         ws_out, ws_m, ws_l, max_partitions, err, st);
  if (e != cudaSuccess) return cuda_fail(e);
  DecodeParams p = make_decode_params(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                      context_lens, num_seqs, num_q_heads, num_kv_heads,
                                      num_blocks, scale);
  p.out = static_cast<__nv_bfloat16*>(out);
  if (write) {
    p.new_key = static_cast<const __nv_bfloat16*>(key);
    p.new_value = static_cast<const __nv_bfloat16*>(value);
    p.slot_mapping = slot_mapping;
  }
  p.ws_o = ws_out;
  p.ws_m = ws_m;
  p.ws_l = ws_l;
  p.counters = counters;
  p.max_partitions = max_partitions;
  p.partition_blocks = partition_size / block_size;
  p.first_partition = splits;
  p.prefix_blocks = prefix_len / block_size;
  p.order = order;
  p.err = err;
  e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, true, st);
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_decode_step(void* out, const void* q, const void* key, const void* value,
                         const int64_t* slot_mapping, void* k_cache, void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         float scale, int partition_size, float* ws_out, float* ws_m,
                         float* ws_l, unsigned* counters, int max_partitions,
                         const int32_t* order, int flags, pa_stream_t stream) {
  return decode_step_impl(out, q, key, value, slot_mapping, k_cache, v_cache, nullptr, nullptr,
                          block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                          num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                          ws_out, ws_m, ws_l, counters, max_partitions, order, flags, 0, stream);
}

pa_status pa_decode_step_int8(void* out, const void* q, const void* key, const void* value,
                              const int64_t* slot_mapping, int8_t* k_cache, int8_t* v_cache,
                              float* k_scales, float* v_scales, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, float scale, int partition_size, float* ws_out,
                              float* ws_m, float* ws_l, unsigned* counters, int max_partitions,
                              const int32_t* order, int flags, pa_stream_t stream) {
  return decode_step_impl(out, q, key, value, slot_mapping, k_cache, v_cache, k_scales, v_scales,
                          block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                          num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                          ws_out, ws_m, ws_l, counters, max_partitions, order, flags, 1, stream);
}

pa_status pa_decode_step_fp8(void* out, const void* q, const void* key, const void* value,
                             const int64_t* slot_mapping, uint8_t* k_cache, uint8_t* v_cache,
                             float* k_scales, float* v_scales, const int32_t* block_tables,
                             int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, float scale, int partition_size, float* ws_out,
                             float* ws_m, float* ws_l, unsigned* counters, int max_partitions,
                             const int32_t* order, int flags, pa_stream_t stream) {
  return decode_step_impl(out, q, key, value, slot_mapping, k_cache, v_cache, k_scales, v_scales,
                          block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                          num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                          ws_out, ws_m, ws_l, counters, max_partitions, order, flags, 2, stream);
}

}  // extern "C"
