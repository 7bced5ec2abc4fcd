// Split-K paged decode for callers that cannot allocate device memory.
//
// Some callers of this library are not allowed to call cudaMalloc: serving
// runtimes that reserve the whole device memory up front for their own KV
// pool and weights (any further allocation either fails or breaks their
// memory budget), and latency-critical host threads that must not take the
// device-wide synchronisation cudaMalloc / cudaFree can imply.  The regular
// split-K entry points (pa_decode_splitk + pa_splitk_reduce) need a caller-
// allocated fp32 workspace; pa_decode_splitk_noalloc runs the same two
// kernels with that workspace placed in a fixed-size array compiled into this
// library instead, so the caller passes only inputs and the output.
//
// The array lives in device memory of every GPU that loads the library, for
// the life of the process.  All calls share it: two calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on
// it.  Nothing in it has to start at zero -- each call writes every partition
// it later reads -- so it is never cleared, and it keeps the last call's
// partials.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pa.h"
#include "internal.h"

namespace pa {
namespace {

constexpr size_t kNoallocFloats = PA_DECODE_NOALLOC_WORKSPACE_BYTES / sizeof(float);

// The shared split-K workspace.  In host code this name is only a stand-in
// for the device object: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_workspace[kNoallocFloats];

constexpr int kMaxDevices = 64;
std::atomic<float*> g_noalloc_ptr[kMaxDevices];

// Device address of the workspace on the current device, looked up once per
// device (the first call on each device does this).
cudaError_t noalloc_workspace(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  float* ptr = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_noalloc_workspace);
    if (e != cudaSuccess) return e;
    ptr = static_cast<float*>(addr);
    g_noalloc_ptr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_splitk_noalloc(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              int max_blocks_per_seq, const int32_t* context_lens,
                                              int num_seqs, int num_q_heads, int num_kv_heads,
                                              int head_dim, int block_size, int num_blocks,
                                              float scale, int partition_size,
                                              int max_context_len, pa_stream_t stream) {
  using namespace pa;
  if (max_context_len < 0 || partition_size <= 0 || partition_size % 16 != 0 || num_seqs < 0 ||
      num_q_heads <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  const size_t parts =
      max_context_len == 0 ? 1 : (static_cast<size_t>(max_context_len) + partition_size - 1) /
                                     partition_size;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * parts;
  if (parts > 65535 || rows * (static_cast<size_t>(head_dim) + 2) > kNoallocFloats)
    return PA_ERR_INVALID_ARG;  // beyond PA_DECODE_NOALLOC_WORKSPACE_BYTES
  float* ws = nullptr;
  cudaError_t e = noalloc_workspace(&ws);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  float* ws_out = ws;
  float* ws_m = ws + rows * head_dim;
  float* ws_l = ws_m + rows;
  const int maxp = static_cast<int>(parts);
  pa_status s = pa_decode_splitk(ws_out, ws_m, ws_l, maxp, q, k_cache, v_cache, block_tables,
                                 max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                                 num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 partition_size, stream);
  if (s != PA_OK) return s;
  return pa_splitk_reduce(out, ws_out, ws_m, ws_l, maxp, context_lens, num_seqs, num_q_heads,
                          head_dim, partition_size, stream);
}
