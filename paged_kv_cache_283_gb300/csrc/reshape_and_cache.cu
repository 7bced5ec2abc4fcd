// Cache write: scatter each new token's K and V into the block pool by slot.
//
// "How LLM Inference Serving Works" (dev.to), section "Putting It Together:
// The Life of a Request in vLLM": each decode step appends one token's K and
// V into the request's current block.  A slot names (block, offset) as
// block * block_size + offset; negative slots are padding and are skipped.
//
// Pure data movement, a few hundred KiB per call: one thread per 16-byte
// chunk of a (token, KV head) row, moving that chunk of K and of V with
// 16-byte loads and stores.  Consecutive threads cover consecutive chunks of
// a row, so both the reads of key/value and the writes into the pool are
// fully coalesced 16-byte accesses.  Bad slots are never written: they set
// PA_DEVERR_SLOT.

#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cache_row.cuh"
#include "device.cuh"
#include "internal.h"

namespace pa {

namespace {

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const CacheWriteParams p) {
  griddep_wait();  // the producer of key / value / slots is complete
  griddep_launch_dependents();
  const int chunks = p.head_dim / 8;  // 16-byte chunks per row
  const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * chunks;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int c = static_cast<int>(idx % chunks);
  const int64_t row = idx / chunks;  // token * Hkv + head
  const int h = static_cast<int>(row % p.num_kv_heads);
  const int64_t t = row / p.num_kv_heads;
  // the new K/V chunk and its slot are independent loads: issue them together
  const int64_t src = row * p.head_dim + c * 8;
  const uint4 kv = __ldg(reinterpret_cast<const uint4*>(p.key + src));
  const uint4 vv = __ldg(reinterpret_cast<const uint4*>(p.value + src));
  const int64_t slot = __ldg(p.slot_mapping + t);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (c == 0) raise_error(p.err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / p.block_size;
  const int64_t off = slot % p.block_size;
  const int64_t dst = ((blk * p.num_kv_heads + h) * p.block_size + off) * p.head_dim + c * 8;
  *reinterpret_cast<uint4*>(p.k_cache + dst) = kv;
  *reinterpret_cast<uint4*>(p.v_cache + dst) = vv;
}

// INT8 / FP8 cache write: one warp per (token, KV head) row quantises it with
// one scale and writes D codes and the scale (write_row_1byte: INT8 scale =
// amax / 127, code = round-half-even(x / scale); FP8 scale = amax / 448, code
// = E4M3 of x / scale, nearest-even, saturated).  Each lane owns D / 32 values.
template <int D, bool F8>
__global__ void __launch_bounds__(256) reshape_and_cache_int8_kernel(const CacheWriteParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(p.num_tokens) * p.num_kv_heads) return;  // warp-uniform
  const int h = static_cast<int>(row % p.num_kv_heads);
  const int64_t t = row / p.num_kv_heads;
  uint32_t kw[D / 64], vw[D / 64];
  load_row_words<D>(p.key + row * D, lane, kw);
  load_row_words<D>(p.value + row * D, lane, vw);
  const int64_t slot = __ldg(p.slot_mapping + t);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (lane == 0) raise_error(p.err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / p.block_size;
  const int off = static_cast<int>(slot % p.block_size);
  const int64_t srow = (blk * p.num_kv_heads + h) * p.block_size + off;  // scale index
  write_row_1byte<D, F8>(kw, vw, p.k8, p.v8, p.k_scales, p.v_scales, srow, off, lane);
}

}  // namespace

cudaError_t launch_reshape_and_cache_int8(const CacheWriteParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (p.head_dim == 128)
    return p.fp8 ? launch_pdl(reshape_and_cache_int8_kernel<128, true>, grid, dim3(256), 0, stream, p)
                 : launch_pdl(reshape_and_cache_int8_kernel<128, false>, grid, dim3(256), 0, stream, p);
  if (p.head_dim == 64)
    return p.fp8 ? launch_pdl(reshape_and_cache_int8_kernel<64, true>, grid, dim3(256), 0, stream, p)
                 : launch_pdl(reshape_and_cache_int8_kernel<64, false>, grid, dim3(256), 0, stream, p);
  return cudaErrorInvalidValue;
}

cudaError_t launch_reshape_and_cache(const CacheWriteParams& p, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(p.num_tokens) * p.num_kv_heads * (p.head_dim / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  return launch_pdl(reshape_and_cache_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
                    stream, p);
}

}  // namespace pa
