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

// INT8 cache write: one warp per (token, KV head) row quantises it with one
// scale (scale = amax / 127, code = round-half-even(x / scale), fp32, as in
// pa.h) and writes D codes and the scale.  Each lane owns D / 32 values.
// F8: the same with FP8 (E4M3) codes: scale = amax / 448 (E4M3's largest
// finite value), code = E4M3 of fp32(x / scale), round to nearest even,
// saturated (cvt.rn.satfinite).
template <int D, bool F8>
__global__ void __launch_bounds__(256) reshape_and_cache_int8_kernel(const CacheWriteParams p) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int PER = D / 32;  // values per lane: 4 at D = 128, 2 at D = 64
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(p.num_tokens) * p.num_kv_heads) return;  // warp-uniform
  const int h = static_cast<int>(row % p.num_kv_heads);
  const int64_t t = row / p.num_kv_heads;
  const __nv_bfloat16* kp = p.key + row * D + lane * PER;
  const __nv_bfloat16* vp = p.value + row * D + lane * PER;
  uint32_t kw[PER / 2], vw[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) {
    kw[i] = __ldg(reinterpret_cast<const unsigned int*>(kp) + i);
    vw[i] = __ldg(reinterpret_cast<const unsigned int*>(vp) + i);
  }
  const int64_t slot = __ldg(p.slot_mapping + t);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (lane == 0) raise_error(p.err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / p.block_size;
  const int64_t off = slot % p.block_size;
  const int64_t srow = (blk * p.num_kv_heads + h) * p.block_size + off;  // scale index
  for (int which = 0; which < 2; ++which) {
    float f[PER];
#pragma unroll
    for (int i = 0; i < PER / 2; ++i) {
      const float2 x = bf16x2_to_float2(which ? vw[i] : kw[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, m));
    const float scale = __fdiv_rn(amax, F8 ? 448.0f : 127.0f);
    uint32_t packed = 0;
    if (scale > 0.f) {
      if constexpr (F8) {
#pragma unroll
        for (int i = 0; i < PER; i += 2) {
          const __nv_fp8x2_storage_t c2 = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(f[i], scale), __fdiv_rn(f[i + 1], scale)), __NV_SATFINITE,
              __NV_E4M3);
          packed |= static_cast<uint32_t>(c2) << (8 * i);
        }
      } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const float c = fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(f[i], scale))));
          packed |= (static_cast<uint32_t>(static_cast<int>(c)) & 0xffu) << (8 * i);
        }
      }
    }
    // K rows are plain; V tiles have their 16-byte units permuted within each
    // 128-byte line (unit u of line L at u ^ ((2L) & 7)), see pa.h
    int64_t col = lane * PER;
    if (which) {
      const int unit = static_cast<int>((off * D + col) >> 4);  // within the tile
      const int line = unit >> 3;
      col = ((((unit & 7) ^ ((2 * line) & 7)) + 8 * line) << 4) - off * D + (col & 15);
    }
    int8_t* dst = (which ? p.v8 : p.k8) + srow * D + col;
    if constexpr (PER == 4)
      *reinterpret_cast<uint32_t*>(dst) = packed;
    else
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
    if (lane == 0) (which ? p.v_scales : p.k_scales)[srow] = scale;
  }
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
