// One (token, KV head) row of the cache write, shared by the cache-write
// kernels and the fused decode step so that both write identical bytes.
//
// "How LLM Inference Serving Works" (dev.to), section "Putting It Together:
// The Life of a Request in vLLM": each decode step appends one token's K and
// V into the request's current block.  For the 1-byte caches every row gets
// one fp32 scale (INT8: amax / 127, code = round-half-even(x / scale);
// FP8: amax / 448, code = E4M3 of fp32(x / scale), nearest-even, saturated),
// and V tiles store their 16-byte units permuted (see pa.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"

namespace pa {

// A row of D values spread over a warp, D / 32 per lane (lane l owns
// [l * D / 32, (l + 1) * D / 32)), quantised with the row's scale.  Returns
// the lane's codes packed little-endian in a word (D / 32 <= 4 bytes) and
// sets *scale_out on every lane.  w: the lane's values as bf16 pairs.  All 32
// lanes must call it.
template <int D, bool F8>
__device__ __forceinline__ uint32_t quantise_row(const uint32_t (&w)[D / 64], float* scale_out) {
  constexpr int PER = D / 32;
  float f[PER];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) {
    const float2 x = bf16x2_to_float2(w[i]);
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
  *scale_out = scale;
  return packed;
}

// Byte offset, within row `off` of a V tile of D-byte rows, at which the code
// of logical column col is stored (16-byte unit u of 128-byte line L of the
// tile sits at unit u ^ ((2L) & 7)).
template <int D>
__device__ __forceinline__ int v_code_col(int off, int col) {
  const int unit = (off * D + col) >> 4;  // within the tile
  const int line = unit >> 3;
  return ((((unit & 7) ^ ((2 * line) & 7)) + 8 * line) << 4) - off * D + (col & 15);
}

// Loads this lane's D / 32 values of a bf16 row as bf16 pairs.
template <int D>
__device__ __forceinline__ void load_row_words(const __nv_bfloat16* row, int lane,
                                               uint32_t (&w)[D / 64]) {
#pragma unroll
  for (int i = 0; i < D / 64; ++i)
    w[i] = __ldg(reinterpret_cast<const unsigned int*>(row + lane * (D / 32)) + i);
}

// Quantises and stores one token's K and V rows of one KV head (kw / vw: the
// lane's values, load_row_words), k8 / v8 the pools, srow = (block * Hkv +
// head) * block_size + offset (the scale index), off = the offset in the
// block.  All 32 lanes must call it.
template <int D, bool F8>
__device__ __forceinline__ void write_row_1byte(const uint32_t (&kw)[D / 64],
                                                const uint32_t (&vw)[D / 64], int8_t* k8,
                                                int8_t* v8, float* k_scales, float* v_scales,
                                                int64_t srow, int off, int lane) {
  constexpr int PER = D / 32;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    float scale;
    const uint32_t packed = quantise_row<D, F8>(which ? vw : kw, &scale);
    const int col = which ? v_code_col<D>(off, lane * PER) : lane * PER;
    int8_t* dst = (which ? v8 : k8) + srow * D + col;
    if constexpr (PER == 4)
      *reinterpret_cast<uint32_t*>(dst) = packed;
    else
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
    if (lane == 0) (which ? v_scales : k_scales)[srow] = scale;
  }
}

}  // namespace pa
