// One (token, KV head) row of the cache write, shared by the cache-write
// kernels and the fused decode step so that both write identical bytes.
//
// "How LLM Inference Serving Works" (dev.to), section "Putting It Together:
// The Life of a Request in vLLM": each decode step appends one token's K and
// V into the request's current block.  For the 1-byte caches every row gets
// one fp32 scale (INT8: amax / 127, code = round-half-even(x / scale);
// FP8: amax / 448, code = E4M3 of fp32(x / scale), nearest-even, saturated),
// and V tiles are stored transposed (v_tile_pos; INT8 V codes offset by 128).
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

// Byte offset of the V code of token t (0..15) and dim d within a 1-byte V
// tile of 16 * D bytes (the layout pa.h states).  The tile is stored
// transposed for the decode's f16 tensor-core PV: lane L = 4 * gid + tig of a
// warp reads the D / 2 bytes at L * D / 2, one 32-bit word per dim it feeds
// to the MMA (dims 16c + gid and 16c + gid + 8 of m-tile c), each word holding
// that dim's codes of tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9 (the MMA's
// k indices of the lane), and the lane's 16-byte chunks are XOR-permuted so
// that the 8 lanes of a shared-memory phase hit 8 different bank groups.
template <int D>
__host__ __device__ __forceinline__ int v_tile_pos(int t, int d) {
  const int r = d & 15;
  const int lane = 4 * (r & 7) + ((t & 7) >> 1);
  const int word = 2 * (d >> 4) + (r >> 3);
  const int byte = (t & 1) | ((t >> 3) << 1);
  const int f = D == 128 ? ((lane >> 1) & 3) : ((lane >> 2) & 1);
  return lane * (D / 2) + 16 * ((word >> 2) ^ f) + 4 * (word & 3) + byte;
}

// V codes as stored: INT8 codes offset by 128 (offset binary, so that the
// decode turns a byte into an exact f16 with one byte permute and one add),
// E4M3 codes unchanged.
template <bool F8>
__device__ __forceinline__ uint32_t v_stored(uint32_t codes) {
  return F8 ? codes : codes ^ 0x80808080u;
}

// Stores the lane's PER = D / 32 V bytes (logical dims lane * PER + i of
// token `off`, packed little-endian in `bytes`) into a V tile at `tile`.
template <int D, typename T>
__device__ __forceinline__ void store_v_row_bytes(T* tile, int off, int lane, uint32_t bytes) {
  constexpr int PER = D / 32;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    reinterpret_cast<unsigned char*>(tile)[v_tile_pos<D>(off, lane * PER + i)] =
        static_cast<unsigned char>(bytes >> (8 * i));
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
// block.  K rows are plain row-major; V bytes go to their places in the
// transposed tile (v_tile_pos).  All 32 lanes must call it.
template <int D, bool F8>
__device__ __forceinline__ void write_row_1byte(const uint32_t (&kw)[D / 64],
                                                const uint32_t (&vw)[D / 64], int8_t* k8,
                                                int8_t* v8, float* k_scales, float* v_scales,
                                                int64_t srow, int off, int lane) {
  constexpr int PER = D / 32;
  float ks, vs;
  const uint32_t kc = quantise_row<D, F8>(kw, &ks);
  const uint32_t vc = quantise_row<D, F8>(vw, &vs);
  int8_t* kdst = k8 + srow * D + lane * PER;
  if constexpr (PER == 4)
    *reinterpret_cast<uint32_t*>(kdst) = kc;
  else
    *reinterpret_cast<uint16_t*>(kdst) = static_cast<uint16_t>(kc);
  store_v_row_bytes<D>(v8 + (srow - off) * D, off, lane, v_stored<F8>(vc));
  if (lane == 0) {
    k_scales[srow] = ks;
    v_scales[srow] = vs;
  }
}

}  // namespace pa
