// The per-tile arithmetic shared by the paged decode kernels: geometry of a
// (block, KV head) tile and one tile's QK, online-softmax update and PV for
// the G query heads of a group (design notes in decode.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "device.cuh"

namespace pa {

constexpr int kBlockSize = 16;

template <int D, int G>
struct Geometry {
  static constexpr int BS = kBlockSize;
  static constexpr int L = D / 8;         // lanes per K/V row, 16 bytes each
  static constexpr int ROWS = 32 / L;     // rows one warp-wide 16-byte load covers
  static constexpr int P = BS / ROWS;     // passes over a tile
  static constexpr int NV = P * G;        // partial dot products per lane
  static constexpr int R = NV / L;        // complete scores per lane after the butterfly
  static constexpr int HEAD_LANES = P / R;  // sub-lanes holding one head's scores
  static constexpr int TILE = BS * D * 2;   // bytes of one (block, KV head) tile
  static_assert(32 % L == 0 && BS % ROWS == 0, "row geometry");
  static_assert(NV % L == 0 && R >= 1 && P % R == 0, "score geometry");
};

// One K/V tile through QK, the online softmax update and PV.
template <int D, int G, bool FULL>
__device__ __forceinline__ void tile_step(const uint4* __restrict__ kt, const uint4* __restrict__ vt,
                                          float* ps, float* alpha_s, const float2 (&q2)[G][4],
                                          float2 (&acc)[G][4], float& m_run, float& l_run,
                                          int nvalid, int lane, int sub, int rg, int my_head,
                                          int my_i0) {
  using Geo = Geometry<D, G>;
  constexpr int L = Geo::L, ROWS = Geo::ROWS, P = Geo::P, NV = Geo::NV, R = Geo::R;

  // QK: partial dots over this lane's 8 dims, value index g * P + i.
  float sc[NV];
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int t = i * ROWS + rg;
    const uint4 w = kt[t * L + sub];
    const float2 k0 = bf16x2_to_float2(w.x), k1 = bf16x2_to_float2(w.y);
    const float2 k2 = bf16x2_to_float2(w.z), k3 = bf16x2_to_float2(w.w);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float2 a = __fmul2_rn(q2[g][0], k0);
      a = __ffma2_rn(q2[g][1], k1, a);
      a = __ffma2_rn(q2[g][2], k2, a);
      a = __ffma2_rn(q2[g][3], k3, a);
      sc[g * P + i] = a.x + a.y;
    }
  }

  // Transposing butterfly across the L lanes of a row: at each level a lane
  // keeps one half of its values (upper half if its mask bit is set), adds
  // the partner's copy of that half, and sends the other half away.  After
  // log2(L) levels lane `sub` holds values [sub*R, sub*R + R), complete.
#pragma unroll
  for (int m = L / 2, n = NV; m >= 1; m >>= 1, n >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = up ? sc[k] : sc[k + n / 2];
      const float keep = up ? sc[k + n / 2] : sc[k];
      sc[k] = keep + __shfl_xor_sync(kFullMask, send, m);
    }
  }

  // Online softmax for this lane's head (all lanes of a head agree on m_run).
  float s[R];
  float mx = -INFINITY;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = (my_i0 + r) * ROWS + rg;
    s[r] = (FULL || t < nvalid) ? sc[r] : -INFINITY;
    mx = fmaxf(mx, s[r]);
  }
#pragma unroll
  for (int m = 1; m < Geo::HEAD_LANES; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
#pragma unroll
  for (int m = L; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
  const float m_new = fmaxf(m_run, mx);  // finite: every tile has a valid token
  const float alpha = exp2f(m_run - m_new);
  float psum = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float pr = exp2f(s[r] - m_new);
    psum += pr;
    ps[((my_i0 + r) * ROWS + rg) * G + my_head] = pr;
  }
  l_run = l_run * alpha + psum;
  m_run = m_new;
  if (sub % Geo::HEAD_LANES == 0 && rg == 0) alpha_s[my_head] = alpha;
  const bool rescale = __any_sync(kFullMask, alpha != 1.0f);
  __syncwarp();

  if (rescale) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float a = alpha_s[g];
      const float2 a2 = make_float2(a, a);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[g][k] = __fmul2_rn(acc[g][k], a2);
    }
  }

  // PV: acc[g][dims] += p[t][g] * V[t][dims] for this lane's tokens.
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int t = i * ROWS + rg;
    if (FULL || t < nvalid) {
      const uint4 w = vt[t * L + sub];
      const float2 v0 = bf16x2_to_float2(w.x), v1 = bf16x2_to_float2(w.y);
      const float2 v2 = bf16x2_to_float2(w.z), v3 = bf16x2_to_float2(w.w);
      float pw[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int g = 0; g < G; g += 4) {
          const float4 x = *reinterpret_cast<const float4*>(ps + t * G + g);
          pw[g] = x.x;
          pw[g + 1] = x.y;
          pw[g + 2] = x.z;
          pw[g + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int g = 0; g < G; g += 2) {
          const float2 x = *reinterpret_cast<const float2*>(ps + t * G + g);
          pw[g] = x.x;
          pw[g + 1] = x.y;
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 pp = make_float2(pw[g], pw[g]);
        acc[g][0] = __ffma2_rn(pp, v0, acc[g][0]);
        acc[g][1] = __ffma2_rn(pp, v1, acc[g][1]);
        acc[g][2] = __ffma2_rn(pp, v2, acc[g][2]);
        acc[g][3] = __ffma2_rn(pp, v3, acc[g][3]);
      }
    }
  }
}

}  // namespace pa

namespace pa {

// ---------------------------------------------------------------------------
// INT8 KV cache (one fp32 scale per token and KV head; see pa.h).  A tile is
// K codes [16][D] int8, V codes [16][D] int8, then the 16 K and 16 V scales.
// QK is an integer dot product (q quantised per head to int8 in the CTA
// prologue), exact in int32 through the cross-lane reduction; the K and q
// scales are applied once per score.  PV stays in fp32: V codes become floats
// and the V scale is folded into each softmax weight.

// 8 int8 codes (two words) to floats: byte b becomes the float 2^23 + b + 128
// (bits 0x4B0000xx), from which 2^23 + 128 is subtracted exactly.
__device__ __forceinline__ void int8x8_to_float(const uint2 w, float2 (&f)[4]) {
  const uint32_t a = w.x ^ 0x80808080u, b = w.y ^ 0x80808080u;
  const float2 off = make_float2(-8388736.0f, -8388736.0f);
  f[0] = make_float2(__uint_as_float(__byte_perm(a, 0x4B000000u, 0x7540)),
                     __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7541)));
  f[1] = make_float2(__uint_as_float(__byte_perm(a, 0x4B000000u, 0x7542)),
                     __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7543)));
  f[2] = make_float2(__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7540)),
                     __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7541)));
  f[3] = make_float2(__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7542)),
                     __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7543)));
#pragma unroll
  for (int k = 0; k < 4; ++k) f[k] = __fadd2_rn(f[k], off);
}

template <int D, int G, bool FULL>
__device__ __forceinline__ void tile_step_i8(const uint2* __restrict__ kt,
                                             const uint2* __restrict__ vt,
                                             const float* __restrict__ ksc,
                                             const float* __restrict__ vsc, float* ps,
                                             float* alpha_s, const int (&qc)[G][2],
                                             const float (&qsc)[G], float2 (&acc)[G][4],
                                             float& m_run, float& l_run, int nvalid, int lane,
                                             int sub, int rg, int my_head, int my_i0) {
  using Geo = Geometry<D, G>;
  constexpr int L = Geo::L, ROWS = Geo::ROWS, P = Geo::P, NV = Geo::NV, R = Geo::R;

  // QK: integer partial dots over this lane's 8 dims, value index g * P + i.
  int sc[NV];
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const uint2 w = kt[(i * ROWS + rg) * L + sub];
#pragma unroll
    for (int g = 0; g < G; ++g)
      sc[g * P + i] = __dp4a(qc[g][1], static_cast<int>(w.y),
                             __dp4a(qc[g][0], static_cast<int>(w.x), 0));
  }
  // the transposing butterfly of tile_step, on exact int32 sums
#pragma unroll
  for (int m = L / 2, n = NV; m >= 1; m >>= 1, n >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const int send = up ? sc[k] : sc[k + n / 2];
      const int keep = up ? sc[k + n / 2] : sc[k];
      sc[k] = keep + __shfl_xor_sync(kFullMask, send, m);
    }
  }

  float s[R];
  float mx = -INFINITY;
  float my_qsc = qsc[0];  // this lane's head's q scale (times scale * log2 e)
#pragma unroll
  for (int g = 1; g < G; ++g)
    if (my_head == g) my_qsc = qsc[g];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = (my_i0 + r) * ROWS + rg;
    s[r] = (FULL || t < nvalid) ? static_cast<float>(sc[r]) * my_qsc * ksc[t] : -INFINITY;
    mx = fmaxf(mx, s[r]);
  }
#pragma unroll
  for (int m = 1; m < Geo::HEAD_LANES; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
#pragma unroll
  for (int m = L; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
  const float m_new = fmaxf(m_run, mx);
  const float alpha = exp2f(m_run - m_new);
  float psum = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = (my_i0 + r) * ROWS + rg;
    const float pr = exp2f(s[r] - m_new);
    psum += pr;
    ps[t * G + my_head] = pr * ((FULL || t < nvalid) ? vsc[t] : 0.f);  // V scale folded in
  }
  l_run = l_run * alpha + psum;
  m_run = m_new;
  if (sub % Geo::HEAD_LANES == 0 && rg == 0) alpha_s[my_head] = alpha;
  const bool rescale = __any_sync(kFullMask, alpha != 1.0f);
  __syncwarp();

  if (rescale) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float a = alpha_s[g];
      const float2 a2 = make_float2(a, a);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[g][k] = __fmul2_rn(acc[g][k], a2);
    }
  }

#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int t = i * ROWS + rg;
    if (FULL || t < nvalid) {
      float2 v[4];
      int8x8_to_float(vt[t * L + sub], v);
      float pw[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int g = 0; g < G; g += 4) {
          const float4 x = *reinterpret_cast<const float4*>(ps + t * G + g);
          pw[g] = x.x;
          pw[g + 1] = x.y;
          pw[g + 2] = x.z;
          pw[g + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int g = 0; g < G; g += 2) {
          const float2 x = *reinterpret_cast<const float2*>(ps + t * G + g);
          pw[g] = x.x;
          pw[g + 1] = x.y;
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 pp = make_float2(pw[g], pw[g]);
        acc[g][0] = __ffma2_rn(pp, v[0], acc[g][0]);
        acc[g][1] = __ffma2_rn(pp, v[1], acc[g][1]);
        acc[g][2] = __ffma2_rn(pp, v[2], acc[g][2]);
        acc[g][3] = __ffma2_rn(pp, v[3], acc[g][3]);
      }
    }
  }
}

}  // namespace pa
