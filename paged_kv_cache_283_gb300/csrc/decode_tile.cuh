// The per-tile arithmetic shared by the paged decode kernels: geometry of a
// (block, KV head) tile and one tile's QK, online-softmax update and PV for
// the G query heads of a group (design notes in decode.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
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
//
// QK is an exact integer dot product of the codes (q is quantised per head
// by the CTA before the loop) and has its own lane geometry: QL lanes share a
// K row, each holding QB = D/QL code bytes of every head of the group in
// registers, so a pass covers 32/QL rows and the butterfly that completes the
// partial dots has only log2(QL) levels (QL = 4: 2 levels; the bf16 step
// needs 4).  The K and q scales are applied once per score.  PV runs on the
// tensor cores (pv_q_mma) with the V scale folded into each softmax weight.
template <int D, int G>
struct I8Geometry {
  static constexpr int BS = kBlockSize;
  static constexpr int QL = G >= 8 ? 8 : 4;  // lanes per K row
  static constexpr int QB = D / QL;          // code bytes per lane and row
  static constexpr int QW = QB / 4;          // 32-bit words of codes per lane and head
  static constexpr int ROWS = 32 / QL;       // rows per pass
  static constexpr int P = BS / ROWS;        // passes over a tile
  static constexpr int NV = P * G;           // partial dots per lane
  static constexpr int R = NV / QL;          // complete scores per lane after the butterfly
  static constexpr int HEAD_LANES = P / R;   // lanes holding one head's scores of a row group
  static_assert(QB == 8 || QB == 16 || QB == 32, "code bytes per lane");
  static_assert(NV % QL == 0 && R >= 1 && P % R == 0, "int8 score geometry");
};

// The 16-byte chunks lane (qrg, qsub) reads from each K row, in order.  With
// 32 bytes per lane, odd row groups take their two chunks in the opposite
// order so that the 8 lanes of a shared-memory phase hit 8 different chunks.
template <int QB>
__device__ __forceinline__ int i8_chunk(int qsub, int qrg, int k) {
  if constexpr (QB == 32) return 2 * qsub + (k ^ (qrg & 1));
  else return qsub;  // QB <= 16: one chunk (or half of one)
}

// Loads this lane's QB code bytes of one row (a K row, or q of one head) in
// i8_chunk order, as QW words.
template <int QB>
__device__ __forceinline__ void i8_load_row(const unsigned char* row, int qsub, int qrg,
                                            int (&w)[QB / 4]) {
  if constexpr (QB == 32) {
    const int4 a = *reinterpret_cast<const int4*>(row + 16 * i8_chunk<32>(qsub, qrg, 0));
    const int4 c = *reinterpret_cast<const int4*>(row + 16 * i8_chunk<32>(qsub, qrg, 1));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = c.x; w[5] = c.y; w[6] = c.z; w[7] = c.w;
  } else if constexpr (QB == 16) {
    const int4 a = *reinterpret_cast<const int4*>(row + 16 * qsub);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else {
    const int2 a = *reinterpret_cast<const int2*>(row + 8 * qsub);
    w[0] = a.x; w[1] = a.y;
  }
}

// One m16n8k8 tf32 tensor-core step, fp32 accumulate: c += a · b.
__device__ __forceinline__ void mma_tf32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// 4 int8 codes (one word) to exact floats, bit patterns for the tf32 MMA.
__device__ __forceinline__ void int8x4_to_tf32(uint32_t w, uint32_t (&f)[4]) {
  const uint32_t a = w ^ 0x80808080u;
  const float2 off = make_float2(-8388736.0f, -8388736.0f);
  float2 lo = make_float2(__uint_as_float(__byte_perm(a, 0x4B000000u, 0x7540)),
                          __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7541)));
  float2 hi = make_float2(__uint_as_float(__byte_perm(a, 0x4B000000u, 0x7542)),
                          __uint_as_float(__byte_perm(a, 0x4B000000u, 0x7543)));
  lo = __fadd2_rn(lo, off);
  hi = __fadd2_rn(hi, off);
  f[0] = __float_as_uint(lo.x);
  f[1] = __float_as_uint(lo.y);
  f[2] = __float_as_uint(hi.x);
  f[3] = __float_as_uint(hi.y);
}

// PV of one INT8 or FP8 tile on the tensor cores: out^T[dim][head] += V^T[dim][token]
// · W[token][head] with m16n8k8 tf32 MMAs (M = 16 dims, N = 8 heads, the
// group padded with zeros, K = 8 tokens), two K steps per tile.  V codes
// (small integers, or E4M3 values) are exact in tf32; each weight W (softmax weight times the
// token's V scale) is split into two tf32 parts, hi + lo, one MMA each, so
// the products keep ~21 bits.  Lane (gid = lane / 4, tig = lane % 4) owns, in
// MMA c, dims d0 = (D/8)·gid + 2c (row gid) and d0 + 1 (row gid + 8), and
// heads 2·tig, 2·tig + 1: acc[c] = {(d0, 2tig), (d0, 2tig+1), (d0+1, 2tig),
// (d0+1, 2tig+1)}.  It reads the D/8 code bytes at dims [(D/8)·gid, +D/8) of
// tokens tig, tig + 4, tig + 8, tig + 12; the V tile's 16-byte units are
// permuted within each 128-byte line (unit u of line L at u ^ (2L & 7)), which
// puts the 8 lanes of every shared-memory phase on 8 different units.
template <int D>
__device__ __forceinline__ const unsigned char* v_i8_row_run(const unsigned char* vt, int t,
                                                              int gid) {
  constexpr int RUN = D / 8;                 // bytes per lane and token: 16 or 8
  const int unit = (t * D + RUN * gid) >> 4;  // logical 16-byte unit in the tile
  const int line = unit >> 3;
  return vt + ((line << 3) + ((unit & 7) ^ ((2 * line) & 7))) * 16 + ((RUN * gid) & 15);
}

// 2 E4M3 codes (16 bits, first code in the low byte) to floats, exact (every
// E4M3 value is exact in f16 and f32).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t h) {
  const __half2_raw r =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(h & 0xFFFFu), __NV_E4M3);
  __half2 v;
  v = *reinterpret_cast<const __half2*>(&r);
  return __half22float2(v);
}

// 4 E4M3 codes (one word) to float bit patterns for the tf32 MMA (exact: 3
// mantissa bits fit tf32's 10).
__device__ __forceinline__ void e4m3x4_to_tf32(uint32_t w, uint32_t (&f)[4]) {
  const float2 lo = e4m3x2_to_float2(w), hi = e4m3x2_to_float2(w >> 16);
  f[0] = __float_as_uint(lo.x);
  f[1] = __float_as_uint(lo.y);
  f[2] = __float_as_uint(hi.x);
  f[3] = __float_as_uint(hi.y);
}

// F8 = false: INT8 codes; true: E4M3 codes.  With E4M3 a code can be NaN, and
// a token past the context (nvalid) has weight 0 but whatever codes the pool
// holds there, so its codes are replaced by 0 (0 * NaN would not be 0).
template <int D, int G, bool F8, bool FULL>
__device__ __forceinline__ void pv_q_mma(const unsigned char* __restrict__ vt,
                                         const float* __restrict__ ps, float (&acc)[D / 16][4],
                                         int lane, int nvalid) {
  constexpr int NWORD = D / 32;  // code words per lane and token
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t whi[4], wlo[4];  // W[token tig + 4j][head gid] = hi + lo
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float w = gid < G ? ps[(tig + 4 * j) * G + gid] : 0.f;
    whi[j] = to_tf32(w);
    wlo[j] = to_tf32(w - __uint_as_float(whi[j]));
  }
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const int t0 = 8 * ks + tig, t1 = t0 + 4;
    const unsigned char* r0 = v_i8_row_run<D>(vt, t0, gid);
    const unsigned char* r1 = v_i8_row_run<D>(vt, t1, gid);
    uint32_t w0[NWORD], w1[NWORD];
    if constexpr (NWORD == 4) {
      const uint4 x = *reinterpret_cast<const uint4*>(r0);
      const uint4 y = *reinterpret_cast<const uint4*>(r1);
      w0[0] = x.x; w0[1] = x.y; w0[2] = x.z; w0[3] = x.w;
      w1[0] = y.x; w1[1] = y.y; w1[2] = y.z; w1[3] = y.w;
    } else {
      const uint2 x = *reinterpret_cast<const uint2*>(r0);
      const uint2 y = *reinterpret_cast<const uint2*>(r1);
      w0[0] = x.x; w0[1] = x.y;
      w1[0] = y.x; w1[1] = y.y;
    }
    if constexpr (F8 && !FULL) {
#pragma unroll
      for (int j = 0; j < NWORD; ++j) {
        if (t0 >= nvalid) w0[j] = 0u;
        if (t1 >= nvalid) w1[j] = 0u;
      }
    }
#pragma unroll
    for (int j = 0; j < NWORD; ++j) {
      uint32_t f0[4], f1[4];
      if constexpr (F8) {
        e4m3x4_to_tf32(w0[j], f0);
        e4m3x4_to_tf32(w1[j], f1);
      } else {
        int8x4_to_tf32(w0[j], f0);
        int8x4_to_tf32(w1[j], f1);
      }
      // word j holds dims 4j .. 4j+3 of the lane's run: MMAs 2j and 2j + 1
      mma_tf32(acc[2 * j], f0[0], f0[1], f1[0], f1[1], whi[2 * ks], whi[2 * ks + 1]);
      mma_tf32(acc[2 * j + 1], f0[2], f0[3], f1[2], f1[3], whi[2 * ks], whi[2 * ks + 1]);
      mma_tf32(acc[2 * j], f0[0], f0[1], f1[0], f1[1], wlo[2 * ks], wlo[2 * ks + 1]);
      mma_tf32(acc[2 * j + 1], f0[2], f0[3], f1[2], f1[3], wlo[2 * ks], wlo[2 * ks + 1]);
    }
  }
}

// One INT8 tile.  (qsub, qrg): this lane in the QK geometry; my_head / my_i0:
// the head and first pass of this lane's scores.
template <int D, int G, bool FULL>
__device__ __forceinline__ void tile_step_i8(const unsigned char* __restrict__ kt,
                                             const unsigned char* __restrict__ vt,
                                             const float* __restrict__ ksc,
                                             const float* __restrict__ vsc, float* ps,
                                             float* alpha_s,
                                             const int (&qc)[G][I8Geometry<D, G>::QW],
                                             const float (&qsc)[G], float (&acc)[D / 16][4],
                                             float& m_run, float& l_run, int nvalid, int lane,
                                             int qsub, int qrg, int my_head, int my_i0) {
  using IG = I8Geometry<D, G>;
  constexpr int QL = IG::QL, QR = IG::ROWS, QP = IG::P, NV = IG::NV, R = IG::R;

  // QK: integer partial dots over this lane's QB bytes, value index g * QP + i.
  int sc[NV];
#pragma unroll
  for (int i = 0; i < QP; ++i) {
    int w[IG::QW];
    i8_load_row<IG::QB>(kt + (i * QR + qrg) * D, qsub, qrg, w);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      int a = 0;
#pragma unroll
      for (int k = 0; k < IG::QW; ++k) a = __dp4a(qc[g][k], w[k], a);
      sc[g * QP + i] = a;
    }
  }
  // the transposing butterfly of tile_step, over QL lanes, on exact int32 sums
#pragma unroll
  for (int m = QL / 2, n = NV; m >= 1; m >>= 1, n >>= 1) {
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
    const int t = (my_i0 + r) * QR + qrg;
    s[r] = (FULL || t < nvalid) ? static_cast<float>(sc[r]) * my_qsc * ksc[t] : -INFINITY;
    mx = fmaxf(mx, s[r]);
  }
#pragma unroll
  for (int m = 1; m < IG::HEAD_LANES; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
#pragma unroll
  for (int m = QL; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
  const float m_new = fmaxf(m_run, mx);
  const float alpha = exp2f(m_run - m_new);
  float psum = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = (my_i0 + r) * QR + qrg;
    const float pr = exp2f(s[r] - m_new);
    psum += pr;
    // V scale folded in; a token past the context gets weight 0 (its codes
    // are finite whatever the pool holds, its scale may not be)
    ps[t * G + my_head] = pr * ((FULL || t < nvalid) ? vsc[t] : 0.f);
  }
  l_run = l_run * alpha + psum;
  m_run = m_new;
  if (qsub % IG::HEAD_LANES == 0 && qrg == 0) alpha_s[my_head] = alpha;
  const bool rescale = __any_sync(kFullMask, alpha != 1.0f);
  __syncwarp();

  if (rescale) {
    const int h0 = 2 * (lane & 3);
    const float a0 = h0 < G ? alpha_s[h0] : 1.f;
    const float a1 = h0 + 1 < G ? alpha_s[h0 + 1] : 1.f;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      acc[c][0] *= a0;
      acc[c][1] *= a1;
      acc[c][2] *= a0;
      acc[c][3] *= a1;
    }
  }
  pv_q_mma<D, G, false, FULL>(vt, ps, acc, lane, nvalid);
}

// One m16n8k16 f16 tensor-core step, fp32 accumulate: c += a · b.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2 E4M3 codes (16 bits, first code in the low byte) to an f16 pair, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t h) {
  const __half2_raw r =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(h & 0xFFFFu), __NV_E4M3);
  return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

// One FP8 (E4M3) tile.  QK on the tensor cores: S[token][head] = K · qᵀ with
// m16n8k16 f16 MMAs (M = the tile's 16 tokens, N = 8 heads, the group padded
// with zeros, K = 16 dims a step).  The codes are exact in f16; q arrives as
// f16 pairs already multiplied by a power of two per head (exact for bf16 q,
// see the kernel's prologue) and qfac undoes it together with scale * log2 e.
// Lane (gid = lane / 4, tig = lane % 4) feeds tokens gid and gid + 8 and reads
// the D/4 code bytes at dims [(D/4)·tig, +D/4) of each; its step-s fragment
// columns 2tig, 2tig+1 | 2tig+8, 2tig+9 are dims (D/4)·tig + 4s + 0, 1 | 2, 3,
// the same dims q's fragment (qf[s], head gid) holds, so the dims reach the
// MMA in a different order than in memory but every one exactly once.  The
// accumulator puts scores (token gid | gid + 8, head 2tig | 2tig + 1) in the
// lane, which are the heads its PV accumulators hold (pv_q_mma), so the
// online softmax state (m_run, l_run: heads 2tig, 2tig + 1) and the rescale
// stay in the lane; l_run is this lane's share, summed over gid at the end.
template <int D, int G, bool FULL>
__device__ __forceinline__ void tile_step_f8(const unsigned char* __restrict__ kt,
                                             const unsigned char* __restrict__ vt,
                                             const float* __restrict__ ksc,
                                             const float* __restrict__ vsc, float* ps,
                                             const uint32_t (&qf)[D / 16][2], float2 qfac,
                                             float (&acc)[D / 16][4], float2& m_run,
                                             float2& l_run, int nvalid, int lane) {
  constexpr int KS = D / 16;  // MMA steps = code words per lane and row
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t w0[KS], w1[KS];  // codes of tokens gid and gid + 8
  {
    const unsigned char* r0 = kt + gid * D + (D / 4) * tig;
    const unsigned char* r1 = r0 + 8 * D;
#pragma unroll
    for (int u = 0; u < KS / 4; ++u) {
      const uint4 x = *reinterpret_cast<const uint4*>(r0 + 16 * u);
      const uint4 y = *reinterpret_cast<const uint4*>(r1 + 16 * u);
      w0[4 * u] = x.x; w0[4 * u + 1] = x.y; w0[4 * u + 2] = x.z; w0[4 * u + 3] = x.w;
      w1[4 * u] = y.x; w1[4 * u + 1] = y.y; w1[4 * u + 2] = y.z; w1[4 * u + 3] = y.w;
    }
  }
  // two independent accumulation chains, summed at the end
  float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int s = 0; s < KS; ++s)
    mma_f16(c[s & 1], e4m3x2_to_f16x2(w0[s]), e4m3x2_to_f16x2(w1[s]),
            e4m3x2_to_f16x2(w0[s] >> 16), e4m3x2_to_f16x2(w1[s] >> 16), qf[s][0], qf[s][1]);

  // scores in base-2 units; a token past the context is masked by position
  // (its codes and scale may be anything, NaN included)
  const bool ok0 = FULL || gid < nvalid, ok1 = FULL || gid + 8 < nvalid;
  const float k0 = ok0 ? ksc[gid] : 0.f, k1 = ok1 ? ksc[gid + 8] : 0.f;
  float s[4];
  s[0] = ok0 ? (c[0][0] + c[1][0]) * k0 * qfac.x : -INFINITY;
  s[1] = ok0 ? (c[0][1] + c[1][1]) * k0 * qfac.y : -INFINITY;
  s[2] = ok1 ? (c[0][2] + c[1][2]) * k1 * qfac.x : -INFINITY;
  s[3] = ok1 ? (c[0][3] + c[1][3]) * k1 * qfac.y : -INFINITY;
  float2 mx = make_float2(fmaxf(s[0], s[2]), fmaxf(s[1], s[3]));
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    mx.x = fmaxf(mx.x, __shfl_xor_sync(kFullMask, mx.x, m));
    mx.y = fmaxf(mx.y, __shfl_xor_sync(kFullMask, mx.y, m));
  }
  const float2 m_new = make_float2(fmaxf(m_run.x, mx.x), fmaxf(m_run.y, mx.y));
  const float2 alpha = make_float2(exp2f(m_run.x - m_new.x), exp2f(m_run.y - m_new.y));
  const float p0 = exp2f(s[0] - m_new.x), p1 = exp2f(s[1] - m_new.y);
  const float p2 = exp2f(s[2] - m_new.x), p3 = exp2f(s[3] - m_new.y);
  l_run = make_float2(l_run.x * alpha.x + (p0 + p2), l_run.y * alpha.y + (p1 + p3));
  m_run = m_new;
  // weights with the V scale folded in; 0 past the context
  const float v0 = ok0 ? vsc[gid] : 0.f, v1 = ok1 ? vsc[gid + 8] : 0.f;
  const int h0 = 2 * tig;
  if (h0 < G) {
    ps[gid * G + h0] = p0 * v0;
    ps[(gid + 8) * G + h0] = p2 * v1;
  }
  if (h0 + 1 < G) {
    ps[gid * G + h0 + 1] = p1 * v0;
    ps[(gid + 8) * G + h0 + 1] = p3 * v1;
  }
  const bool rescale = __any_sync(kFullMask, alpha.x != 1.0f || alpha.y != 1.0f);
  __syncwarp();
  if (rescale) {
#pragma unroll
    for (int cc = 0; cc < D / 16; ++cc) {
      acc[cc][0] *= alpha.x;
      acc[cc][1] *= alpha.y;
      acc[cc][2] *= alpha.x;
      acc[cc][3] *= alpha.y;
    }
  }
  pv_q_mma<D, G, true, FULL>(vt, ps, acc, lane, nvalid);
}

}  // namespace pa
