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
// tensor cores (pv_f16) with the V scale folded into each softmax weight.
// (INT8 tensor-core MMAs do no more multiply-adds per cycle than dp4a on this
// GPU, measured, so QK stays on dp4a.)
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

// One m16n8k16 f16 tensor-core step, fp32 accumulate: c += a · b.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One m16n8k32 E4M3 tensor-core step, fp32 accumulate: c += a · b.
__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 4 E4M3 codes (one word, first code in the low byte) to two exact f16 pairs:
// codes 0, 1 -> lo, codes 2, 3 -> hi (the conversion reads each 16-bit half
// of the word directly).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two offset-binary INT8 V codes (bytes SEL picks: 0x4140 -> bytes 0, 1;
// 0x4342 -> bytes 2, 3 of w) to an exact f16 pair: the byte permute makes
// each byte b the mantissa of an f16 with the exponent of 1024 (the value
// 1024 + b), and subtracting 1152 leaves b - 128, the code.
template <unsigned SEL>
__device__ __forceinline__ uint32_t ob8x2_to_f16x2(uint32_t w) {
  const uint32_t x = __byte_perm(w, 0x64646464u, SEL);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x64806480u));
  return r;
}

// Two floats to an f16 pair (first in the low half), round to nearest even.
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
  __half2 v;
  v = *reinterpret_cast<const __half2*>(&h);
  return __half22float2(v);
}

// A pair of weights as an f16 hi part and an f16 lo part: hi = f16(u),
// lo = f16(u - hi); their sum keeps ~22 significant bits of u (for u <= 2^8
// down to f16's subnormals, far below anything that matters next to 1).
__device__ __forceinline__ void split_f16x2(float u0, float u1, uint32_t& hi, uint32_t& lo) {
  hi = f16x2_rn(u0, u1);
  const float2 h = f16x2_to_float2(hi);
  lo = f16x2_rn(u0 - h.x, u1 - h.y);
}

// The N = 8 columns of the 1-byte decode's MMAs for a group of G heads.  G = 8:
// one head per column.  G <= 4: column n holds part n / G of head n % G (QK:
// the two E4M3 parts of q; PV: the hi and lo f16 parts of the weights; parts
// >= 2 are zero), so one MMA carries both parts and the lanes holding part 1
// mirror those holding part 0.  Lane tig's accumulator columns 2 tig, 2 tig + 1
// are heads head(2 tig), head(2 tig) + 1.
template <int G>
struct QCols {
  static constexpr bool PACKED = G < 8;
  static constexpr int NQ = PACKED ? 1 : 2;  // q fragment sets (G = 8: one per part)
  static __device__ __forceinline__ int head(int n) { return PACKED ? n % G : n; }
  static __device__ __forceinline__ int part(int n) { return PACKED ? n / G : 0; }
  // a lane whose accumulator columns hold part 0 (writes weights and results)
  static __device__ __forceinline__ bool part0(int tig) { return !PACKED || 2 * tig < G; }
};

// The lane's D / 8 words of a 1-byte V tile laid out as v_tile_pos (cache_row.cuh)
// states: word 2c is dim 16c + gid, word 2c + 1 dim 16c + gid + 8, each with the
// codes of tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9 in bytes 0..3.
template <int D>
__device__ __forceinline__ void load_v_words(const unsigned char* vt, int lane,
                                             uint32_t (&w)[D / 8]) {
  const int f = D == 128 ? ((lane >> 1) & 3) : ((lane >> 2) & 1);
  const unsigned char* base = vt + lane * (D / 2);
#pragma unroll
  for (int u = 0; u < D / 32; ++u) {
    const uint4 x = *reinterpret_cast<const uint4*>(base + 16 * (u ^ f));
    w[4 * u] = x.x;
    w[4 * u + 1] = x.y;
    w[4 * u + 2] = x.z;
    w[4 * u + 3] = x.w;
  }
}

// 2^x by the hardware's approximate exponential (relative error below
// 2^-22; results below 2^-126 flush to zero, and exp2(-inf) is 0).  The
// 1-byte decode's weights are relative to a reference at most 2^8 below the
// largest score, so nothing that matters is that small.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The 1-byte decode's softmax reference: it moves to the tile's maximum only
// when that exceeds it by more than 2^8 (base-2 units), so most tiles keep
// the reference and skip rescaling their accumulators.  Weights exp2(s - m)
// are then at most 2^8 (times V scale / bound: still far inside f16), and the
// (m, l) pairs a partition emits hold for any reference.  Starts from -inf.
__device__ __forceinline__ float lazy_max(float m_ref, float tile_max) {
  return tile_max > m_ref + 8.f ? tile_max : m_ref;
}

// The warp's power-of-two bound on the V scales it has weighted: the PV
// weights enter the MMA as p * v_scale / bound, at most 2^8 (lazy_max) and
// so safe in f16 whatever the scales are.  For a tile whose largest valid scale (vmax,
// warp-uniform) is above the bound, raises it to the next power of two and
// returns old / new (exact), the factor the accumulators take; else 1.
__device__ __forceinline__ float raise_v_bound(float vmax, float& bound, float& inv) {
  if (!(vmax > bound)) return 1.f;
  const float nb = __uint_as_float((__float_as_uint(vmax) + 0x007FFFFFu) & 0x7F800000u);
  const float r = bound / nb;
  bound = nb;
  inv = 1.0f / nb;
  return r;
}

// PV of one 1-byte tile on the tensor cores (f16 in, fp32 accumulate):
// out^T[dim][column] += V^T[dim][token] · W[token][column], m16n8k16 MMAs with
// M = 16 dims, N = the 8 QCols columns, K = the tile's 16 tokens.  V codes are
// exact in f16 (INT8 offset-binary through ob8x2_to_f16x2, E4M3 through the
// conversion instruction); each weight (ps: softmax weight times the token's V
// scale, [16 tokens][G], 0 past the context) times inv_s enters as an f16 hi
// and an f16 lo part (G <= 4: the two column halves of one MMA; G = 8: a
// second MMA).  Lane (gid, tig) feeds dims 16c + gid and 16c + gid + 8 of
// m-tile c; acc[c] holds (dim 16c + gid; columns 2 tig, 2 tig + 1) and (dim
// 16c + gid + 8; the same columns).  E4M3 codes of tokens past the context
// may be NaN and are zeroed (0 * NaN is not 0); INT8 codes are always finite.
template <int D, int G, bool F8, bool FULL>
__device__ __forceinline__ void pv_f16(const unsigned char* __restrict__ vt,
                                       const float* __restrict__ ps, float inv_s,
                                       float (&acc)[D / 16][4], int lane, int nvalid) {
  using C = QCols<G>;
  const int gid = lane >> 2, tig = lane & 3;
  const float* pc = ps + C::head(gid);
  uint32_t h0, l0, h1, l1;
  split_f16x2(pc[(2 * tig) * G] * inv_s, pc[(2 * tig + 1) * G] * inv_s, h0, l0);
  split_f16x2(pc[(2 * tig + 8) * G] * inv_s, pc[(2 * tig + 9) * G] * inv_s, h1, l1);
  uint32_t b0 = h0, b1 = h1;  // G = 8: the hi parts here, the lo parts by a second MMA
  if constexpr (C::PACKED) {
    const int pn = C::part(gid);
    b0 = pn == 0 ? h0 : (pn == 1 ? l0 : 0u);
    b1 = pn == 0 ? h1 : (pn == 1 ? l1 : 0u);
  }
  uint32_t w[D / 8];
  load_v_words<D>(vt, lane, w);
  if constexpr (F8 && !FULL) {
    const uint32_t keep = (2 * tig < nvalid ? 0x000000FFu : 0u) |
                          (2 * tig + 1 < nvalid ? 0x0000FF00u : 0u) |
                          (2 * tig + 8 < nvalid ? 0x00FF0000u : 0u) |
                          (2 * tig + 9 < nvalid ? 0xFF000000u : 0u);
#pragma unroll
    for (int j = 0; j < D / 8; ++j) w[j] &= keep;
  }
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    uint32_t a0, a1, a2, a3;
    if constexpr (F8) {
      e4m3x4_to_f16x2x2(w[2 * c], a0, a2);
      e4m3x4_to_f16x2x2(w[2 * c + 1], a1, a3);
    } else {
      a0 = ob8x2_to_f16x2<0x4140>(w[2 * c]);
      a2 = ob8x2_to_f16x2<0x4342>(w[2 * c]);
      a1 = ob8x2_to_f16x2<0x4140>(w[2 * c + 1]);
      a3 = ob8x2_to_f16x2<0x4342>(w[2 * c + 1]);
    }
    mma_f16(acc[c], a0, a1, a2, a3, b0, b1);
    if constexpr (!C::PACKED) mma_f16(acc[c], a0, a1, a2, a3, l0, l1);
  }
}

// Multiplies the PV accumulators of columns 2 tig (fa) and 2 tig + 1 (fb).
template <int D>
__device__ __forceinline__ void scale_acc(float (&acc)[D / 16][4], float fa, float fb) {
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    acc[c][0] *= fa;
    acc[c][1] *= fb;
    acc[c][2] *= fa;
    acc[c][3] *= fb;
  }
}

// One INT8 tile.  (qsub, qrg): this lane in the QK geometry; my_head / my_i0:
// the head and first pass of this lane's scores.  vbound / vinv: the warp's
// V-scale bound (raise_v_bound) and its reciprocal.
template <int D, int G, bool FULL>
__device__ __forceinline__ void tile_step_i8(const unsigned char* __restrict__ kt,
                                             const unsigned char* __restrict__ vt,
                                             const float* __restrict__ ksc,
                                             const float* __restrict__ vsc, float* ps,
                                             float* alpha_s,
                                             const int (&qc)[G][I8Geometry<D, G>::QW],
                                             const float (&qsc)[G], float (&acc)[D / 16][4],
                                             float& m_run, float& l_run, float& vbound,
                                             float& vinv, int nvalid, int lane, int qsub, int qrg,
                                             int my_head, int my_i0) {
  using IG = I8Geometry<D, G>;
  using C = QCols<G>;
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
  const float m_new = lazy_max(m_run, mx);
  const float alpha = ex2_fast(m_run - m_new);
  float psum = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int t = (my_i0 + r) * QR + qrg;
    const float pr = ex2_fast(s[r] - m_new);
    psum += pr;
    // V scale folded in; a token past the context gets weight 0 (its codes
    // are finite whatever the pool holds, its scale may not be)
    ps[t * G + my_head] = pr * ((FULL || t < nvalid) ? vsc[t] : 0.f);
  }
  l_run = l_run * alpha + psum;
  m_run = m_new;
  if (qsub % IG::HEAD_LANES == 0 && qrg == 0) alpha_s[my_head] = alpha;
  // the tile's largest valid V scale, against the warp's bound (reduced only
  // when some lane sees a scale above it)
  float vm = (FULL || (lane & 15) < nvalid) ? vsc[lane & 15] : 0.f;
  float r = 1.f;
  if (__any_sync(kFullMask, vm > vbound)) {
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) vm = fmaxf(vm, __shfl_xor_sync(kFullMask, vm, m));
    r = raise_v_bound(vm, vbound, vinv);
  }
  const bool rescale = __any_sync(kFullMask, alpha != 1.0f) || r != 1.0f;
  __syncwarp();

  if (rescale) {
    const int ha = C::head(2 * (lane & 3));
    scale_acc<D>(acc, alpha_s[ha] * r, alpha_s[ha + 1] * r);
  }
  pv_f16<D, G, false, FULL>(vt, ps, vinv, acc, lane, nvalid);
}

// One FP8 (E4M3) tile.  QK on the tensor cores in E4M3: S[token][column] =
// K · q^T with m16n8k32 MMAs (M = the tile's 16 tokens, N = the QCols columns,
// K = 32 dims a step), q entering as two E4M3 parts whose sum is q times a
// power of two per head (the kernel's prologue builds qb; the codes need no
// conversion; the second part is scaled by 2^5 and counts 2^-5).  Lane (gid,
// tig) feeds tokens gid and gid + 8 with the D / 4
// code bytes at dims [(D/4) tig, +D/4) of each: a step's k indices 4 tig..+3
// and 16 + 4 tig..+3 are dims (D/4) tig + 8s + 0..3 and + 4..7, which are the
// dims of q's fragment for those k, so each dim reaches the MMA exactly once.
// The accumulator holds (token gid | gid + 8; column 2 tig | 2 tig + 1); the
// two parts of q are summed across lanes (G <= 4: lane tig ^ G / 2) or
// accumulators (G = 8).  The online softmax state (m_run, l_run) is that of
// heads head(2 tig), head(2 tig) + 1, the heads of the lane's PV columns, so
// the rescale stays in the lane; l_run is this lane's share, summed over gid
// at the end.  qfac: 2^-k * scale * log2 e of those two heads.
template <int D, int G, bool FULL>
__device__ __forceinline__ void tile_step_f8(const unsigned char* __restrict__ kt,
                                             const unsigned char* __restrict__ vt,
                                             const float* __restrict__ ksc,
                                             const float* __restrict__ vsc, float* ps,
                                             const uint32_t (&qb)[QCols<G>::NQ][D / 32][2],
                                             float2 qfac, float (&acc)[D / 16][4],
                                             float2& m_run, float2& l_run, float& vbound,
                                             float& vinv, int nvalid, int lane) {
  using C = QCols<G>;
  constexpr int KB = D / 4;  // code bytes per lane and row
  constexpr int KS = D / 32; // MMA steps
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t k0[KB / 4], k1[KB / 4];  // codes of tokens gid and gid + 8
  {
    const unsigned char* r0 = kt + gid * D + KB * tig;
    const unsigned char* r1 = r0 + 8 * D;
#pragma unroll
    for (int u = 0; u < KB / 16; ++u) {
      const uint4 x = *reinterpret_cast<const uint4*>(r0 + 16 * u);
      const uint4 y = *reinterpret_cast<const uint4*>(r1 + 16 * u);
      k0[4 * u] = x.x; k0[4 * u + 1] = x.y; k0[4 * u + 2] = x.z; k0[4 * u + 3] = x.w;
      k1[4 * u] = y.x; k1[4 * u + 1] = y.y; k1[4 * u + 2] = y.z; k1[4 * u + 3] = y.w;
    }
  }
  float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int st = 0; st < KS; ++st) {
    if constexpr (C::PACKED) {  // two independent chains, summed below
      mma_e4m3(c[st & 1], k0[2 * st], k1[2 * st], k0[2 * st + 1], k1[2 * st + 1], qb[0][st][0],
               qb[0][st][1]);
    } else {  // one chain per part of q
      mma_e4m3(c[0], k0[2 * st], k1[2 * st], k0[2 * st + 1], k1[2 * st + 1], qb[0][st][0],
               qb[0][st][1]);
      mma_e4m3(c[1], k0[2 * st], k1[2 * st], k0[2 * st + 1], k1[2 * st + 1], qb[1][st][0],
               qb[1][st][1]);
    }
  }
  // q = q1 + 2^-5 q2: part 1 counts 2^-5
  float sc[4];
  if constexpr (C::PACKED) {
    const float w = C::part(2 * tig) == 1 ? 0.03125f : 1.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sc[i] = (c[0][i] + c[1][i]) * w;
      sc[i] += __shfl_xor_sync(kFullMask, sc[i], G / 2);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] = fmaf(c[1][i], 0.03125f, c[0][i]);
  }

  // scores in base-2 units; a token past the context is masked by position
  // (its codes and scale may be anything, NaN included)
  const bool ok0 = FULL || gid < nvalid, ok1 = FULL || gid + 8 < nvalid;
  const float ks0 = ok0 ? ksc[gid] : 0.f, ks1 = ok1 ? ksc[gid + 8] : 0.f;
  float s[4];
  s[0] = ok0 ? sc[0] * ks0 * qfac.x : -INFINITY;
  s[1] = ok0 ? sc[1] * ks0 * qfac.y : -INFINITY;
  s[2] = ok1 ? sc[2] * ks1 * qfac.x : -INFINITY;
  s[3] = ok1 ? sc[3] * ks1 * qfac.y : -INFINITY;
  float2 mx = make_float2(fmaxf(s[0], s[2]), fmaxf(s[1], s[3]));
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    mx.x = fmaxf(mx.x, __shfl_xor_sync(kFullMask, mx.x, m));
    mx.y = fmaxf(mx.y, __shfl_xor_sync(kFullMask, mx.y, m));
  }
  const float2 m_new = make_float2(lazy_max(m_run.x, mx.x), lazy_max(m_run.y, mx.y));
  const float2 alpha = make_float2(ex2_fast(m_run.x - m_new.x), ex2_fast(m_run.y - m_new.y));
  const float p0 = ex2_fast(s[0] - m_new.x), p1 = ex2_fast(s[1] - m_new.y);
  const float p2 = ex2_fast(s[2] - m_new.x), p3 = ex2_fast(s[3] - m_new.y);
  l_run = make_float2(l_run.x * alpha.x + (p0 + p2), l_run.y * alpha.y + (p1 + p3));
  m_run = m_new;
  // the tile's largest valid V scale, against the warp's bound (reduced only
  // when some lane sees a scale above it)
  const float v0 = ok0 ? vsc[gid] : 0.f, v1 = ok1 ? vsc[gid + 8] : 0.f;
  float vm = fmaxf(v0, v1);
  float r = 1.f;
  if (__any_sync(kFullMask, vm > vbound)) {
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) vm = fmaxf(vm, __shfl_xor_sync(kFullMask, vm, m));
    r = raise_v_bound(vm, vbound, vinv);
  }
  // weights with the V scale folded in (0 past the context), written once per
  // (token, head) by the lanes holding part 0
  if (C::part0(tig)) {
    const int ha = C::head(2 * tig);
    ps[gid * G + ha] = p0 * v0;
    ps[gid * G + ha + 1] = p1 * v0;
    ps[(gid + 8) * G + ha] = p2 * v1;
    ps[(gid + 8) * G + ha + 1] = p3 * v1;
  }
  const float fa = alpha.x * r, fb = alpha.y * r;
  const bool rescale = __any_sync(kFullMask, fa != 1.0f || fb != 1.0f);
  __syncwarp();
  if (rescale) scale_acc<D>(acc, fa, fb);
  pv_f16<D, G, true, FULL>(vt, ps, vinv, acc, lane, nvalid);
}

}  // namespace pa
