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
// 1-byte KV caches (INT8, FP8; one fp32 scale per token and KV head).  A
// tile is K codes [16][D] (row-major), V codes [16 * D] (transposed,
// v_tile_pos), then the 16 K and 16 V scales.
//
// The 1-byte caches (INT8, FP8): QK and PV both on the tensor cores
// (mma.sync), the softmax weights never leaving registers.
//
// QK is computed transposed, S^T = q . K^T: the MMA's rows are the group's
// query heads (and, for FP8, the two parts of q), its N = 8 columns are 8 of
// the tile's 16 tokens (two MMA chains: tokens 0..7 and 8..15) and its K
// dimension is the head dimension.  The accumulator fragment a lane receives,
// (row gid; tokens 2 tig, 2 tig + 1), is then exactly the lane's share of
// the B operand of the PV MMA (out^T = V^T . W: K = tokens 2 tig, 2 tig + 1,
// 2 tig + 8, 2 tig + 9; N = column gid), so the weights go from the
// exponential into the PV MMA without a shared-memory round trip.
//
// Columns of the PV MMA (QCols): G = 8: one head per column, the weights'
// hi and lo f16 parts in two MMAs; G <= 4: column n holds part n / G of
// head n % G (hi, lo, then zeros), one MMA.  Lane gid computes the scores of
// head(gid) (rows gid and gid + 8 of the QK MMA both belong to it), so the
// lanes of one head's hi and lo columns compute the same scores; the
// softmax maximum is taken over all of them, so they also share one
// reference.

// The N = 8 columns of the 1-byte decode's PV MMAs for a group of G heads.
template <int G>
struct QCols {
  static constexpr bool PACKED = G < 8;
  static __device__ __forceinline__ int head(int n) { return PACKED ? n % G : n; }
  static __device__ __forceinline__ int part(int n) { return PACKED ? n / G : 0; }
  // a lane whose PV accumulator columns 2 tig, 2 tig + 1 hold part 0
  static __device__ __forceinline__ bool part0(int tig) { return !PACKED || 2 * tig < G; }
};

// One m16n8k16 f16 tensor-core step, fp32 accumulate: c += a . b.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One m16n8k32 E4M3 tensor-core step, fp32 accumulate: c += a . b.
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

// Two offset-binary INT8 codes (bytes SEL picks: 0x4140 -> bytes 0, 1;
// 0x4342 -> bytes 2, 3 of w) to an exact f16 pair: the byte permute makes
// each byte b the mantissa of an f16 with the exponent of 1024 (the value
// 1024 + b), and subtracting 1152 leaves b - 128, the code.  Signed codes
// enter with their sign bits flipped (x ^ 0x80 = code + 128).
template <unsigned SEL>
__device__ __forceinline__ uint32_t ob8x2_to_f16x2(uint32_t w) {
  const uint32_t x = __byte_perm(w, 0x64646464u, SEL);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x64806480u));
  return r;
}

// Two bytes (SEL as for ob8x2_to_f16x2) to an f16 pair holding them as
// subnormals: byte b becomes b * 2^-24 exactly (the byte is the f16's
// mantissa, its exponent field zero).  The 1-byte decode feeds INT8 codes to
// the f16 MMAs this way, offset by 128 (code + 128 in [1, 255]), and removes
// the offset from the sums: one byte permute per pair, no arithmetic.
template <unsigned SEL>
__device__ __forceinline__ uint32_t u8x2_to_f16x2_sub(uint32_t w) {
  return __byte_perm(w, 0u, SEL);
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

// The lane's words of q for the QK MMAs (D / 8 of them, both caches), built
// once per CTA.  Lane (gid, tig) holds rows gid and gid + 8 of the A operand,
// both for head(gid), over the dims [(D/4) tig, +D/4), the same dims whose K
// codes it feeds as the B operand:
//  * FP8 (m16n8k32 E4M3, D / 32 steps): q times a power of two per head is
//    split into two exact E4M3 parts, x = q1 + 2^-5 q2; row gid is q1, row
//    gid + 8 is q2.  Step s: words 4s, 4s + 2 = q1 at dims (D/4) tig + 8s +
//    0..3 and + 4..7 (the MMA's k = 4 tig + 0..3 and 16 + 4 tig + 0..3), words
//    4s + 1, 4s + 3 = q2 at the same dims.
//  * INT8 (m16n8k16 f16, D / 16 steps): q's int8 codes as exact f16; row
//    gid + 8 is zero.  Step s: word 2s = dims (D/4) tig + 4s + 0, 1 (k = 2 tig,
//    2 tig + 1), word 2s + 1 = dims + 2, 3 (k = 2 tig + 8, 2 tig + 9).
// The lane's K words (load_k_words) cover the same dims in the same order.

// The K codes lane (gid, tig) feeds to the QK MMAs: tokens gid (k0) and
// gid + 8 (k1), the D / 4 bytes at dims [(D/4) tig, +D/4) of each.
template <int D>
__device__ __forceinline__ void load_k_words(const unsigned char* kt, int lane,
                                             uint32_t (&k0)[D / 16], uint32_t (&k1)[D / 16]) {
  constexpr int KB = D / 4;
  const int gid = lane >> 2, tig = lane & 3;
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

// One 1-byte tile (F8: E4M3 codes; else INT8).  qa / qf: the lane's q words
// (above) and its head's score factor (FP8: 2^-k * scale * log2 e; INT8: q's
// scale * scale * log2 e).  m_run / l_run: the online softmax state of
// head(gid), l_run this lane's share (its 4 tokens of every tile).  acc:
// out^T[dim][column] in units of vbound, the warp's V-scale bound
// (raise_v_bound; vinv its reciprocal): (dim 16c + gid; columns 2 tig,
// 2 tig + 1) and (dim 16c + gid + 8; the same columns).
//
// INT8 codes enter the MMAs as subnormal f16s of code + 128
// (u8x2_to_f16x2_sub): K codes with their sign bits flipped, V codes as
// stored (offset binary).  So the QK accumulator is 2^-24 (q . k + 128 sum(q))
// and each dot is recovered exactly as 2^24 acc - qoff (qoff = 128 sum(q),
// the lane's head; every term is an integer below 2^24); and the PV
// accumulators hold 2^-24 (sum w v + 128 sum w), the offset removed once at
// the end with wsum, this lane's share of its column's weights (part-0 rows
// only; rescaled with the accumulators).
template <int D, int G, bool F8, bool FULL>
__device__ __forceinline__ void tile_step_1b(const unsigned char* __restrict__ kt,
                                             const unsigned char* __restrict__ vt,
                                             const float* __restrict__ ksc,
                                             const float* __restrict__ vsc,
                                             const uint32_t (&qa)[D / 8], float qf, float qoff,
                                             float (&acc)[D / 16][4], float& m_run,
                                             float& l_run, float& wsum, float& vbound,
                                             float& vinv, int nvalid, int lane) {
  using C = QCols<G>;
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t k0[D / 16], k1[D / 16];
  load_k_words<D>(kt, lane, k0, k1);

  // S^T: ca = tokens 0..7, cb = tokens 8..15; the lane receives rows gid
  // (c[0], c[1]) and gid + 8 (c[2], c[3]) at tokens 2 tig, 2 tig + 1 of each
  float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (F8) {
#pragma unroll
    for (int s = 0; s < D / 32; ++s) {
      mma_e4m3(ca, qa[4 * s], qa[4 * s + 1], qa[4 * s + 2], qa[4 * s + 3], k0[2 * s],
               k0[2 * s + 1]);
      mma_e4m3(cb, qa[4 * s], qa[4 * s + 1], qa[4 * s + 2], qa[4 * s + 3], k1[2 * s],
               k1[2 * s + 1]);
    }
  } else {
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      const uint32_t x0 = k0[s] ^ 0x80808080u, x1 = k1[s] ^ 0x80808080u;
      mma_f16(ca, qa[2 * s], 0u, qa[2 * s + 1], 0u, u8x2_to_f16x2_sub<0x4140>(x0),
              u8x2_to_f16x2_sub<0x4342>(x0));
      mma_f16(cb, qa[2 * s], 0u, qa[2 * s + 1], 0u, u8x2_to_f16x2_sub<0x4140>(x1),
              u8x2_to_f16x2_sub<0x4342>(x1));
    }
  }
  // head(gid)'s dot products with tokens t0, t0 + 1, t0 + 8, t0 + 9 (FP8:
  // q1's plus 2^-5 q2's; INT8: exact integers)
  float d0, d1, d2, d3;
  if constexpr (F8) {
    d0 = fmaf(ca[2], 0.03125f, ca[0]);
    d1 = fmaf(ca[3], 0.03125f, ca[1]);
    d2 = fmaf(cb[2], 0.03125f, cb[0]);
    d3 = fmaf(cb[3], 0.03125f, cb[1]);
  } else {
    d0 = fmaf(ca[0], 0x1p24f, -qoff);
    d1 = fmaf(ca[1], 0x1p24f, -qoff);
    d2 = fmaf(cb[0], 0x1p24f, -qoff);
    d3 = fmaf(cb[1], 0x1p24f, -qoff);
  }
  const int t0 = 2 * tig;
  const float2 ka = *reinterpret_cast<const float2*>(ksc + t0);
  const float2 kb = *reinterpret_cast<const float2*>(ksc + t0 + 8);
  float2 va = *reinterpret_cast<const float2*>(vsc + t0);
  float2 vb = *reinterpret_cast<const float2*>(vsc + t0 + 8);
  // scores in base-2 units; a token past the context is masked by position
  // (its codes and scales may be anything, NaN included) and weighs 0
  float s0 = d0 * (qf * ka.x), s1 = d1 * (qf * ka.y);
  float s2 = d2 * (qf * kb.x), s3 = d3 * (qf * kb.y);
  if constexpr (!FULL) {
    if (!(t0 < nvalid)) { s0 = -INFINITY; va.x = 0.f; }
    if (!(t0 + 1 < nvalid)) { s1 = -INFINITY; va.y = 0.f; }
    if (!(t0 + 8 < nvalid)) { s2 = -INFINITY; vb.x = 0.f; }
    if (!(t0 + 9 < nvalid)) { s3 = -INFINITY; vb.y = 0.f; }
  }
  // the tile's maximum for head(gid): over the 4 lanes of the row, then over
  // the rows of the same head (G <= 4)
  float mx = fmaxf(fmaxf(s0, s1), fmaxf(s2, s3));
  mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2));
#pragma unroll
  for (int m = 4 * G; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
  const float m_new = lazy_max(m_run, mx);
  const float alpha = ex2_fast(m_run - m_new);
  const float p0 = ex2_fast(s0 - m_new), p1 = ex2_fast(s1 - m_new);
  const float p2 = ex2_fast(s2 - m_new), p3 = ex2_fast(s3 - m_new);
  l_run = fmaf(l_run, alpha, (p0 + p1) + (p2 + p3));
  m_run = m_new;
  // the tile's largest valid V scale, against the warp's bound (reduced only
  // when some lane sees a scale above it; every row sees all 16 tokens)
  float vm = fmaxf(fmaxf(va.x, va.y), fmaxf(vb.x, vb.y));
  float r = 1.f;
  if (__any_sync(kFullMask, vm > vbound)) {
    vm = fmaxf(vm, __shfl_xor_sync(kFullMask, vm, 1));
    vm = fmaxf(vm, __shfl_xor_sync(kFullMask, vm, 2));
    r = raise_v_bound(vm, vbound, vinv);
  }
  // this lane's PV column gid: the weights p * v_scale / bound of head(gid),
  // as their f16 hi part, their lo part, or zeros (G <= 4, parts >= 2)
  const float wm = (C::PACKED && C::part(gid) >= 2) ? 0.f : vinv;
  const float u0 = p0 * (va.x * wm), u1 = p1 * (va.y * wm);
  const float u2 = p2 * (vb.x * wm), u3 = p3 * (vb.y * wm);
  uint32_t h01, l01, h23, l23;
  split_f16x2(u0, u1, h01, l01);
  split_f16x2(u2, u3, h23, l23);
  if constexpr (!F8)  // the weights this column's rows take (hi + lo = u), on the part-0 rows
    wsum = fmaf(wsum, alpha * r, C::part(gid) == 0 ? (u0 + u1) + (u2 + u3) : 0.f);
  uint32_t b0 = h01, b1 = h23;
  if constexpr (C::PACKED) {
    if (C::part(gid) == 1) {
      b0 = l01;
      b1 = l23;
    }
  }
  // rescale the accumulators to the new reference and bound: columns 2 tig
  // and 2 tig + 1 take the factors of the lanes computing them (rows 2 tig
  // and 2 tig + 1)
  if (__any_sync(kFullMask, alpha != 1.0f) || r != 1.0f) {
    const float fa = __shfl_sync(kFullMask, alpha, 8 * tig) * r;
    const float fb = __shfl_sync(kFullMask, alpha, 8 * tig + 4) * r;
    scale_acc<D>(acc, fa, fb);
  }

  // PV: out^T[dim][column] += V^T[dim][token] . W[token][column], m16n8k16
  // f16 MMAs with M = 16 dims, N = 8 columns, K = the tile's 16 tokens.  V
  // codes are exact in f16 (INT8 as offset subnormals, E4M3 through the
  // conversion instruction).  E4M3 codes of tokens past the context may be
  // NaN and are zeroed (0 * NaN is not 0); INT8 codes are always finite.
  uint32_t w[D / 8];
  load_v_words<D>(vt, lane, w);
  if constexpr (F8 && !FULL) {
    const uint32_t keep = (t0 < nvalid ? 0x000000FFu : 0u) |
                          (t0 + 1 < nvalid ? 0x0000FF00u : 0u) |
                          (t0 + 8 < nvalid ? 0x00FF0000u : 0u) |
                          (t0 + 9 < nvalid ? 0xFF000000u : 0u);
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
      a0 = u8x2_to_f16x2_sub<0x4140>(w[2 * c]);
      a2 = u8x2_to_f16x2_sub<0x4342>(w[2 * c]);
      a1 = u8x2_to_f16x2_sub<0x4140>(w[2 * c + 1]);
      a3 = u8x2_to_f16x2_sub<0x4342>(w[2 * c + 1]);
    }
    mma_f16(acc[c], a0, a1, a2, a3, b0, b1);
    if constexpr (!C::PACKED) mma_f16(acc[c], a0, a1, a2, a3, l01, l23);
  }
}

}  // namespace pa
