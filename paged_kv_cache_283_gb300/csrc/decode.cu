// Paged decode attention (plain and split-K) and the split-K merge, sm_103a.
//
// What is computed: "How LLM Inference Serving Works" (dev.to), sections
// "What the KV Cache Is, and How Big It Gets" (the new token's query against
// every cached key, a softmax-weighted mix of the cached values; 32 query
// heads share 8 KV heads) and "PagedAttention: Virtual Memory for the KV
// Cache" (the kernel follows the block table to wherever each block lives).
// Decode is memory-bound ("Two Phases: Prefill and Decode"), so the design
// is about moving each K/V byte from HBM exactly once at full bandwidth:
//
//  * One CTA per (sequence, KV head[, partition]).  All G query heads of the
//    group are evaluated against each K/V block while it sits in shared
//    memory, so the block is read from HBM once, not G times.
//  * Pool layout [num_blocks, Hkv, 16, D] makes one (block, head) tile a
//    contiguous 16*D*2-byte run (4 KiB at D = 128).  Each warp runs its own
//    S-stage ring of such tiles, filled by single-instruction bulk async
//    copies (cp.async.bulk, completion counted on an mbarrier) with an
//    evict-first L2 policy; the warps of a CTA take the sequence's blocks
//    round-robin and never wait on one another until the final merge.
//  * Compute is CUDA-core fp32 (packed f32x2 FMAs): lane (row group rg, sub
//    s) owns dims [8s, 8s+8) of tokens rg, rg+ROWS, ...  QK partial dots are
//    finished by a transposing butterfly (each level halves the values a
//    lane holds), which leaves every lane with R complete scores of one
//    head; the softmax is online per warp in base-2 units (q is pre-scaled
//    by scale*log2 e); P is handed to the PV loop through a 256-byte smem
//    buffer; warps merge (m, l, acc) through shared memory at the end.
//  * Split-K writes per-partition (m, l, o/l) in fp32, merged by the
//    log-sum-exp identity either by a second small kernel (splitk_reduce.cu,
//    pa_decode_splitk + pa_splitk_reduce) or, in the fused decode step with
//    at most 16 partitions per sequence, inside the same launch by the last
//    CTA of each (sequence, KV head) to finish.
//  * Every device-resident index is checked: bad block ids read block 0 and
//    set PA_DEVERR_BLOCK_ID; bad context lengths are clamped; every mbarrier
//    wait is bounded.  Nothing traps.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "cache_row.cuh"
#include "decode_tile.cuh"
#include "device.cuh"
#include "internal.h"

namespace pa {

namespace {

constexpr float kLn2 = 0.6931471805599453f;

// Pipeline shape: warps per CTA and stages per warp (each stage holds one K
// and one V tile), per head_dim and per kernel (whole sequence vs split-K
// partition).  Chosen by measurement on the batch-64 Llama-8B decode: 4 warps
// x 2 stages lets three split-K CTAs share an SM; whole-sequence CTAs do
// better with 8 warps x 2 stages, one long CTA per SM.  Overridable at compile
// time for tuning.
#ifndef PA_SPLIT_WARPS_D128
#define PA_SPLIT_WARPS_D128 4
#endif
#ifndef PA_SPLIT_STAGES_D128
#define PA_SPLIT_STAGES_D128 2
#endif
#ifndef PA_WHOLE_WARPS_D128
#define PA_WHOLE_WARPS_D128 8
#endif
#ifndef PA_WHOLE_STAGES_D128
#define PA_WHOLE_STAGES_D128 2
#endif
// MINB is the number of CTAs meant to share an SM, handed to the register
// allocator through __launch_bounds__.
template <int D, bool SPLIT, int Q>
struct Pipe {  // head_dim 64: 2 KiB tiles, deeper rings
  static constexpr int NW = 4;
  static constexpr int S = Q != 0 ? 6 : 4;
};
template <bool SPLIT, int Q>
struct Pipe<128, SPLIT, Q> {
  static constexpr int NW = SPLIT ? PA_SPLIT_WARPS_D128 : PA_WHOLE_WARPS_D128;
  static constexpr int S = Q == 1 ? 3 : Q == 2 ? 2 : (SPLIT ? PA_SPLIT_STAGES_D128 : PA_WHOLE_STAGES_D128);
};
// Small bf16 CTAs share an SM three at a time (<= 168 registers); groups of 8
// heads need more registers than that and get one CTA's worth.  The 1-byte
// kernels need fewer registers and more warps to hide their latencies: four
// 4-warp INT8 CTAs per SM (<= 128 registers, 3 stages of 4.2 KiB per warp at
// head_dim 128), five FP8 ones (<= 102 registers, 2 stages: measured faster
// than 4 x 3 on the batch-64 and 32-layer steps; INT8 spills at that budget);
// 8-warp CTAs two per SM.
template <int NW, int G, int Q>
constexpr int min_blocks() {
  if constexpr (Q != 0) return NW <= 4 ? (G <= 4 ? (Q == 2 ? 5 : 4) : 3) : 2;
  else return (NW <= 4 && G <= 4) ? 3 : 1;  // bf16
}

template <int D, int G, int NW, int S, bool I8>
struct SmemLayout {
  using Geo = Geometry<D, G>;
  // one stage: K tile, V tile (bf16, or int8 codes followed by 16 K and 16 V scales)
  static constexpr int KT = I8 ? Geo::BS * D : Geo::TILE;      // bytes of one K (or V) tile
  static constexpr int STAGE = I8 ? 2 * KT + 2 * Geo::BS * 4 : 2 * KT;
  static constexpr int TILES = S * STAGE;
  // bf16: softmax weights of one tile and the heads' rescale factors (the
  // 1-byte caches keep both in registers)
  static constexpr int PS = I8 ? 0 : Geo::BS * G * 4;
  static constexpr int ALPHA = I8 ? 0 : ((G * 4 + 15) / 16) * 16;
  static constexpr int BARS = S * 8;
  static constexpr int MERGE = (G * D + 2 * G) * 4;  // aliases TILES after the loop
  static constexpr int WARP = ((TILES + PS + ALPHA + BARS + 127) / 128) * 128;
  // 1-byte caches: the int8 cache's quantised q, codes [G][D] then scales
  // [G] (the fp8 cache's warps each build their own q words)
  static constexpr int QOFF = NW * WARP;
  static constexpr int QI8 = ((G * D + G * 4 + 127) / 128) * 128;
  static constexpr int QREG = I8 ? QI8 : 0;
  // fused decode step: the new row staged for the patch (bf16: K and V rows;
  // 1-byte: K codes, V codes, the two scales)
  static constexpr int PATCHOFF = QOFF + QREG;
  static constexpr int PATCH = 4 * D + 32;
  static constexpr int TOTAL = PATCHOFF + PATCH;
  static_assert(MERGE <= TILES, "merge area must fit in the tile ring");
  static_assert(STAGE % 16 == 0 && KT % 16 == 0, "bulk copy sizes");
};
// Fused decode step: the new token of sequence b (position ctx - 1) goes to
// its slot, K and V rows of KV head kvh.  Called by the one warp that will
// read that position (the warp owning the sequence's last block, in the CTA
// whose range holds it).  The rows go to the pool with plain stores, and a
// copy of them (for the 1-byte caches: the codes and scales as stored) goes
// to `stage` in shared memory: the warp patches them into its tile once the
// tile's own copy of that block has landed, so nothing waits for the stores
// (the copy may read the old or the new row; either is overwritten).  The
// slot must be the one the block table gives for that position, since any
// other slot could be read by another CTA while it is written: otherwise
// nothing is written and PA_DEVERR_SLOT is raised.  Negative slots are
// padding.  Returns whether the row was written (then the tile needs the
// patch).  The pools are held const in the parameters for the readers; this
// is their one writer.
template <int D, int Q>
__device__ __forceinline__ bool fused_cache_write(const DecodeParams& p, int b, int kvh, int ctx,
                                                  const int32_t* tbl, int lane,
                                                  unsigned char* stage) {
  const int64_t slot = __ldg(p.slot_mapping + b);
  const size_t src = (static_cast<size_t>(b) * p.num_kv_heads + kvh) * D;
  constexpr int C = D / 8;  // 16-byte chunks of a bf16 row
  uint4 x = make_uint4(0, 0, 0, 0);
  uint32_t kw[D / 64], vw[D / 64];
  if constexpr (Q == 0) {  // lanes [0, C) hold K chunks, [C, 2C) V chunks
    if (lane < 2 * C)
      x = __ldg(reinterpret_cast<const uint4*>((lane >= C ? p.new_value : p.new_key) + src) +
                (lane % C));
  } else {
    load_row_words<D>(p.new_key + src, lane, kw);
    load_row_words<D>(p.new_value + src, lane, vw);
  }
  if (slot < 0) return false;
  int64_t want = -1;
  if (ctx >= 1) {
    const int id = __ldg(tbl + (ctx - 1) / kBlockSize);
    if (id >= 0 && id < p.num_blocks)
      want = static_cast<int64_t>(id) * kBlockSize + (ctx - 1) % kBlockSize;
  }
  if (slot != want) {
    if (lane == 0) raise_error(p.err, PA_DEVERR_SLOT);
    return false;
  }
  const int off = static_cast<int>(slot % kBlockSize);
  const int64_t srow = ((slot / kBlockSize) * p.num_kv_heads + kvh) * kBlockSize + off;
  if constexpr (Q == 0) {
    if (lane < 2 * C) {
      __nv_bfloat16* dst =
          const_cast<__nv_bfloat16*>(lane >= C ? p.v_cache : p.k_cache) + srow * D;
      reinterpret_cast<uint4*>(dst)[lane % C] = x;
      reinterpret_cast<uint4*>(stage)[lane] = x;  // [K row | V row]
    }
  } else {
    constexpr int PER = D / 32;
    float ks, vs;
    const uint32_t kc = quantise_row<D, Q == 2>(kw, &ks);
    const uint32_t vc = v_stored<Q == 2>(quantise_row<D, Q == 2>(vw, &vs));
    int8_t* k8 = const_cast<int8_t*>(p.k8) + srow * D;
    store_v_row_bytes<D>(const_cast<int8_t*>(p.v8) + (srow - off) * D, off, lane, vc);
    if constexpr (PER == 4) {
      *reinterpret_cast<uint32_t*>(k8 + lane * PER) = kc;
      *reinterpret_cast<uint32_t*>(stage + lane * PER) = kc;      // K codes
      *reinterpret_cast<uint32_t*>(stage + D + lane * PER) = vc;  // V bytes, logical dim order
    } else {
      *reinterpret_cast<uint16_t*>(k8 + lane * PER) = static_cast<uint16_t>(kc);
      *reinterpret_cast<uint16_t*>(stage + lane * PER) = static_cast<uint16_t>(kc);
      *reinterpret_cast<uint16_t*>(stage + D + lane * PER) = static_cast<uint16_t>(vc);
    }
    if (lane == 0) {
      const_cast<float*>(p.k_scales)[srow] = ks;
      const_cast<float*>(p.v_scales)[srow] = vs;
      reinterpret_cast<float*>(stage + 2 * D)[0] = ks;
      reinterpret_cast<float*>(stage + 2 * D)[1] = vs;
    }
  }
  return true;
}

// Patches the staged new row (fused_cache_write) into row `off` of a landed
// tile: K tile, V tile, and for the 1-byte caches the two scales.  The stage
// holds the 1-byte V bytes (as stored) in logical dim order; the tile holds
// them transposed.
template <int D, int Q>
__device__ __forceinline__ void patch_tile(unsigned char* tile, int kt_bytes,
                                           const unsigned char* stage, int off, int lane) {
  if constexpr (Q == 0) {
    constexpr int C = D / 8;
    if (lane < 2 * C)
      reinterpret_cast<uint4*>(tile + (lane >= C ? kt_bytes : 0) + off * D * 2)[lane % C] =
          reinterpret_cast<const uint4*>(stage)[lane];
  } else {
    constexpr int PER = D / 32;
    // the lane's PER codes of the K row, and its V bytes at their places in
    // the transposed V tile
    if constexpr (PER == 4) {
      *reinterpret_cast<uint32_t*>(tile + off * D + lane * PER) =
          *reinterpret_cast<const uint32_t*>(stage + lane * PER);
      store_v_row_bytes<D>(tile + kt_bytes, off, lane,
                           *reinterpret_cast<const uint32_t*>(stage + D + lane * PER));
    } else {
      *reinterpret_cast<uint16_t*>(tile + off * D + lane * PER) =
          *reinterpret_cast<const uint16_t*>(stage + lane * PER);
      store_v_row_bytes<D>(tile + kt_bytes, off, lane,
                           *reinterpret_cast<const uint16_t*>(stage + D + lane * PER));
    }
    if (lane == 0) {
      float* sc = reinterpret_cast<float*>(tile + 2 * kt_bytes);  // 16 K then 16 V scales
      sc[off] = reinterpret_cast<const float*>(stage + 2 * D)[0];
      sc[kBlockSize + off] = reinterpret_cast<const float*>(stage + 2 * D)[1];
    }
  }
}

// Q: the cache's element type: 0 = bf16, 1 = INT8, 2 = FP8 (E4M3).  INT8 and
// FP8 share the 1-byte-code tile layout (codes + per-token scales) and the
// tile step (tile_step_1b: QK and PV on the tensor cores, weights in
// registers); INT8 quantises q and its QK is exact in integers (f16 MMAs on
// the codes), FP8 takes QK in E4M3 on two exact parts of q.
template <int D, int G, int NW, int S, bool SPLIT, int Q>
__global__ void __launch_bounds__(NW * 32, (min_blocks<NW, G, Q>()))
    paged_decode_kernel(const DecodeParams p) {
  constexpr bool I8 = Q != 0;   // 1-byte codes + scales
  using Geo = Geometry<D, G>;
  using Lay = SmemLayout<D, G, NW, S, I8>;
  constexpr int BS = Geo::BS, L = Geo::L, P = Geo::P, R = Geo::R;
  extern __shared__ __align__(128) unsigned char smem[];

  // The previous kernel (e.g. the cache write) is complete after this wait.
  // With early reads (the caller's promise that tables, lengths, order and
  // pools are not written by it) the wait comes after the first copies are
  // out, and before anything else is read or anything is written.
  // After a shared prefix (first_partition > 0) the preceding kernel computes
  // the prefix's partitions and reads nothing this one writes, and its own
  // predecessor is complete once it runs: wait for it only before reading its
  // partitions (the merge) and before exiting.
  const bool after_prefix = SPLIT && p.first_partition > 0;
  if (!p.early_read && !after_prefix) griddep_wait();
  griddep_launch_dependents();
  const int kvh = blockIdx.x;
  // (sequence, partition): the grid's, or the order array's entry for this
  // CTA (its grid is then (Hkv, B * max_partitions, 1)); an entry out of
  // range is refused (the item it displaced does not run: the error says so)
  int b = blockIdx.y, part = blockIdx.z + (SPLIT ? p.first_partition : 0);
  if (SPLIT && p.order != nullptr) {  // (items over the partitions from first_partition)
    const int item = __ldg(p.order + blockIdx.y);
    if (item < 0 || item >= p.num_seqs * (p.max_partitions - p.first_partition)) {
      if (threadIdx.x == 0) raise_error(p.err, PA_DEVERR_ORDER);
      if (after_prefix) griddep_wait();
      return;
    }
    b = item % p.num_seqs;
    part = item / p.num_seqs + p.first_partition;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane % L;
  const int rg = lane / L;

  // The context length, this warp's first 32 block ids and q are independent
  // loads, so they go out together (q after the first copies with early
  // reads): the ids are read speculatively from the table slots this CTA may
  // use (in bounds whatever the context length is) and only those below the
  // context length are used, after a range check.
  // Split-K partitions: partition_blocks each from block 0, or after a shared
  // prefix, first_partition prefix partitions (another kernel's) and then
  // partition_blocks each from block prefix_blocks.
  auto part_start = [&](int pt) -> int64_t {
    return after_prefix ? p.prefix_blocks + static_cast<int64_t>(pt - p.first_partition) *
                                                p.partition_blocks
                        : static_cast<int64_t>(pt) * p.partition_blocks;
  };
  auto parts_of = [&](int n) -> int {  // partitions of a sequence of n blocks
    return after_prefix
               ? p.first_partition + max(0, (n - p.prefix_blocks + p.partition_blocks - 1) /
                                                p.partition_blocks)
               : (n + p.partition_blocks - 1) / p.partition_blocks;
  };
  const int64_t part_first = SPLIT ? part_start(part) : 0;
  const int tbl_end = SPLIT ? static_cast<int>(min(static_cast<int64_t>(p.max_blocks_per_seq),
                                                   part_first + p.partition_blocks))
                            : p.max_blocks_per_seq;
  const int32_t* tbl = p.block_tables + static_cast<size_t>(b) * p.max_blocks_per_seq;
  auto load_ids = [&](int win) -> int {
    const int64_t j = part_first + warp + static_cast<int64_t>(win * 32 + lane) * NW;
    return j < tbl_end ? __ldg(tbl + j) : 0;
  };
  int ctx = __ldg(p.context_lens + b);
  int ids_cur = load_ids(0);
  float2 q2[G][4];
  // 1-byte caches: the lane's q words for the QK MMAs and its head's score
  // factor (tile_step_1b)
  uint32_t qa[D / 8];
  float qf = 0.f;
  float qoff = 0.f;  // int8 cache: 128 * the sum of head(gid)'s q codes (tile_step_1b)
  // q of the group into this lane's registers (or, for the int8 cache,
  // quantised through shared memory): the inputs a preceding kernel may
  // still be writing, so with early reads this runs after the wait.
  auto load_q = [&]() {
    if constexpr (Q == 2) {
      // Every warp builds its own words (no barrier): lane (gid, tig) takes
      // head hn = head(gid), dims [(D/4) tig, +D/4).  The head's values times
      // 2^k, k chosen per head so that its largest |q| lands in [128, 256),
      // are split into two E4M3 parts, x = q1 + 2^-5 q2 with q1 = E4M3(x),
      // q2 = E4M3(32 (x - q1)): a bf16 value has 8 significant bits and q1
      // keeps 4 of them, and |x - q1| <= 8 (half a step of q1 below 256), so
      // 32 (x - q1) <= 256 is exact in q2 except where it falls below E4M3's
      // normal range: an error under 2^-14 absolute, about 2^-21 of the
      // head's largest |q|.
      using C = QCols<G>;
      constexpr int E = D / 4;
      const int gid = lane >> 2, tig = lane & 3;
      const int hn = C::head(gid);
      float f[E];
      const __nv_bfloat16* qh =
          p.q + (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(kvh) * G + hn) * D +
          E * tig;
  #pragma unroll
      for (int u = 0; u < E / 8; ++u) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(qh) + u);
        const float2 a = bf16x2_to_float2(w.x), c = bf16x2_to_float2(w.y);
        const float2 d = bf16x2_to_float2(w.z), e = bf16x2_to_float2(w.w);
        f[8 * u] = a.x; f[8 * u + 1] = a.y; f[8 * u + 2] = c.x; f[8 * u + 3] = c.y;
        f[8 * u + 4] = d.x; f[8 * u + 5] = d.y; f[8 * u + 6] = e.x; f[8 * u + 7] = e.y;
      }
      float amax = 0.f;
  #pragma unroll
      for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(f[k]));
      amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
      // biased exponent of amax (0 for 0 and subnormals); k = 7 - unbiased
      const int ebits = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
      const int kexp = min(127, max(-126, 134 - ebits));
      const float up = __uint_as_float(static_cast<uint32_t>(kexp + 127) << 23);
  #pragma unroll
      for (int j = 0; j < E / 4; ++j) {  // word j: dims (D/4) tig + 4j + 0..3
        uint32_t w1 = 0, w2 = 0;
  #pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float x0 = f[4 * j + 2 * h] * up, x1 = f[4 * j + 2 * h + 1] * up;
          const __nv_fp8x2_storage_t c1 =
              __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
          const __half2_raw r1 = __nv_cvt_fp8x2_to_halfraw2(c1, __NV_E4M3);
          __half2 r1h;
          r1h = *reinterpret_cast<const __half2*>(&r1);
          const float2 q1 = __half22float2(r1h);
          const __nv_fp8x2_storage_t c2 = __nv_cvt_float2_to_fp8x2(
              make_float2((x0 - q1.x) * 32.f, (x1 - q1.y) * 32.f), __NV_SATFINITE, __NV_E4M3);
          w1 |= static_cast<uint32_t>(c1) << (16 * h);
          w2 |= static_cast<uint32_t>(c2) << (16 * h);
        }
        qa[4 * (j / 2) + 2 * (j % 2)] = w1;      // row gid: q1
        qa[4 * (j / 2) + 2 * (j % 2) + 1] = w2;  // row gid + 8: q2
      }
      qf = ldexpf(p.scale_log2, -kexp);
    } else if constexpr (Q == 0) {
      const __nv_bfloat16* qb =
          p.q + (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(kvh) * G) * D + sub * 8;
      uint4 qw[G];
  #pragma unroll
      for (int g = 0; g < G; ++g)
        qw[g] = __ldg(reinterpret_cast<const uint4*>(qb + static_cast<size_t>(g) * D));
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
  #pragma unroll
      for (int g = 0; g < G; ++g) {
        q2[g][0] = __fmul2_rn(bf16x2_to_float2(qw[g].x), sc2);
        q2[g][1] = __fmul2_rn(bf16x2_to_float2(qw[g].y), sc2);
        q2[g][2] = __fmul2_rn(bf16x2_to_float2(qw[g].z), sc2);
        q2[g][3] = __fmul2_rn(bf16x2_to_float2(qw[g].w), sc2);
      }
    } else {
      // q of each head to int8 codes with one fp32 scale, by the cache's rule
      // (scale = amax / 127, code = round-half-even(q / scale)), once per CTA:
      // warp w quantises heads w, w + NW, ... into shared memory, then every
      // lane loads the codes it needs.  The scores carry scale_q * scale * log2 e.
      constexpr int E = D / 32;  // values per lane
      unsigned char* q8 = smem + Lay::QOFF;
      float* qs = reinterpret_cast<float*>(smem + Lay::QOFF + G * D);
      for (int g = warp; g < G; g += NW) {
        const __nv_bfloat16* qh =
            p.q + (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(kvh) * G + g) * D +
            lane * E;
        float f[E];
        if constexpr (E == 4) {
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(qh));
          const float2 a = bf16x2_to_float2(w.x), c = bf16x2_to_float2(w.y);
          f[0] = a.x; f[1] = a.y; f[2] = c.x; f[3] = c.y;
        } else {
          const float2 a = bf16x2_to_float2(__ldg(reinterpret_cast<const unsigned int*>(qh)));
          f[0] = a.x; f[1] = a.y;
        }
        float amax = 0.f;
  #pragma unroll
        for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(f[k]));
  #pragma unroll
        for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, m));
        const float qscale = __fdiv_rn(amax, 127.0f);
        uint32_t packed = 0;
        if (qscale > 0.f) {
  #pragma unroll
          for (int k = 0; k < E; ++k) {
            const float c8 = fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(f[k], qscale))));
            packed |= (static_cast<uint32_t>(static_cast<int>(c8)) & 0xffu) << (8 * k);
          }
        }
        if constexpr (E == 4)
          *reinterpret_cast<uint32_t*>(q8 + g * D + lane * E) = packed;
        else
          *reinterpret_cast<uint16_t*>(q8 + g * D + lane * E) = static_cast<uint16_t>(packed);
        if (lane == 0) qs[g] = qscale;
      }
      __syncthreads();
      // the lane's words: head(gid)'s codes at dims [(D/4) tig, +D/4) as
      // exact f16 pairs
      const int gid = lane >> 2, tig = lane & 3;
      const int hn = QCols<G>::head(gid);
      const unsigned char* row = q8 + hn * D + (D / 4) * tig;
      int qsum = 0;
  #pragma unroll
      for (int u = 0; u < D / 64; ++u) {
        const uint4 x = *reinterpret_cast<const uint4*>(row + 16 * u);
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
  #pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t ob = xw[k] ^ 0x80808080u;
          qa[2 * (4 * u + k)] = ob8x2_to_f16x2<0x4140>(ob);
          qa[2 * (4 * u + k) + 1] = ob8x2_to_f16x2<0x4342>(ob);
          qsum = __dp4a(static_cast<int>(xw[k]), 0x01010101, qsum);
        }
      }
      qsum += __shfl_xor_sync(kFullMask, qsum, 1);
      qsum += __shfl_xor_sync(kFullMask, qsum, 2);
      qoff = 128.f * static_cast<float>(qsum);
      qf = qs[hn] * p.scale_log2;
    }
  };
  if (!p.early_read) load_q();

  // Context length lives in device memory: check it here.
  const int ctx_cap = p.max_blocks_per_seq * BS;
  if (ctx < 0 || ctx > ctx_cap) {
    if (threadIdx.x == 0 && part == 0) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    ctx = ctx < 0 ? 0 : ctx_cap;
  }
  const int nblk = (ctx + BS - 1) / BS;
  int jb = 0, je = nblk;
  const int pidx = part;  // partition this CTA computes
  // Fused cache write: done by the warp that reads position ctx - 1 (the
  // owner of the sequence's last block, in the CTA whose range holds it),
  // once its first copies are out; it patches its tile with the new row at
  // iteration patch_it.
  // (after a shared prefix only a block past the prefix is ever written)
  const bool writer_cta =
      p.slot_mapping != nullptr &&
      (!SPLIT || (nblk > 0 ? (!after_prefix || nblk - 1 >= p.prefix_blocks) &&
                                 part == parts_of(nblk) - 1
                           : part == 0));
  const int last_blk = nblk > 0 ? nblk - 1 - (SPLIT ? static_cast<int>(part_first) : 0) : 0;
  if constexpr (SPLIT) {
    if (part == (after_prefix ? p.first_partition : 0) && threadIdx.x == 0 &&
        parts_of(nblk) > p.max_partitions)
      raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    if (part_first >= nblk) {  // past the end of this sequence; CTA-uniform, nothing issued
      if (p.early_read || after_prefix) griddep_wait();
      if (writer_cta && threadIdx.x == 0 && __ldg(p.slot_mapping + b) >= 0)
        raise_error(p.err, PA_DEVERR_SLOT);  // a new token for an empty sequence
      if (p.counters != nullptr && nblk == 0 && part == 0) {
        // merged output of an empty sequence: zeros, as the merge gives
        for (int idx = threadIdx.x; idx < G * (D / 8); idx += NW * 32) {
          const int hq = kvh * G + idx / (D / 8);
          *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(b) * p.num_q_heads + hq) * D +
                                    (idx % (D / 8)) * 8) = make_uint4(0, 0, 0, 0);
        }
      }
      return;
    }
    jb = static_cast<int>(part_first);
    je = min(nblk, jb + p.partition_blocks);
  }

  unsigned char* wbase = smem + warp * Lay::WARP;
  unsigned char* tiles = wbase;
  float* ps = reinterpret_cast<float*>(wbase + Lay::TILES);
  float* alpha_s = reinterpret_cast<float*>(wbase + Lay::TILES + Lay::PS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + Lay::TILES + Lay::PS + Lay::ALPHA);

  // This warp's share: logical blocks jb + warp + i * NW for i < nw.
  const int span = je - jb;
  const int nw = span > warp ? (span - warp + NW - 1) / NW : 0;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Block ids: 32 tiles per window, lane l holding tile (window * 32 + l);
  // the next window is prefetched while the current one is in use.
  int ids_win = 0;
  int ids_next = nw > 32 ? load_ids(1) : 0;

  const uint64_t policy = l2_policy_evict_first();
  const size_t block_stride = static_cast<size_t>(p.num_kv_heads) * BS * D;
  const size_t head_off = static_cast<size_t>(kvh) * BS * D;
  int issued = 0;
  // Called by the whole warp, in tile order, with the tile's ring stage: lane
  // 0 arms the stage's mbarrier with its bytes, and lanes 0 .. NCOPY - 1 each
  // issue one of its bulk copies (K tile, V tile, and for the 1-byte caches the
  // K and V scale runs).  A copy landing before the arming is fine: the
  // stage's phase cannot complete while lane 0's arrival is pending.
  auto issue = [&](int i, int st) {
    if ((i >> 5) != ids_win) {
      ids_cur = ids_next;
      ++ids_win;
      ids_next = (ids_win + 1) * 32 < nw ? load_ids(ids_win + 1) : 0;
    }
    int id = __shfl_sync(kFullMask, ids_cur, i & 31);
    constexpr int NCOPY = I8 ? 4 : 2;
    if (lane < NCOPY) {
      if (id < 0 || id >= p.num_blocks) {  // never dereferenced: read block 0 instead
        if (lane == 0) raise_error(p.err, PA_DEVERR_BLOCK_ID);
        id = 0;
      }
      uint64_t* bar = &bars[st];
      unsigned char* dst = tiles + st * Lay::STAGE;
      const size_t off = static_cast<size_t>(id) * block_stride + head_off;  // elements
      if (lane == 0) mbar_arrive_expect_tx(bar, Lay::STAGE);
      const void* src;
      unsigned bytes = Lay::KT;
      if constexpr (!I8) {
        src = lane == 0 ? static_cast<const void*>(p.k_cache + off)
                        : static_cast<const void*>(p.v_cache + off);
        dst += lane * Lay::KT;
      } else if (lane < 2) {
        src = lane == 0 ? static_cast<const void*>(p.k8 + off) : static_cast<const void*>(p.v8 + off);
        dst += lane * Lay::KT;
      } else {
        const size_t soff = off / D;  // scales: one per token
        src = lane == 2 ? static_cast<const void*>(p.k_scales + soff)
                        : static_cast<const void*>(p.v_scales + soff);
        bytes = BS * 4;
        dst += 2 * Lay::KT + (lane - 2) * BS * 4;
      }
      bulk_copy_g2s(dst, src, bytes, bar, policy);
    }
    issued = i + 1;
  };

  float2 acc[G][4];  // bf16 cache: this lane's dims of each head
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[g][k] = make_float2(0.f, 0.f);
  float acc8[D / 16][4];  // 1-byte caches: PV accumulators (pv_f16's layout)
#pragma unroll
  for (int c = 0; c < D / 16; ++c)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc8[c][k] = 0.f;
  float m_run = -INFINITY;  // running max of this lane's head, base-2 units
  float l_run = 0.f;        // this lane's share of that head's exp-sum
  float wsum = 0.f;         // int8 cache: this lane's share of its PV column's weights
  // 1-byte caches: the warp's power-of-two bound on the V scales it has
  // weighted (raise_v_bound) and its reciprocal; acc8 is in units of it
  float vbound = 0x1p-126f, vinv = 0x1p126f;
  const int my_head = (sub * R) / P;  // bf16 cache: the lane's score head and first pass
  const int my_i0 = (sub * R) % P;

  const int npro = nw < S ? nw : S;
  for (int i = 0; i < npro; ++i) issue(i, i);
  if (p.early_read) {
    griddep_wait();
    load_q();
  }
  // this warp patches its tile of the sequence's last block (the only
  // block with ctx - j * BS <= BS)
  const bool patch_row =
      writer_cta && warp == last_blk % NW &&
      fused_cache_write<D, Q>(p, b, kvh, ctx, tbl, lane, smem + Lay::PATCHOFF);

  int consumed = 0;
  int st = 0;        // ring stage of tile i
  unsigned ph = 0;   // its mbarrier phase parity
  for (int i = 0; i < nw; ++i) {
    const bool ready = __all_sync(kFullMask, mbar_wait_bounded(&bars[st], ph, p.err));
    if (!ready) break;
    const int j = jb + warp + i * NW;
    const int nvalid = min(BS, ctx - j * BS);
    const unsigned char* stage = tiles + st * Lay::STAGE;
    if (patch_row && nvalid == ctx - j * BS) {  // the new token's row (fused decode step)
      patch_tile<D, Q>(tiles + st * Lay::STAGE, Lay::KT, smem + Lay::PATCHOFF, nvalid - 1, lane);
      __syncwarp();
    }
    if constexpr (!I8) {
      const uint4* kt = reinterpret_cast<const uint4*>(stage);
      const uint4* vt = reinterpret_cast<const uint4*>(stage + Lay::KT);
      if (nvalid == BS)
        tile_step<D, G, true>(kt, vt, ps, alpha_s, q2, acc, m_run, l_run, nvalid, lane, sub, rg,
                              my_head, my_i0);
      else
        tile_step<D, G, false>(kt, vt, ps, alpha_s, q2, acc, m_run, l_run, nvalid, lane, sub,
                               rg, my_head, my_i0);
    } else {
      const float* ksc = reinterpret_cast<const float*>(stage + 2 * Lay::KT);
      const float* vsc = ksc + BS;
      if (nvalid == BS)
        tile_step_1b<D, G, Q == 2, true>(stage, stage + Lay::KT, ksc, vsc, qa, qf, qoff, acc8,
                                         m_run, l_run, wsum, vbound, vinv, nvalid, lane);
      else
        tile_step_1b<D, G, Q == 2, false>(stage, stage + Lay::KT, ksc, vsc, qa, qf, qoff, acc8,
                                          m_run, l_run, wsum, vbound, vinv, nvalid, lane);
    }
    consumed = i + 1;
    __syncwarp();  // every lane is done with this stage (and, bf16, with ps / alpha_s)
    if (i + S < nw) issue(i + S, st);
    if (++st == S) {
      st = 0;
      ph ^= 1u;
    }
  }
  // Only after a timed-out wait: let copies still in flight land (bounded)
  // before this CTA's shared memory can be reused.
  for (int i = consumed; i < issued; ++i) mbar_wait_bounded(&bars[i % S], (i / S) & 1, p.err);

  // partitions of this sequence that have a CTA (split-K)
  const int nparts = SPLIT ? min(parts_of(nblk), p.max_partitions) : 1;
  // of which this launch computes (the rest: a shared prefix's)
  const int nparts_here = nparts - (after_prefix ? p.first_partition : 0);
  // In-kernel split-K merge: count this CTA in now (the count's round trip
  // overlaps the merge of the warps below).  Counter word: arrivals in the
  // low 16 bits, partitions published in the high 16 bits.
  const bool merging = SPLIT && p.counters != nullptr && nparts > 1;
  unsigned* cnt = merging ? p.counters + static_cast<size_t>(b) * p.num_kv_heads + kvh : nullptr;
  unsigned arrival = 0;
  if (merging && threadIdx.x == 0)
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(arrival)
                 : "l"(cnt)
                 : "memory");

  // Per-warp totals: l over the lanes of each head, acc over row groups.
  if constexpr (I8) {  // the 4 lanes of each row of the QK MMA
    l_run += __shfl_xor_sync(kFullMask, l_run, 1);
    l_run += __shfl_xor_sync(kFullMask, l_run, 2);
  } else {
#pragma unroll
    for (int m = 1; m < Geo::HEAD_LANES; m <<= 1) l_run += __shfl_xor_sync(kFullMask, l_run, m);
#pragma unroll
    for (int m = L; m < 32; m <<= 1) l_run += __shfl_xor_sync(kFullMask, l_run, m);
  }
  // Merge warps through shared memory (each warp writes into its own, now
  // idle, tile ring): [G][D] acc, then m[G], l[G].
  float* mrg = reinterpret_cast<float*>(wbase);
  if constexpr (!I8) {
#pragma unroll
    for (int m = L; m < 32; m <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[g][k].x += __shfl_xor_sync(kFullMask, acc[g][k].x, m);
          acc[g][k].y += __shfl_xor_sync(kFullMask, acc[g][k].y, m);
        }
    if (rg == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float4* dst = reinterpret_cast<float4*>(mrg + g * D + sub * 8);
        dst[0] = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
        dst[1] = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
      }
    }
  } else {
    // acc8: (dims 16c + gid, 16c + gid + 8; columns 2 tig, 2 tig + 1), in
    // units of the warp's V-scale bound; G <= 4: each head's hi and lo parts
    // sit in the lanes tig and tig ^ G / 2 and are summed here
    using C = QCols<G>;
    if constexpr (C::PACKED) {
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc8[c][k] += __shfl_xor_sync(kFullMask, acc8[c][k], G / 2);
    }
    const int gid = lane >> 2, tig = lane & 3;
    if constexpr (Q == 1) {
      // int8: the sums held 2^-24 (w . v + 128 sum w); the weights of
      // columns 2 tig, 2 tig + 1 (heads 2 tig, 2 tig + 1 on the part-0
      // lanes) come from rows 2 tig and 2 tig + 1
      wsum += __shfl_xor_sync(kFullMask, wsum, 1);
      wsum += __shfl_xor_sync(kFullMask, wsum, 2);
      const float wa = 128.f * __shfl_sync(kFullMask, wsum, 8 * tig);
      const float wb = 128.f * __shfl_sync(kFullMask, wsum, 8 * tig + 4);
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        acc8[c][0] = fmaf(acc8[c][0], 0x1p24f, -wa);
        acc8[c][1] = fmaf(acc8[c][1], 0x1p24f, -wb);
        acc8[c][2] = fmaf(acc8[c][2], 0x1p24f, -wa);
        acc8[c][3] = fmaf(acc8[c][3], 0x1p24f, -wb);
      }
    }
    if (C::part0(tig)) {
      const int ha = C::head(2 * tig);
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        const int d0 = 16 * c + gid;
        mrg[ha * D + d0] = acc8[c][0] * vbound;
        mrg[(ha + 1) * D + d0] = acc8[c][1] * vbound;
        mrg[ha * D + d0 + 8] = acc8[c][2] * vbound;
        mrg[(ha + 1) * D + d0 + 8] = acc8[c][3] * vbound;
      }
    }
  }
  if constexpr (I8) {  // head gid's state, from its part-0 row
    if (lane % 4 == 0 && lane / 4 < G) {
      mrg[G * D + lane / 4] = m_run;
      mrg[G * D + G + lane / 4] = l_run;
    }
  } else if (rg == 0 && sub % Geo::HEAD_LANES == 0) {
    mrg[G * D + my_head] = m_run;
    mrg[G * D + G + my_head] = l_run;
  }
  __syncthreads();

  // A merged split-K launch whose sequence has one partition writes the
  // output directly (the merge of one partition is the identity).
  const bool direct = !SPLIT || (p.counters != nullptr && nparts == 1);
  for (int idx = threadIdx.x; idx < G * (D / 8); idx += NW * 32) {
    const int g = idx / (D / 8);
    const int d0 = (idx % (D / 8)) * 8;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(smem + w * Lay::WARP)[G * D + g]);
    float o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = 0.f;
    float Ls = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float* mw = reinterpret_cast<const float*>(smem + w * Lay::WARP);
        const float c = exp2f(mw[G * D + g] - M);
        Ls += mw[G * D + G + g] * c;
        const float4 a = *reinterpret_cast<const float4*>(mw + g * D + d0);
        const float4 bq = *reinterpret_cast<const float4*>(mw + g * D + d0 + 4);
        o[0] += a.x * c;
        o[1] += a.y * c;
        o[2] += a.z * c;
        o[3] += a.w * c;
        o[4] += bq.x * c;
        o[5] += bq.y * c;
        o[6] += bq.z * c;
        o[7] += bq.w * c;
      }
      const float inv = 1.0f / Ls;
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] *= inv;
    }
    const int hq = kvh * G + g;
    if (SPLIT && !direct) {
      const size_t row =
          (static_cast<size_t>(b) * p.num_q_heads + hq) * p.max_partitions + pidx;
      float4* dst = reinterpret_cast<float4*>(p.ws_o + row * D + d0);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
      if (d0 == 0) {
        p.ws_m[row] = M * kLn2;  // back to natural-log units
        p.ws_l[row] = Ls;
      }
    } else {
      __nv_bfloat162 h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = __float22bfloat162_rn(make_float2(o[2 * k], o[2 * k + 1]));
      *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(b) * p.num_q_heads + hq) * D + d0) =
          *reinterpret_cast<const uint4*>(h);
    }
  }

  if constexpr (SPLIT) {
    if (!merging) {
      if (after_prefix) griddep_wait();
      return;
    }
    // Every CTA but the last to arrive publishes its rows (a release on the
    // counter) and leaves; the last waits until all the others have
    // published -- they arrived before it, so they are running and finish
    // without waiting on anything -- then merges all partitions by the
    // log-sum-exp identity (as pa_splitk_reduce) and zeroes the counter for
    // the next launch.  The wait is bounded like every other.
    __shared__ unsigned s_last;
    __syncthreads();  // every thread's workspace rows are written
    if (threadIdx.x == 0) {
      if ((arrival & 0xFFFFu) + 1u != static_cast<unsigned>(nparts_here)) {
        asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(cnt), "r"(0x10000u)
                     : "memory");
        s_last = 0u;
      } else {
        const uint64_t t0 = global_timer_ns();
        bool ok = true;
        for (;;) {
          unsigned v;
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
          if ((v >> 16) + 1u >= static_cast<unsigned>(nparts_here)) break;
          if (global_timer_ns() - t0 > 2000000000ull) {
            raise_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          __nanosleep(64);
        }
        s_last = ok ? 1u : 0u;
      }
    }
    __syncthreads();
    if (after_prefix) griddep_wait();  // the prefix's partitions are written
    if (!s_last) return;
    for (int idx = threadIdx.x; idx < G * (D / 4); idx += NW * 32) {
      const int hq = kvh * G + idx / (D / 4);
      const int d0 = (idx % (D / 4)) * 4;
      const size_t row0 = (static_cast<size_t>(b) * p.num_q_heads + hq) * p.max_partitions;
      // one pass, rescaling to the running maximum (natural-log units); the
      // rows of up to MU partitions are loaded together (one round trip)
      constexpr int MU = 8;
      float M = -INFINITY, Ls = 0.f;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i0 = 0; i0 < nparts; i0 += MU) {
        float mv[MU], lv[MU];
        float4 ov[MU];
#pragma unroll
        for (int u = 0; u < MU; ++u) {
          if (i0 + u < nparts) {
            mv[u] = __ldcg(p.ws_m + row0 + i0 + u);
            lv[u] = __ldcg(p.ws_l + row0 + i0 + u);
            ov[u] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + (row0 + i0 + u) * D + d0));
          }
        }
#pragma unroll
        for (int u = 0; u < MU; ++u) {
          if (i0 + u >= nparts) break;
          const float m = mv[u];
          if (m > M) {
            const float c = expf(M - m);  // 0 on the first partition
            Ls *= c;
            a.x *= c;
            a.y *= c;
            a.z *= c;
            a.w *= c;
            M = m;
          }
          const float w = lv[u] * expf(m - M);
          Ls += w;
          a.x += w * ov[u].x;
          a.y += w * ov[u].y;
          a.z += w * ov[u].z;
          a.w += w * ov[u].w;
        }
      }
      const float inv = 1.0f / Ls;  // every partition has a token: Ls >= 1
      const __nv_bfloat162 h0 = __float22bfloat162_rn(make_float2(a.x * inv, a.y * inv));
      const __nv_bfloat162 h1 = __float22bfloat162_rn(make_float2(a.z * inv, a.w * inv));
      uint2 packed;
      packed.x = *reinterpret_cast<const uint32_t*>(&h0);
      packed.y = *reinterpret_cast<const uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(b) * p.num_q_heads + hq) * D + d0) =
          packed;
    }
    if (threadIdx.x == 0) *cnt = 0u;
  }
}

// Raises the dynamic shared-memory limit of a kernel once per device.
template <typename K>
cudaError_t allow_smem(K kernel, int bytes, std::atomic<uint64_t>& done_mask) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done_mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done_mask.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <int D, int G, bool SPLIT, int Q>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  constexpr bool I8 = Q != 0;
  constexpr int NW = Pipe<D, SPLIT, Q>::NW, S = Pipe<D, SPLIT, Q>::S;
  using Lay = SmemLayout<D, G, NW, S, I8>;
  static std::atomic<uint64_t> smem_set{0};
  auto kernel = paged_decode_kernel<D, G, NW, S, SPLIT, Q>;
  cudaError_t e = allow_smem(kernel, Lay::TOTAL, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid =
      (SPLIT && p.order != nullptr)
          ? dim3(p.num_kv_heads, p.num_seqs * (p.max_partitions - p.first_partition), 1)
                        : dim3(p.num_kv_heads, p.num_seqs,
                               SPLIT ? p.max_partitions - p.first_partition : 1);
  return launch_pdl(kernel, grid, dim3(NW * 32), Lay::TOTAL, stream, p);
}

template <int D, int G, int Q>
cudaError_t launch_decode_g(const DecodeParams& p, bool split, cudaStream_t stream) {
  return split ? launch_decode_t<D, G, true, Q>(p, stream)
               : launch_decode_t<D, G, false, Q>(p, stream);
}

template <int D, int Q>
cudaError_t launch_decode_d(const DecodeParams& p, int group, bool split, cudaStream_t stream) {
  switch (group) {
    case 2:
      return launch_decode_g<D, 2, Q>(p, split, stream);
    case 4:
      return launch_decode_g<D, 4, Q>(p, split, stream);
    case 8:
      return launch_decode_g<D, 8, Q>(p, split, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_shape_supported(int head_dim, int group, int block_size) {
  return block_size == kBlockSize && (head_dim == 64 || head_dim == 128) &&
         (group == 2 || group == 4 || group == 8);
}

cudaError_t launch_decode(const DecodeParams& p, int head_dim, int group, bool split,
                          cudaStream_t stream) {
  const int q = p.k8 == nullptr ? 0 : (p.fp8 ? 2 : 1);
  if (head_dim == 128)
    return q == 0 ? launch_decode_d<128, 0>(p, group, split, stream)
                  : q == 1 ? launch_decode_d<128, 1>(p, group, split, stream)
                           : launch_decode_d<128, 2>(p, group, split, stream);
  if (head_dim == 64)
    return q == 0 ? launch_decode_d<64, 0>(p, group, split, stream)
                  : q == 1 ? launch_decode_d<64, 1>(p, group, split, stream)
                           : launch_decode_d<64, 2>(p, group, split, stream);
  return cudaErrorInvalidValue;
}


}  // namespace pa
