// Paged (chunked) prefill attention on the 5th-generation tensor cores, sm_103a.
//
// What is computed: "How LLM Inference Serving Works" (dev.to), sections "Two
// Phases: Prefill and Decode" (prefill runs the prompt's tokens together and
// is compute-bound) and "Chunked prefill" (a long prompt is split into chunks
// that share steps with decodes).  A chunk of n new tokens of a sequence with
// context length ctx (chunk included, its K/V already in the cache) holds
// positions ctx - n .. ctx - 1; the query at position p attends to the cached
// keys 0 .. p through the block table ("PagedAttention: Virtual Memory for
// the KV Cache").  n = 1 is a decode step.
//
// Design (one CTA per 128 query rows: 4 softmax warps, an MMA warp, two copy
// warps; two CTAs per SM):
//  * Rows are (token, head) pairs of one GQA group: 128 / G tokens x G heads,
//    so each K/V tile loaded serves the whole group.  Q arrives by one 3-D TMA
//    per 64-column half; K and V arrive per 16-token block by 2-D TMA (the
//    block table is a gather of 16-row boxes), kKeys = 64 keys (4 blocks) per
//    chunk by default (PA_PREFILL_KEYS: 64 or 128), in rings of kStages chunk
//    stages each.  TMA writes the 128-byte-swizzled layout the tensor cores
//    read.
//  * S = Q K^T (M = 128 rows, N = kKeys, K = 128 dims) and O += P V
//    (M = 128, N = 128 dims, K = kKeys) are tcgen05.mma kind::f16 (bf16 in,
//    fp32 accumulate) issued by one thread of the MMA warp, with S and O in
//    tensor memory (kSBuf S buffers + O).  V is the MN-major operand.  At 64
//    keys: Q 32 KiB, K and V 2 x 16 KiB each, 2 S buffers, 256 tensor-memory
//    columns, so two CTAs share an SM and one's MMAs overlap the other's
//    softmax; at 128 keys: 3 stages of 32 KiB, 3 S buffers, all 512 columns,
//    one CTA per SM.
//  * The online softmax reads its row of S from tensor memory (one thread
//    per row = TMEM lane, four softmax warps, by default; or two threads per
//    row with flags, maxima and sums combined through shared memory), masks
//    causally, keeps a reference maximum that is only raised when the row
//    grows past it by more than 2^8 (then O's row is rescaled in tensor
//    memory) -- so a chunk's weights are taken against the reference first,
//    and only a chunk whose weights could exceed 2^8 (a sum of the thread's
//    weights above 2^7) takes its maxima and redoes them -- and writes P
//    back into tensor memory, over its own S, as two
//    bf16 parts, hi = p truncated to bf16 and lo = bf16(p - hi), each multiplied with V
//    by its own MMA reading A from tensor memory: the weights keep ~17 bits
//    instead of bf16's 8 (a single bf16 P puts elementwise errors of several
//    per cent on outputs that are small by cancellation).
//  * Every wait is bounded; on a timeout the CTA records PA_DEVERR_WAIT_TIMEOUT,
//    lets its own copies and MMAs in flight land (bounded), frees tensor
//    memory and returns.  Block ids and lengths in device memory are checked.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/pa.h"
#include "device.cuh"
#include "internal.h"

namespace pa {
namespace {

// Keys per chunk (the N of S = Q K^T): 128, one CTA per SM holding 3 S
// buffers and 3-stage K and V rings; or 64, two CTAs per SM (so four softmax
// warps per scheduler instead of two), each with 2 S buffers and 2-stage rings.
#ifndef PA_PREFILL_KEYS
#define PA_PREFILL_KEYS 64
#endif
constexpr int kD = 128;                 // head_dim
constexpr int kRows = 128;              // query rows per CTA = MMA M
constexpr int kKeys = PA_PREFILL_KEYS;  // keys per chunk = MMA N of S = Q K^T
constexpr int kCtasPerSm = kKeys == 128 ? 1 : 2;
constexpr int kBS = 16;                 // tokens per cache block
constexpr int kChunkBlocks = kKeys / kBS;
constexpr int kHalf = kRows * 128;      // one 64-column half of Q (128 rows x 128 bytes)
constexpr int kKVHalf = kKeys * 128;    // one 64-column half of a K or V chunk
constexpr int kBox = kBS * 128;         // one TMA box of K or V: 16 rows x 128 bytes
constexpr int kSBuf = kKeys == 128 ? 3 : 2;  // S (then P) buffers in tensor memory
constexpr int kAhead = kSBuf - 1;       // chunks of scores issued ahead of PV
constexpr uint32_t kTO = kSBuf * kKeys;  // O's first column (after the S buffers)
constexpr uint32_t kTmemCols = kKeys == 128 ? 512 : 256;  // S buffers + O (128 columns)
static_assert(kTO + 128 <= kTmemCols, "tensor memory");

// Shared memory, from a 1024-byte aligned base (the swizzle atom).
constexpr int kQ = 0;                   // Q: 2 halves
constexpr int kStages = kKeys == 128 ? 3 : 2;  // K and V ring depth (chunks)
constexpr int kK = kQ + 2 * kHalf;      // K: kStages stages x 2 halves
constexpr int kV = kK + 2 * kStages * kKVHalf;  // V: kStages stages x 2 halves
constexpr int kBar = kV + 2 * kStages * kKVHalf;  // mbarriers and the TMEM address slot
// Softmax threads per row of S (TMEM lane): 1 (all kKeys columns), or 2
// (kKeys / 2 columns each, the two warps of a lane quarter exchanging through
// shared memory; measured slower: 806 against 842 TFLOP/s on the 16 x 512
// step at 64 keys).
#ifndef PA_PREFILL_ROW_THREADS
#define PA_PREFILL_ROW_THREADS 1
#endif
constexpr int kRowThreads = PA_PREFILL_ROW_THREADS;
static_assert(kRowThreads == 1 || kRowThreads == 2, "softmax threads per row");
constexpr int kSoftmaxThreads = 128 * kRowThreads;
constexpr int kOCols = kD / kRowThreads;  // columns of O per softmax thread
// Two threads per row exchange, per row and column half: the flags "this
// chunk may move the reference", double-buffered by chunk parity; the final
// sums; the maxima of a chunk that may move it.
constexpr int kRed = kBar + 256;
constexpr int kSmemBytes = kRed + (kRowThreads == 2 ? 4 * 2 * kRows * 4 : 0) + 1024;  // + slack
constexpr int kThreads = kSoftmaxThreads + 96;  // + an MMA warp and two copy warps
static_assert(kCtasPerSm * kSmemBytes <= 232448, "shared memory per SM");

struct PrefillParams {
  __nv_bfloat16* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  unsigned* err;
  int max_blocks_per_seq;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int total_q;
  float scale_log2;
  // Shared-prefix mode (split_blocks > 0): one virtual sequence whose
  // "tokens" are a decode batch's queries (q [total_q = B, Hq, D]), each row
  // (query b, head) attending, without a causal mask, to the keys of blocks
  // [s * split_blocks, (s + 1) * split_blocks) of block-table row 0 (s =
  // blockIdx.z), and its partial result going to a split-K workspace [B, Hq,
  // max_partitions] at partition s: o / l, m (natural-log units) and l.
  int split_blocks;
  float* ws_o;
  float* ws_m;
  float* ws_l;
  int max_partitions;
};

// ---- tcgen05 / TMA wrappers -------------------------------------------------

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), descriptor version 1 (bit 46),
// swizzle mode 2 (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(lbo >> 4) << 16) | (static_cast<uint64_t>(sbo >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), A / B major (bit 15 / 16: 0 = K-major, 1 =
// MN-major), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t idesc_bf16(int m, int n, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}
constexpr uint32_t kIdescQK = idesc_bf16(kRows, kKeys, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(kRows, kD, 0, 1);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// The same with A (M x K, K-major) read from tensor memory: bf16 pairs packed
// in 32-bit columns, row m in lane m.
__device__ __forceinline__ void umma_bf16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes become visible to the async proxy (MMA).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
// 16 consecutive columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// ---- the kernel ------------------------------------------------------------

// exp2 on the special-function unit (flushes subnormal results to zero; the
// arguments here are <= 8 and the results are weights of at most 2^8).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Barrier of the two warps that share a TMEM lane quarter (warps w, w + 4).
__device__ __forceinline__ void pair_sync(int warp) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
}

// grid (query tiles, KV heads, sequences), kThreads threads.  The first
// kSoftmaxThreads run the softmax: thread t handles row t % 128 (TMEM lane;
// with two threads per row, warps w and w + 4 share a lane quarter), columns
// [h HK, (h + 1) HK) of S and [h kOCols, (h + 1) kOCols) of O, h = t / 128.
// The next warp issues the MMAs (lane 0), the one after it the Q and K
// copies and the last the V copies (one block per lane), so that no chain
// waits on another's latencies.
//
// Tensor memory: kSBuf S buffers of kKeys columns, then O (128 columns).  P of
// chunk c replaces S of chunk c in place, buffer c % kSBuf: each softmax
// thread writes its HK keys' weights over the HK columns of S it read, the hi
// parts in the first half of them and the lo parts in the second (bf16 pairs
// packed per column), so with two threads per row neither writes a column
// the other still has to read.  K and V run in kStages-chunk rings.  Every
// ring slot has its own barriers ("full": copies landed; "free": committed
// after the MMA that read it; "pv_done": PV read the P it holds), so that
// each wait names one use of one slot and no parity wait can match an older
// phase.
//
// MMA warp, per chunk c (A = kAhead = kSBuf - 1): wait PV(c-1) (its buffer
//   S[(c+A)%kSBuf] held P(c-1)) and K(c+A): S[(c+A)%kSBuf] = Q K(c+A)^T; wait
//   V(c) and P(c): O += P V(c).
// Copy warps, per chunk c: wait K slot of c free: copy K(c+kStages) (K warp);
//   wait V slot of c-1 free: copy V(c+kStages-1) (V warp).
// Softmax warps, per chunk c: wait S(c); read it; exponentials against the
//   reference; flags "may move the reference" (with two threads per row,
//   combined by the pair of warps); only if a row of the warp is flagged:
//   read S again, row maxima, move the reference, exponentials again;
//   rescale O only if the reference moved (after PV(c-1)); P into
//   S[c%kSBuf]; arrive on p_ready[c%kSBuf].
// No softmax thread leaves the loop early (the pair barriers must stay
// matched): one whose wait timed out keeps iterating without waiting or working.
template <int G>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, const PrefillParams p) {
  constexpr int TQ = kRows / G;  // query tokens per CTA
  constexpr int HK = kKeys / kRowThreads;  // columns of S per softmax thread
  constexpr int kMmaWarp = kSoftmaxThreads / 32, kCopyWarp = kMmaWarp + 1;
  griddep_wait();
  griddep_launch_dependents();
  const bool shared_prefix = p.split_blocks > 0;  // CTA-uniform
  const int tile = blockIdx.x, kvh = blockIdx.y, b = shared_prefix ? 0 : blockIdx.z;
  const int split = shared_prefix ? blockIdx.z : 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Lengths live in device memory: check them (CTA-uniform).  A shared
  // prefix split: every query sees the split's keys (sizes checked on the host).
  const int q0 = shared_prefix ? 0 : __ldg(p.query_start + b);
  const int q1 = shared_prefix ? p.total_q : __ldg(p.query_start + b + 1);
  const int ctx = shared_prefix ? p.split_blocks * kBS : __ldg(p.context_lens + b);
  const int n = q1 - q0;
  if (!shared_prefix &&
      (q0 < 0 || q1 > p.total_q || n < 0 || n > ctx || ctx > p.max_blocks_per_seq * kBS)) {
    if (tid == 0 && tile == 0 && kvh == 0) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    return;
  }
  const int i0 = tile * TQ;
  if (i0 >= n) return;
  // keys the tile's last query sees
  const int nk = shared_prefix ? ctx : ctx - n + min(n, i0 + TQ);
  const int nchunks = (nk + kKeys - 1) / kKeys;
  const int nblk_all = (nk + kBS - 1) / kBS;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* k_full = reinterpret_cast<uint64_t*>(sm + kBar);  // [3] copies landed
  uint64_t* v_full = k_full + 3;                               // [3]
  uint64_t* k_free = k_full + 6;                               // [3] QK that read it done
  uint64_t* v_free = k_full + 9;                               // [3] PV that read it done
  uint64_t* s_done = k_full + 12;                              // [3] per S buffer
  // [3] per S buffer: PV of the chunk whose P the buffer holds is done.  Its
  // commit covers every MMA issued before, so "PV(c) done" also means every
  // earlier PV is done; the next phase of the same barrier (PV(c + 3)) cannot
  // complete before the waiter's own arrival for c + 3, so no parity wait on
  // it can match a stale or a future phase.
  uint64_t* pv_done = k_full + 15;
  uint64_t* q_full = k_full + 18;
  // [3] per S buffer, 8 warp arrivals per chunk.  One barrier per buffer: a
  // softmax warp can be up to kAhead chunks ahead of another (the scores of
  // c + kAhead need only PV(c - 1)), and its arrivals must not count for an
  // earlier chunk.
  uint64_t* p_ready = k_full + 19;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kBar + 240);
  float* red = reinterpret_cast<float*>(sm + kRed);  // [4][2][128], two threads per row

  if (tid == 0) {
    for (int i = 0; i < 19; ++i) mbar_init(k_full + i, 1);
    for (int i = 0; i < kSBuf; ++i) mbar_init(&p_ready[i], kSoftmaxThreads / 32);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kCopyWarp) {
    // ------------------------------------------------------------ copies
    // Warp kCopyWarp copies Q and the K ring, warp kCopyWarp + 1 the V ring:
    // a 32 KiB chunk is 16 tensor-map boxes whose issue takes ~1.6k cycles,
    // so one warp issuing both rings paced the whole pipeline.
    const bool vwarp = warp == kCopyWarp + 1;
    const int32_t* tbl = p.block_tables + static_cast<size_t>(b) * p.max_blocks_per_seq +
                         static_cast<size_t>(split) * p.split_blocks;
    int last_k = -1, last_v = -1;  // last chunk copied into each ring (for the drain)
    bool ok = true;                // lane 0: every wait so far succeeded
    auto uniform = [&](bool v) { return __shfl_sync(kFullMask, v ? 1 : 0, 0) != 0; };
    // Lane j < 8: the raw table entry of block j of chunk c (checked at use),
    // fetched a chunk ahead so that the table's latency stays off the copies.
    auto fetch_id = [&](int c) -> int {
      if (c >= nchunks || lane >= min(kChunkBlocks, nblk_all - c * kChunkBlocks)) return 0;
      return __ldg(tbl + c * kChunkBlocks + lane);
    };
    // K (or V) of chunk c into stage c % 3, one block per lane
    auto load = [&](int c, bool is_v, int id) {
      const int st = c % kStages;
      const int nb = min(kChunkBlocks, nblk_all - c * kChunkBlocks);
      uint64_t* bar = is_v ? &v_full[st] : &k_full[st];
      unsigned char* dst = sm + (is_v ? kV : kK) + 2 * st * kKVHalf + lane * kBox;
      if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nb * 2 * kBox));
      __syncwarp();
      if (lane < nb) {
        if (id < 0 || id >= p.num_blocks) {  // never dereferenced: block 0 is read instead
          raise_error(p.err, PA_DEVERR_BLOCK_ID);
          id = 0;
        }
        const int row = (id * p.num_kv_heads + kvh) * kBS;
        tma_2d(dst, is_v ? &tv : &tk, 0, row, bar);
        tma_2d(dst + kKVHalf, is_v ? &tv : &tk, 64, row, bar);
      }
      __syncwarp();
      if (is_v) last_v = c; else last_k = c;
    };
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(vwarp ? &tv : &tk))
                   : "memory");
      if (!vwarp) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tq)) : "memory");
        mbar_arrive_expect_tx(q_full, 2 * kHalf);
        tma_3d(sm + kQ, &tq, 0, kvh * G, q0 + i0, q_full);
        tma_3d(sm + kQ + kHalf, &tq, 64, kvh * G, q0 + i0, q_full);
      }
    }
    {
      int ids[kStages];
#pragma unroll
      for (int c = 0; c < kStages; ++c) ids[c] = fetch_id(c);
#pragma unroll
      for (int c = 0; c < kStages; ++c)
        if (c < nchunks) load(c, vwarp, ids[c]);
    }
    // Block ids run kIdAhead chunks ahead of the copies (idq[i]: the chunk
    // i copies after the next), so that no copy waits on a table load.
    constexpr int kIdAhead = 4;
    int idq[kIdAhead];
#pragma unroll
    for (int i = 0; i < kIdAhead; ++i) idq[i] = fetch_id(kStages + i);
    // K warp, iteration c: QK(c) has read K stage c % kStages -> copy
    // K(c + kStages).  V warp, iteration c: PV(c - 1) has read V stage
    // (c - 1) % kStages -> copy V(c - 1 + kStages).
    for (int c = vwarp ? 1 : 0; uniform(ok); ++c) {
      const int next = vwarp ? c - 1 + kStages : c + kStages;  // the chunk this iteration copies
      if (next >= nchunks) break;
      const int freed = vwarp ? c - 1 : c;     // the chunk whose use frees the stage
      if (lane == 0)
        ok = mbar_wait_bounded(vwarp ? &v_free[freed % kStages] : &k_free[freed % kStages],
                               (freed / kStages) & 1, p.err);
      if (!uniform(ok)) break;
      load(next, vwarp, idq[0]);
#pragma unroll
      for (int i = 0; i + 1 < kIdAhead; ++i) idq[i] = idq[i + 1];
      idq[kIdAhead - 1] = fetch_id(next + kIdAhead);
    }
    // A shared prefix: the V warp of each KV head 0 CTA checks that its
    // tile's sequences hold this split's blocks (the same table entries as
    // sequence 0) and, in the first split, that their contexts go past the
    // prefix.
    if (shared_prefix && vwarp && kvh == 0) {
      const int32_t* row0 = p.block_tables + static_cast<size_t>(split) * p.split_blocks;
      const int prefix_tokens = p.split_blocks * kBS * static_cast<int>(gridDim.z);
      const int seqs = min(TQ, n - i0);
      const int pairs = seqs * p.split_blocks;  // (sequence, block) pairs, spread over the lanes
      bool bad = false;
#pragma unroll 4
      for (int e = lane; e < pairs; e += 32) {
        const int t = e / p.split_blocks, j = e - t * p.split_blocks;
        bad |= __ldg(row0 + static_cast<size_t>(i0 + t) * p.max_blocks_per_seq + j) !=
               __ldg(row0 + j);
      }
      if (split == 0)
        for (int t = lane; t < seqs; t += 32) bad |= __ldg(p.context_lens + i0 + t) <= prefix_tokens;
      if (__any_sync(kFullMask, bad) && lane == 0) raise_error(p.err, PA_DEVERR_PREFIX);
    }
    // Copies this warp issued land before the CTA's shared memory is given up
    // (earlier uses of a stage completed before its last copy was issued).
    if (lane == 0) {
      for (int st = 0; st < kStages; ++st) {
        const int ck = last_k - ((last_k - st) % kStages + kStages) % kStages;
        const int cv = last_v - ((last_v - st) % kStages + kStages) % kStages;
        if (ck >= 0) mbar_wait_bounded(&k_full[st], (ck / kStages) & 1, p.err);
        if (cv >= 0) mbar_wait_bounded(&v_full[st], (cv / kStages) & 1, p.err);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMAs
    const uint32_t sQ = smem_u32(sm + kQ), sK = smem_u32(sm + kK), sV = smem_u32(sm + kV);
    int s_iss = 0, o_iss = 0;  // MMAs committed (for the drain)
    if (lane == 0) {
      // lane 0: S[c % 3] = Q K(c)^T
      const uint64_t qdesc = sw128_desc(sQ, 16, 1024);
      auto qk = [&](int c) {
        const int sb = c % kSBuf, st = c % kStages;
        const uint64_t kdesc = sw128_desc(sK + 2 * st * kKVHalf, 16, 1024);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          // descriptor units (16 bytes): kk's 32-byte column step within a
          // 64-column half, and the half's offset
          const uint32_t qoff = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
          const uint32_t koff = ((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4;
          umma_bf16(tmem + sb * kKeys, qdesc + qoff, kdesc + koff, kIdescQK, kk > 0);
        }
        umma_commit(&s_done[sb]);
        umma_commit(&k_free[st]);
        ++s_iss;
      };
      bool ok = mbar_wait_bounded(q_full, 0, p.err);
      for (int c = 0; c < kAhead && c < nchunks && ok; ++c) {
        ok = mbar_wait_bounded(&k_full[c % kStages], (c / kStages) & 1, p.err);
        if (ok) qk(c);
      }
      for (int c = 0; c < nchunks && ok; ++c) {
        const int sb = c % kSBuf, st = c % kStages;
        if (c + kAhead < nchunks) {
          // scores kAhead chunks ahead: PV(c-1) is done with P(c-1) in
          // S[(c + kAhead) % kSBuf]
          if (c >= 1)
            ok = mbar_wait_bounded(&pv_done[(c + kAhead) % kSBuf], ((c - 1) / kSBuf) & 1,
                                   p.err);
          ok = ok && mbar_wait_bounded(&k_full[(c + kAhead) % kStages],
                                       ((c + kAhead) / kStages) & 1, p.err);
          if (!ok) break;
          qk(c + kAhead);
        }
        ok = mbar_wait_bounded(&v_full[st], (c / kStages) & 1, p.err) &&
             mbar_wait_bounded(&p_ready[sb], (c / kSBuf) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint64_t vdesc = sw128_desc(sV + 2 * st * kKVHalf, kKVHalf, 1024);
        // keys 16 kk .. 16 kk + 15: softmax thread kk / (HK / 16) of each row
        // wrote their hi pairs 8 (kk % (HK / 16)) columns into its HK columns
        // of S, the lo pairs HK / 2 columns further
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint32_t hi = sb * kKeys + HK * (kk / (HK / 16)) + 8 * (kk % (HK / 16));
          umma_bf16_ts(tmem + kTO, tmem + hi, vdesc + kk * (2048 >> 4), kIdescPV,
                       (c > 0 || kk > 0) ? 1u : 0u);
          umma_bf16_ts(tmem + kTO, tmem + hi + HK / 2, vdesc + kk * (2048 >> 4), kIdescPV, 1u);
        }
        umma_commit(&pv_done[sb]);
        umma_commit(&v_free[st]);
        ++o_iss;
      }
      // The MMAs issued complete before tensor and shared memory are given up
      // (each commit covers every MMA before it).
      if (o_iss > 0)
        mbar_wait_bounded(&pv_done[(o_iss - 1) % kSBuf], ((o_iss - 1) / kSBuf) & 1, p.err);
      if (s_iss > 0)
        mbar_wait_bounded(&s_done[(s_iss - 1) % kSBuf], ((s_iss - 1) / kSBuf) & 1, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int hcol = tid >> 7;  // column half
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_base + kTO + kOCols * hcol;
    const int r = tid & (kRows - 1);  // row: token r / G of the tile, head r % G
    const int qi = i0 + r / G;
    const bool row_ok = qi < n;
    const int pos = shared_prefix ? nk - 1 : ctx - n + qi;  // sees keys 0 .. pos
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY;  // reference maximum of the exponentials (base 2)
    float l_sum = 0.f;
    bool ok = true;  // sticky: this thread's waits all succeeded
    const int prow = (r >> 3) * 1024 + (r & 7) * 128;  // row in a swizzled 128-row tile

    for (int c = 0; c < nchunks; ++c) {
      const int sb = c % kSBuf;
      bool lok = ok && mbar_wait_bounded(&s_done[sb], (c / kSBuf) & 1, p.err);
      lok = __all_sync(kFullMask, lok);
      uint32_t sv[HK];
      if (lok) {
        tc_fence_after();
#pragma unroll
        for (int q4 = 0; q4 < HK / 32; ++q4) {
          uint32_t(&chunk)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * q4);
          tmem_ld32(tmem + lane_base + sb * kKeys + HK * hcol + 32 * q4, chunk);
        }
        tmem_wait_ld();
      }
      // causal mask
      const int lim = row_ok ? pos - c * kKeys - HK * hcol : -1;  // visible: j <= lim
      const bool masked = !__all_sync(kFullMask, lim >= HK - 1);
      if (lok && masked) {
#pragma unroll
        for (int j = 0; j < HK; ++j)
          if (j > lim) sv[j] = __float_as_uint(-INFINITY);
      }
      // The weights against the current reference (none yet: offset 0, and a
      // row without a reference has only masked scores so far, which give
      // exp2(-inf) = 0).  The reference moves only when the chunk's maximum
      // exceeds it by more than 2^8, which makes a weight above 2^8 and so
      // this thread's sum above 2^7: only then (or with no reference yet) are
      // the chunk's maxima taken, the scores read again and the weights redone.
      const float2 sl2x2 = make_float2(sl2, sl2);
      float psum = 0.f;
      auto weights = [&]() {
        const bool live = m_used != -INFINITY;
        const float2 neg2 = make_float2(live ? -m_used : 0.f, live ? -m_used : 0.f);
        float2 ps4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};  // independent partial sums
#pragma unroll
        for (int j = 0; j < HK; j += 2) {
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])), sl2x2, neg2);
          const float2 e = make_float2(ex2(x.x), ex2(x.y));
          ps4[(j >> 1) & 3] = __fadd2_rn(ps4[(j >> 1) & 3], e);
          sv[j] = __float_as_uint(e.x);
          sv[j + 1] = __float_as_uint(e.y);
        }
        const float2 pa = __fadd2_rn(__fadd2_rn(ps4[0], ps4[2]), __fadd2_rn(ps4[1], ps4[3]));
        psum = pa.x + pa.y;
      };
      // (a row of the tile without a reference yet takes the maxima anyway:
      // its weights wait for them; a row past the tile's queries has only
      // masked scores, weights 0)
      if (lok && (m_used != -INFINITY || !row_ok)) weights();
      const bool want = lok && row_ok && (m_used == -INFINITY || !(psum <= 128.f));
      // with two threads per row, both halves' flags (warps w and w + 4),
      // through a buffer of this chunk's parity: the partner's read of the
      // same buffer two chunks ago came before its arrival on the last
      // barrier, which this thread has passed
      bool row_want = want;
      if constexpr (kRowThreads == 2) {
        float* redc = red + (c & 1) * 2 * kRows;
        tc_fence_before();
        redc[hcol * kRows + r] = want ? 1.f : 0.f;
        pair_sync(warp);
        row_want = redc[r] != 0.f || redc[kRows + r] != 0.f;
        tc_fence_after();
      }
      float alpha = 1.f;
      // warp-uniform (the tensor-memory loads are warp-wide; with two threads
      // per row the same decision in both warps of the pair: the same rows)
      if (__any_sync(kFullMask, row_want)) {
        float mx = -INFINITY;
        if (lok) {
#pragma unroll
          for (int q4 = 0; q4 < HK / 32; ++q4) {
            uint32_t(&chunk)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * q4);
            tmem_ld32(tmem + lane_base + sb * kKeys + HK * hcol + 32 * q4, chunk);
          }
          tmem_wait_ld();
          if (masked) {
#pragma unroll
            for (int j = 0; j < HK; ++j)
              if (j > lim) sv[j] = __float_as_uint(-INFINITY);
          }
          // eight independent partial maxima (max is exact in any order)
          float m8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = __uint_as_float(sv[k]);
#pragma unroll
          for (int j = 8; j < HK; ++j) m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(sv[j]));
#pragma unroll
          for (int k = 0; k < 4; ++k) m8[k] = fmaxf(m8[k], m8[k + 4]);
          mx = fmaxf(fmaxf(m8[0], m8[2]), fmaxf(m8[1], m8[3]));
        }
        // the row's maximum over both halves; this buffer's previous reads
        // came before both threads' arrivals on this chunk's first barrier
        if constexpr (kRowThreads == 2) {
          float* redm = red + 6 * kRows;
          tc_fence_before();
          redm[hcol * kRows + r] = mx;
          pair_sync(warp);
          mx = fmaxf(redm[r], redm[kRows + r]);
          tc_fence_after();
        }
        mx *= sl2;
        if (lok) {
          if (mx != -INFINITY) {
            if (m_used == -INFINITY) {
              m_used = mx;
            } else if (mx > m_used + 8.f) {
              alpha = ex2(m_used - mx);
              m_used = mx;
            }
          }
          weights();  // the scores were read again: weights against the reference
        }
      }
      if (lok) {
        l_sum = l_sum * alpha + psum;
        // rescale this half of O's row when the reference maximum moved; PV(c-1)
        // (and so every earlier PV) must be done with O first (c == 0: the
        // first PV overwrites O)
        if (c > 0 && __any_sync(kFullMask, alpha != 1.f)) {
          lok = mbar_wait_bounded(&pv_done[(c - 1) % kSBuf], ((c - 1) / kSBuf) & 1, p.err);
          lok = __all_sync(kFullMask, lok);
          if (lok) {
            tc_fence_after();
#pragma unroll
            for (int q4 = 0; q4 < kOCols / 16; ++q4) {
              uint32_t o[16];
              tmem_ld16(tO + 16 * q4, o);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
              tmem_st16(tO + 16 * q4, o);
            }
          }
        }
      }
      if (lok) {
        // P into S[sb] as hi + lo bf16 parts, pairs packed: hi = p truncated to
        // bf16 (its upper 16 bits), lo = bf16(p - hi) (p - hi is exact and
        // below 2^-7 p, so hi + lo keeps p to ~2^-16)
#pragma unroll
        for (int q2 = 0; q2 < HK / 32; ++q2) {
          uint32_t wh[16], wl[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const uint32_t ua = sv[32 * q2 + 2 * k], ue = sv[32 * q2 + 2 * k + 1];
            wh[k] = __byte_perm(ua, ue, 0x7632);
            const float2 r2 = __fadd2_rn(
                make_float2(__uint_as_float(ua), __uint_as_float(ue)),
                make_float2(-__uint_as_float(ua & 0xFFFF0000u), -__uint_as_float(ue & 0xFFFF0000u)));
            const __nv_bfloat162 lo = __floats2bfloat162_rn(r2.x, r2.y);
            wl[k] = *reinterpret_cast<const uint32_t*>(&lo);
          }
          // over this thread's own S columns: hi pairs in the first half, lo
          // pairs in the second
          tmem_st16(tmem + lane_base + sb * kKeys + HK * hcol + 16 * q2, wh);
          tmem_st16(tmem + lane_base + sb * kKeys + HK * hcol + HK / 2 + 16 * q2, wl);
        }
        tmem_wait_st();
      }
      // V of the final chunk: keys past the last visible one may hold anything
      // (a partly filled block, or blocks not loaded); P is 0 there, but
      // 0 * NaN is not, so those rows are zeroed once the copies have landed.
      const int vk = nk - c * kKeys;  // valid keys in this chunk
      if (lok && vk < kKeys) {
        const int st = c % kStages;
        lok = mbar_wait_bounded(&v_full[st], (c / kStages) & 1, p.err);
        if (lok && r >= vk && r < kKeys) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int hh = hcol; hh < 2; hh += kRowThreads) {  // the 64-column halves
            uint4* row = reinterpret_cast<uint4*>(sm + kV + (2 * st + hh) * kKVHalf + prow);
#pragma unroll
            for (int k = 0; k < 8; ++k) row[k] = z;
          }
        }
      }
      ok = lok;
      // hand P, O and the zeroed V rows to the MMA warp: one arrival per warp
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[sb]);
    }

    // Epilogue: O / l, both halves' sums combined through shared memory, once
    // the last PV (and so every PV) is done.
    bool lok = ok && mbar_wait_bounded(&pv_done[(nchunks - 1) % kSBuf],
                                       ((nchunks - 1) / kSBuf) & 1, p.err);
    lok = __all_sync(kFullMask, lok);
    float lt = l_sum;
    if constexpr (kRowThreads == 2) {
      float* reds = red + 4 * kRows;  // not a buffer the loop's last reads may still use
      reds[hcol * kRows + r] = l_sum;
      asm volatile("bar.sync 5, %0;" ::"n"(kSoftmaxThreads) : "memory");
      lt = reds[r] + reds[kRows + r];
    }
    if (lok && shared_prefix) {
      // the row's partial: o / l, and (m, l) with m in natural-log units
      tc_fence_after();
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const size_t wrow =
          (static_cast<size_t>(row_ok ? qi : 0) * p.num_q_heads + kvh * G + r % G) *
              p.max_partitions + split;
      float* orow = p.ws_o + wrow * kD + kOCols * hcol;
#pragma unroll
      for (int q4 = 0; q4 < kOCols / 16; ++q4) {
        uint32_t o[16];
        tmem_ld16(tO + 16 * q4, o);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<float4*>(orow + 16 * q4 + 4 * k) = make_float4(
                __uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
        }
      }
      if (row_ok && hcol == 0) {
        p.ws_m[wrow] = m_used * 0.6931471805599453f;
        p.ws_l[wrow] = lt;
      }
    } else if (lok) {
      tc_fence_after();
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      __nv_bfloat16* orow = p.out +
                            (static_cast<size_t>(q0 + (row_ok ? qi : 0)) * p.num_q_heads +
                             kvh * G + r % G) * kD + kOCols * hcol;
#pragma unroll
      for (int q4 = 0; q4 < kOCols / 16; ++q4) {
        uint32_t o[16];
        tmem_ld16(tO + 16 * q4, o);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 h2 =
                  __floats2bfloat162_rn(__uint_as_float(o[8 * k + 2 * e]) * inv,
                                        __uint_as_float(o[8 * k + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(orow + 16 * q4 + 8 * k) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---- host side -------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// K or V pool as a 2-D bf16 tensor [num_blocks * Hkv * 16 rows][128], boxes of
// 16 rows x 64 columns, 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* base, int64_t rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, kBS};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// q as a 3-D bf16 tensor [T][Hq][128], boxes of (128 / G tokens) x G heads x
// 64 columns, 128-byte swizzle: one box is one 64-column half of a CTA's rows.
bool encode_q_map(CUtensorMap* map, const void* base, int total_q, int num_q_heads, int group) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_q_heads),
                              static_cast<cuuint64_t>(total_q)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                 static_cast<cuuint64_t>(num_q_heads) * kD * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group),
                             static_cast<cuuint32_t>(kRows / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int G>
cudaError_t launch_prefill_g(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const PrefillParams& p, int max_query_len, int num_seqs,
                             cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  auto kernel = paged_prefill_kernel<G>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(smem_set.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    smem_set.fetch_or(bit);
  }
  const int tiles = (max_query_len + kRows / G - 1) / (kRows / G);
  const dim3 grid(tiles, p.num_kv_heads, num_seqs);
  return launch_pdl(kernel, grid, dim3(kThreads), kSmemBytes, stream, tq, tk, tv, p);
}

bool aligned16(const void* ptr) { return ptr && (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

}  // namespace

// The shared-prefix partials of a decode batch (see PrefillParams): grid
// (query tiles, KV heads, splits).  Arguments checked by the caller.
cudaError_t launch_prefix_partials(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int num_blocks, float scale,
                                   int split_blocks, int splits, float* ws_o, float* ws_m,
                                   float* ws_l, int max_partitions, unsigned* err,
                                   cudaStream_t stream) {
  const int group = num_q_heads / num_kv_heads;
  const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * kBS;
  CUtensorMap tq, tk, tv;
  if (!encode_q_map(&tq, q, num_seqs, num_q_heads, group) ||
      !encode_pool_map(&tk, k_cache, rows) || !encode_pool_map(&tv, v_cache, rows))
    return cudaErrorInvalidValue;
  PrefillParams p{};
  p.block_tables = block_tables;
  p.err = err;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.total_q = num_seqs;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.split_blocks = split_blocks;
  p.ws_o = ws_o;
  p.ws_m = ws_m;
  p.ws_l = ws_l;
  p.max_partitions = max_partitions;
  p.context_lens = context_lens;
  switch (group) {
    case 1: return launch_prefill_g<1>(tq, tk, tv, p, num_seqs, splits, stream);
    case 2: return launch_prefill_g<2>(tq, tk, tv, p, num_seqs, splits, stream);
    case 4: return launch_prefill_g<4>(tq, tk, tv, p, num_seqs, splits, stream);
    default: return launch_prefill_g<8>(tq, tk, tv, p, num_seqs, splits, stream);
  }
}

}  // namespace pa

extern "C" int pa_prefill_supported(int head_dim, int group, int block_size) {
  return head_dim == 128 && block_size == 16 && (group == 1 || group == 2 || group == 4 ||
                                                  group == 8);
}

extern "C" pa_status pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, const int32_t* query_start_loc,
                                int max_query_len, int num_seqs, int total_query_tokens,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, float scale, pa_stream_t stream) {
  using namespace pa;
  if (num_seqs < 0 || max_query_len < 0 || total_query_tokens < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0 || !(scale > 0.f) || num_seqs > 65535)
    return PA_ERR_INVALID_ARG;
  const int group = num_q_heads / num_kv_heads;
  if (!pa_prefill_supported(head_dim, group, block_size)) return PA_ERR_UNSUPPORTED_SHAPE;
  if (num_seqs == 0 || max_query_len == 0 || total_query_tokens == 0) return PA_OK;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !block_tables || !context_lens || !query_start_loc)
    return PA_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * kBS;
  if (rows > 0x7fffffffll || static_cast<int64_t>(max_blocks_per_seq) * kBS > 0x7fffffffll)
    return PA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv;
  if (!encode_q_map(&tq, q, total_query_tokens, num_q_heads, group) ||
      !encode_pool_map(&tk, k_cache, rows) || !encode_pool_map(&tv, v_cache, rows))
    return cuda_fail(cudaErrorInvalidValue);  // tensor-map encoding refused the pools
  PrefillParams p{};
  p.out = static_cast<__nv_bfloat16*>(out);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start_loc;
  p.err = device_error_word();
  if (!p.err) return cuda_fail(cudaGetLastError());
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.total_q = total_query_tokens;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (group) {
    case 1: e = launch_prefill_g<1>(tq, tk, tv, p, max_query_len, num_seqs, s); break;
    case 2: e = launch_prefill_g<2>(tq, tk, tv, p, max_query_len, num_seqs, s); break;
    case 4: e = launch_prefill_g<4>(tq, tk, tv, p, max_query_len, num_seqs, s); break;
    default: e = launch_prefill_g<8>(tq, tk, tv, p, max_query_len, num_seqs, s); break;
  }
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}
