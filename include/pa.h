/*
 * pa.h -- C ABI of libpa.so: PagedAttention decode on GB300 (sm_103a).
 *
 * Two device operations make up the decode hot path, plus a host-side block
 * allocator that produces their index inputs:
 *
 *   pa_reshape_and_cache   write each new token's K and V into the block pool
 *   pa_decode              single-query grouped-query attention over each
 *                          sequence's blocks, found through its block table
 *   pa_decode_splitk       the same, one CTA per 512-token (configurable)
 *   pa_splitk_reduce       partition, then a log-sum-exp merge of partitions
 *   pa_decode_step         cache write + decode (+ merge) in one launch
 *   pa_copy_blocks         copy-on-write: copy shared blocks a branch writes into
 *   *_int8, *_fp8          the cache write and decode over an INT8 / FP8 KV cache
 *   pa_prefill             causal attention of chunks of new tokens (prefill)
 *   pa_alloc_*             fixed-size block allocator with reference counts,
 *                          copy-on-write and automatic prefix caching (host
 *                          only, never on the GPU path)
 *
 * Passages these follow (page title, section):
 *   [KV]   "How LLM Inference Serving Works: KV Cache, PagedAttention and
 *          Continuous Batching", section "What the KV Cache Is, and How Big It
 *          Gets" -- each decode step compares the new token's query with the
 *          keys of the earlier tokens and mixes their values; K and V are
 *          cached per token; 32 query heads share 8 KV heads (GQA).
 *   [PA]   same page, "PagedAttention: Virtual Memory for the KV Cache" --
 *          fixed-size blocks, a block table from logical to physical blocks,
 *          blocks allocated on demand, the attention kernel follows the table.
 *   [SH]   same page, "Sharing comes for free" -- blocks shared by several
 *          tables with reference counts, copied only when a branch writes.
 *   [LIFE] same page, "Putting It Together: The Life of a Request in vLLM" --
 *          each decode step appends one token's K and V into the request's
 *          current block; a new block only when that block fills; counts
 *          drop when the request ends.
 *   [OOM]  same page, "When memory runs out anyway" -- when blocks run out
 *          the engine preempts a request.
 *   [PFX]  same page, "Prefix Caching and Chunked Prefill" -- blocks named
 *          by a hash of their tokens and the prefix before them are reused
 *          by later prompts; unused cached blocks are evicted in LRU order.
 *   [WALK] "LLM serving (vLLM, quantized inference): Visual walkthrough",
 *          Steps 7-8 -- block_size 16, at most block_size-1 slots wasted,
 *          shared prefixes stored once.
 *
 * Conventions shared by every device entry point:
 *   - Pointers named *_cache, q, out, key, value, ws_* and the index arrays
 *     are DEVICE pointers owned by the caller.  The library allocates no
 *     device memory on these paths and keeps no pointer after returning.
 *   - Element types: K/V/q/out/key/value are bf16 (2 bytes, stored as raw
 *     bits); the split-K workspace is fp32; block tables and context lengths
 *     are int32; slots are int64.
 *   - Layouts (row-major, contiguous):
 *       k_cache, v_cache : [num_blocks, num_kv_heads, block_size, head_dim]
 *       q, out           : [num_seqs, num_q_heads, head_dim]
 *       key, value       : [num_tokens, num_kv_heads, head_dim]
 *       slot_mapping     : [num_tokens]; slot = block * block_size + offset;
 *                          a negative slot means "skip this token"
 *       block_tables     : [num_seqs, max_blocks_per_seq]; entry j of row b
 *                          is the physical block holding tokens
 *                          [j*block_size, (j+1)*block_size) of sequence b
 *       context_lens     : [num_seqs]; tokens attended by sequence b, i.e.
 *                          positions [0, context_lens[b]) (the new token,
 *                          written first by pa_reshape_and_cache, included)
 *     Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - Alignment: bf16 and fp32 arrays 16-byte aligned; int32 arrays 4-byte;
 *     int64 arrays 8-byte.  A misaligned pointer is PA_ERR_INVALID_ARG.
 *   - All work is enqueued asynchronously on `stream`; a return of PA_OK
 *     means the launch was accepted, not that the kernel has finished.
 *   - Arguments are checked on the host before any launch.  Values that
 *     live in device memory (block ids, context lengths, slots) are checked
 *     by the kernels: an out-of-range value sets a bit in a per-device error
 *     word (pa_get_device_error) and is never dereferenced -- a bad block id
 *     reads block 0 instead, a bad slot is not written, a context length
 *     beyond max_blocks_per_seq * block_size is clamped.  Kernels never trap.
 *   - No C++ exception crosses this ABI.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* pa_stream_t;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,       /* null / misaligned pointer, bad size, unknown sequence */
  PA_ERR_UNSUPPORTED_SHAPE = 2, /* a (head_dim, group, block_size) with no compiled kernel */
  PA_ERR_OUT_OF_BLOCKS = 3,     /* allocator: too few free blocks; state unchanged */
  PA_ERR_CUDA = 4               /* a CUDA runtime call or launch failed */
} pa_status;

/* Bits of the per-device error word written by the kernels. */
#define PA_DEVERR_BLOCK_ID 0x1u     /* block table entry outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT_LEN 0x2u  /* context length < 0 or > max_blocks_per_seq*block_size */
#define PA_DEVERR_SLOT 0x4u         /* slot >= num_blocks * block_size */
#define PA_DEVERR_WAIT_TIMEOUT 0x8u /* an asynchronous copy did not complete in time */
#define PA_DEVERR_ORDER 0x10u       /* a work-order entry outside [0, num_seqs * max_partitions) */
#define PA_DEVERR_PREFIX 0x20u      /* a sequence does not hold the shared prefix it was given */

/* Static description of a status code; never NULL. */
const char* pa_status_string(pa_status status);

/* Text of the last CUDA error seen by this thread inside the library
 * ("" if none).  Valid until the next call from the same thread. */
const char* pa_last_cuda_error(void);

/* Reads the error word of the current device into *bits (0 = no error).
 * Synchronises the device.  PA_ERR_INVALID_ARG if bits is NULL. */
pa_status pa_get_device_error(unsigned* bits);

/* Resets the current device's error word to 0 (synchronous). */
pa_status pa_clear_device_error(void);

/* PA_OK if pa_decode / pa_decode_splitk have a kernel for this shape:
 * block_size 16, head_dim in {64, 128}, num_q_heads / num_kv_heads in
 * {2, 4, 8}; otherwise PA_ERR_UNSUPPORTED_SHAPE (or PA_ERR_INVALID_ARG for
 * non-positive or non-divisible values). */
pa_status pa_decode_supported(int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size);

/*
 * Cache write [KV], [LIFE]: for every t in [0, num_tokens) with
 * s = slot_mapping[t] >= 0,
 *   k_cache[s / block_size, h, s % block_size, :] = key[t, h, :]
 *   v_cache[s / block_size, h, s % block_size, :] = value[t, h, :]
 * for every KV head h.  A bit copy.  Slots must be distinct (two tokens
 * writing one slot race).  head_dim must be a multiple of 8; num_tokens == 0
 * is a no-op.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value,
                               void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int num_tokens,
                               int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, pa_stream_t stream);

/*
 * Copy-on-write block copy [SH]: for every pair i, with src = block_mapping[2i]
 * and dst = block_mapping[2i + 1] (device int64 [num_pairs, 2]), copies the
 * whole block in the K pool and the V pool of every layer:
 *   k_caches[l][dst, :, :, :] = k_caches[l][src, :, :, :]  (and V), l < num_layers.
 * k_caches / v_caches are HOST arrays of num_layers device pointers, each a
 * pool [num_blocks, num_kv_heads, block_size, head_dim] bf16.  These are the
 * (cow_src, cow_dst) pairs pa_alloc_append_slot(s) report; copying the whole
 * block is a superset of the rows the new owner needs.  No destination may
 * appear twice or also as a source (such copies race).  Ids outside
 * [0, num_blocks) set PA_DEVERR_BLOCK_ID and the pair is skipped; src == dst
 * is a no-op.  num_pairs == 0 or num_layers == 0 is a no-op.
 */
pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                         const int64_t* block_mapping, int num_pairs,
                         int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, pa_stream_t stream);

/*
 * Paged decode attention [KV], [PA]: for every sequence b and query head h
 * (g = h / (num_q_heads / num_kv_heads), n = context_lens[b]),
 *   s_j   = scale * dot(q[b, h, :], K_j),   K_j = k_cache[tbl(j), g, j % bs, :]
 *   out[b, h, :] = sum_j softmax(s)_j * V_j over j in [0, n),
 * with tbl(j) = block_tables[b * max_blocks_per_seq + j / bs], fp32
 * accumulation, bf16 output rounded to nearest even.  n == 0 gives zeros.
 * One CTA per (sequence, KV head) reads each K/V block once for all the
 * query heads of its group.  No workspace.
 */
pa_status pa_decode(void* out, const void* q, const void* k_cache,
                    const void* v_cache, const int32_t* block_tables,
                    int max_blocks_per_seq, const int32_t* context_lens,
                    int num_seqs, int num_q_heads, int num_kv_heads,
                    int head_dim, int block_size, int num_blocks, float scale,
                    pa_stream_t stream);

/*
 * INT8 KV cache (quantised KV; "Visual walkthrough", Step 1: one stored number
 * costs p = 2 bytes in FP16/BF16, 1 byte in INT8).  The pages give no scaling
 * scheme; here every (token, KV head) row is quantised symmetrically with its
 * own fp32 scale, so a token is written once and never re-quantised:
 *   scale = max|x| / 127,  code = clamp(round_half_even(x / scale), -127, 127)
 * (fp32 arithmetic; scale 0 and codes 0 for an all-zero row).  Pools:
 *   k_cache, v_cache   : [num_blocks, num_kv_heads, block_size, head_dim] int8
 *   k_scales, v_scales : [num_blocks, num_kv_heads, block_size] fp32
 * 2 * (head_dim + 4) bytes per token and KV head instead of 4 * head_dim.
 * k_cache is plain row-major.  v_cache holds each (block, head) tile of
 * 16 * D bytes (D = head_dim) transposed, for the decode's tensor-core PV:
 * the code of token t (0..15) and dim d sits at byte
 *   L * (D / 2) + 16 * ((w / 4) XOR f) + 4 * (w % 4) + y
 * of the tile, with r = d % 16, L = 4 * (r % 8) + (t % 8) / 2,
 * w = 2 * (d / 16) + r / 8, y = (t % 2) + 2 * (t / 8), and
 * f = (L / 2) % 4 for D = 128, (L / 4) % 2 for D = 64; and an INT8 V byte is
 * the code plus 128 (offset binary: uint8 0..254 for codes -127..127).  Lane L
 * of a decoding warp then finds, in one 32-bit word per dim it feeds to the
 * MMA, that dim's codes of the 4 tokens it feeds, with no shared-memory bank
 * conflicts.  Whole-block copies (pa_copy_blocks) are unaffected.
 * Decode quantises each query head the same way and takes QK as an integer
 * dot product, s_j = scale * scale_q * k_scale_j * sum_d q_code_d * k_code_jd
 * (exact in int32); PV weights w_j = softmax weight j * v_scale_j mix the V
 * codes on the tensor cores with fp32 accumulation (each weight, divided by
 * a power of two bounding the V scales seen so far, carried as an f16 hi part
 * plus an f16 lo part, ~2^-22 relative).  head_dim 64 or 128; otherwise as
 * the bf16 calls.
 */
pa_status pa_reshape_and_cache_int8(const void* key, const void* value,
                                    int8_t* k_cache, int8_t* v_cache,
                                    float* k_scales, float* v_scales,
                                    const int64_t* slot_mapping, int num_tokens,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, pa_stream_t stream);
pa_status pa_decode_int8(void* out, const void* q, const int8_t* k_cache,
                         const int8_t* v_cache, const float* k_scales,
                         const float* v_scales, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* context_lens,
                         int num_seqs, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, float scale,
                         pa_stream_t stream);
/* Split-K partition pass over an INT8 cache; merge with pa_splitk_reduce. */
pa_status pa_decode_splitk_int8(float* ws_out, float* ws_m, float* ws_l,
                                int max_partitions, const void* q,
                                const int8_t* k_cache, const int8_t* v_cache,
                                const float* k_scales, const float* v_scales,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, float scale,
                                int partition_size, pa_stream_t stream);

/*
 * FP8 KV cache (the other 1-byte format of "Visual walkthrough", Step 1).  The
 * pages give no scheme; here E4M3 as NVIDIA's FP8 "e4m3" (bias 7, 3 mantissa
 * bits, no infinities, 0x7F / 0xFF NaN, largest finite 448), one fp32 scale per
 * (token, KV head) row:
 *   scale = max|x| / 448,  code = E4M3(x / scale) round to nearest even,
 *   saturated to +-448 (fp32 arithmetic; scale 0 and codes 0 for an all-zero row).
 * Pools, scales, the transposed V tile and sizes exactly as the INT8 cache,
 * with uint8 codes (V codes stored as they are, not offset).  Decode keeps q
 * unquantised: scores are scale * q . (decode(k_code) * k_scale) with fp32
 * accumulation, taken on the tensor cores in E4M3 with each query head, times
 * a power of two, split into two E4M3 parts q1 + 2^-5 q2 (exact for bf16 q up
 * to about 2^-21 of the head's largest |q|); PV as the INT8 decode (weights times
 * v_scale, f16 hi + lo on the tensor cores, exact codes).  A token past the
 * context is masked by position; its codes may be NaN and are never
 * multiplied.  head_dim 64 or 128.
 */
pa_status pa_reshape_and_cache_fp8(const void* key, const void* value,
                                   uint8_t* k_cache, uint8_t* v_cache,
                                   float* k_scales, float* v_scales,
                                   const int64_t* slot_mapping, int num_tokens,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int num_blocks, pa_stream_t stream);
pa_status pa_decode_fp8(void* out, const void* q, const uint8_t* k_cache,
                        const uint8_t* v_cache, const float* k_scales,
                        const float* v_scales, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens,
                        int num_seqs, int num_q_heads, int num_kv_heads,
                        int head_dim, int block_size, int num_blocks, float scale,
                        pa_stream_t stream);
/* Split-K partition pass over an FP8 cache; merge with pa_splitk_reduce. */
pa_status pa_decode_splitk_fp8(float* ws_out, float* ws_m, float* ws_l,
                               int max_partitions, const void* q,
                               const uint8_t* k_cache, const uint8_t* v_cache,
                               const float* k_scales, const float* v_scales,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, float scale,
                               int partition_size, pa_stream_t stream);

/* Bytes of fp32 workspace pa_decode_splitk needs for contexts up to
 * max_context_len: ws_out [B, Hq, P, D] + ws_m [B, Hq, P] + ws_l [B, Hq, P]
 * with P = ceil(max_context_len / partition_size).  0 on invalid input. */
size_t pa_splitk_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                 int max_context_len, int partition_size);

/*
 * Split-K partition pass: the decode above restricted to partition p, i.e.
 * tokens [p * partition_size, min(n, (p + 1) * partition_size)), for every
 * p < ceil(n / partition_size).  Writes, at index [b, h, p] (row stride
 * max_partitions):
 *   ws_m  = max_j s_j                       (natural-log units)
 *   ws_l  = sum_j exp(s_j - ws_m)
 *   ws_out[.., :] = sum_j exp(s_j - ws_m) * V_j / ws_l
 * Partitions at or beyond ceil(n / partition_size) are not written.
 * partition_size must be a positive multiple of block_size, and every
 * context length must satisfy ceil(n / partition_size) <= max_partitions
 * (else PA_DEVERR_CONTEXT_LEN and the excess is dropped).
 */
pa_status pa_decode_splitk(float* ws_out, float* ws_m, float* ws_l,
                           int max_partitions, const void* q,
                           const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int num_blocks, float scale,
                           int partition_size, pa_stream_t stream);

/*
 * Log-sum-exp merge of the partitions written by pa_decode_splitk:
 *   M = max_p ws_m[b,h,p],  w_p = ws_l[b,h,p] * exp(ws_m[b,h,p] - M),
 *   out[b, h, :] = sum_p w_p * ws_out[b,h,p,:] / sum_p w_p   (bf16),
 * over p < ceil(context_lens[b] / partition_size); zeros if n == 0.
 * Arguments must match the pa_decode_splitk call that filled the workspace.
 */
pa_status pa_splitk_reduce(void* out, const float* ws_out, const float* ws_m,
                           const float* ws_l, int max_partitions,
                           const int32_t* context_lens, int num_seqs,
                           int num_q_heads, int head_dim, int partition_size,
                           pa_stream_t stream);

/*
 * Split-K decode with no allocation.  The pages have no counterpart to this
 * entry point: it exists for callers that cannot call cudaMalloc -- serving
 * runtimes that reserve all device memory up front for their own pools, and
 * latency-critical threads that must not take the device synchronisation an
 * allocation can imply.  It computes exactly pa_decode_splitk followed by
 * pa_splitk_reduce (same kernels, same results), but their fp32 workspace is
 * a fixed array of PA_DECODE_NOALLOC_WORKSPACE_BYTES compiled into the
 * library, resident on every GPU that loads it until the process exits.
 *   max_context_len: an upper bound on every context_lens[b] (host value);
 *   the workspace holds B * Hq * P rows of (head_dim + 2) floats with
 *   P = ceil(max_context_len / partition_size).  A call needing more than
 *   PA_DECODE_NOALLOC_WORKSPACE_BYTES (or P > 65535) returns
 *   PA_ERR_INVALID_ARG before any launch.  A context longer than
 *   max_context_len sets PA_DEVERR_CONTEXT_LEN and its excess is dropped.
 * Calls no cudaMalloc / cudaFree.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  All calls share the one
 * array: calls whose kernels overlap on the GPU (other streams, other
 * threads) race on it.  Nothing in it needs to start at zero; it keeps the
 * last call's partials.
 */
#define PA_DECODE_NOALLOC_WORKSPACE_BYTES ((size_t)8 << 20)
pa_status pa_decode_splitk_noalloc(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, int num_blocks,
                                   float scale, int partition_size, int max_context_len,
                                   pa_stream_t stream);

/*
 * Fused decode step [LIFE], [KV], [PA]: each sequence's new token written
 * into the cache and every query attended, in ONE kernel launch.  Computes
 * exactly what
 *   pa_reshape_and_cache(key, value, ..., slot_mapping, num_tokens = num_seqs)
 * followed by pa_decode (partition_size == 0) or by pa_decode_splitk +
 * pa_splitk_reduce (partition_size > 0) compute, under one condition on the
 * slots: slot_mapping[b] (device int64 [num_seqs]) is negative (nothing to
 * write) or the slot of position n - 1 of sequence b, n = context_lens[b],
 *   block_tables[b][(n - 1) / block_size] * block_size + (n - 1) % block_size,
 * i.e. the new token is the last one its own query attends to, as in a
 * decode step.  The CTA that reads that position writes the row first; a slot
 * that is not that position's (or n == 0 with a slot >= 0) is not written and
 * sets PA_DEVERR_SLOT, since another CTA could be reading it.
 *   key, value: device bf16 [num_seqs, num_kv_heads, head_dim], one new token
 *     per sequence; key, value and slot_mapping are all NULL to skip the
 *     write (attention only).
 *   partition_size == 0: one CTA per (sequence, KV head); ws_* / counters /
 *     max_partitions are ignored (may be NULL / 0).
 *   partition_size > 0: split-K as pa_decode_splitk (same workspace and
 *     limits).  With max_partitions <= 16 the partitions are merged inside
 *     the same launch (the last CTA of each (sequence, KV head) to finish
 *     merges them; a sequence with one partition writes out directly); with
 *     more, the merge is a second launch, as pa_splitk_reduce.  counters:
 *     device uint32 [num_seqs * num_kv_heads], all zero before the first call;
 *     each call leaves them zero again, unless it sets PA_DEVERR_WAIT_TIMEOUT
 *     or PA_DEVERR_ORDER: then a (sequence, KV head) may have missed an
 *     arrival and its counter stays nonzero, and the next call with those
 *     counters would merge before all partitions are written -- zero them
 *     before the next call.  Concurrent calls must not share counters or
 *     workspace.
 *   order (split-K only, may be NULL): device int32 [num_seqs * max_partitions],
 *     a permutation of the items item = part * num_seqs + b, the order in
 *     which the block scheduler receives the (sequence, partition) CTAs
 *     (pa_splitk_order gives the longest first).  Every item runs whatever the
 *     order, so an order made for other context lengths only costs speed; an
 *     entry outside the range sets PA_DEVERR_ORDER and that CTA does nothing
 *     (its item is then missing: a non-permutation gives wrong results).
 *     num_seqs * max_partitions <= 65535 (else PA_ERR_UNSUPPORTED_SHAPE).
 *   flags: 0, or PA_STEP_EARLY_READ: the caller promises that block_tables,
 *     context_lens, order and the pools (and scales) are not written by the
 *     kernel launched just before this one on the stream (in a model, that
 *     kernel writes q and the new K/V, never these).  The launch then reads
 *     them -- the first block ids and the first K/V tiles -- before waiting
 *     for that kernel (programmatic dependent launch), overlapping its start
 *     with the previous kernel's end; q, key, value and slot_mapping are read,
 *     and anything is written, only after the wait.  Other bits:
 *     PA_ERR_INVALID_ARG.
 * Pools, scales and other arguments as pa_decode / pa_decode_splitk and the
 * _int8 / _fp8 cache writes (the 1-byte variants quantise the new rows by the
 * same rule, bit-identically).
 */
#define PA_STEP_EARLY_READ 0x1
pa_status pa_decode_step(void* out, const void* q, const void* key, const void* value,
                         const int64_t* slot_mapping, void* k_cache, void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         float scale, int partition_size, float* ws_out, float* ws_m,
                         float* ws_l, unsigned* counters, int max_partitions,
                         const int32_t* order, int flags, pa_stream_t stream);
pa_status pa_decode_step_int8(void* out, const void* q, const void* key, const void* value,
                              const int64_t* slot_mapping, int8_t* k_cache, int8_t* v_cache,
                              float* k_scales, float* v_scales, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, float scale, int partition_size, float* ws_out,
                              float* ws_m, float* ws_l, unsigned* counters, int max_partitions,
                              const int32_t* order, int flags, pa_stream_t stream);
pa_status pa_decode_step_fp8(void* out, const void* q, const void* key, const void* value,
                             const int64_t* slot_mapping, uint8_t* k_cache, uint8_t* v_cache,
                             float* k_scales, float* v_scales, const int32_t* block_tables,
                             int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, float scale, int partition_size, float* ws_out,
                             float* ws_m, float* ws_l, unsigned* counters, int max_partitions,
                             const int32_t* order, int flags, pa_stream_t stream);

/*
 * Fused decode step of a batch sharing a prefix [SH], [WALK] Step 8: every
 * sequence's first prefix_len tokens are the same blocks (block_tables[b][j]
 * == block_tables[0][j] for j < prefix_len / block_size, e.g. forks of one
 * prompt) and its context goes past them (context_lens[b] > prefix_len).
 * Computes what pa_decode_step computes (the new tokens' cache write, then
 * attention) but reads the prefix's K/V once per KV head for the whole batch
 * instead of once per sequence.  Two launches: (1) the prefix in partitions
 * of prefix_split tokens, each one tensor-core pass in which the queries of
 * all sequences and heads of a KV group attend to that partition's keys
 * together (the chunked-prefill kernel without a causal mask), writing
 * split-K partials to workspace partitions 0 .. prefix_len / prefix_split -
 * 1; (2) the split-K decode with the cache write over the rest of each
 * context, in partitions of partition_size tokens from the prefix's end
 * (workspace partitions from prefix_len / prefix_split on), overlapping (1)
 * and merging all of a sequence's partitions in its last CTA (counters as
 * pa_decode_step's).  A sequence whose table does not hold the prefix, or
 * whose context does not go past it, sets PA_DEVERR_PREFIX (its output is
 * then wrong).
 *   prefix_split: a multiple of block_size dividing prefix_len;
 *   partition_size: a multiple of block_size; workspace as pa_decode_splitk's
 *   with max_partitions > prefix_len / prefix_split and at least
 *   prefix_len / prefix_split + ceil((context_lens[b] - prefix_len) /
 *   partition_size) for every b (else PA_DEVERR_CONTEXT_LEN).
 *   order (may be NULL): the work order of launch (2)'s CTAs, device int32
 *     [num_seqs * (max_partitions - prefix_len / prefix_split)], a
 *     permutation of its items item = part * num_seqs + b over the
 *     partitions past the prefix (pa_splitk_order of the lengths past the
 *     prefix gives the longest first); as pa_decode_step's order otherwise.
 *   bf16 cache, head_dim and group supported by both pa_decode_supported
 *     and pa_prefill_supported (else PA_ERR_UNSUPPORTED_SHAPE); scale > 0,
 *     as pa_prefill's (else PA_ERR_INVALID_ARG); other
 *     arguments as pa_decode_step (key / value / slot_mapping all NULL:
 *     attention only).
 * Asynchronous on `stream`.
 */
pa_status pa_decode_step_shared_prefix(void* out, const void* q, const void* key,
                                       const void* value, const int64_t* slot_mapping,
                                       void* k_cache, void* v_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int num_blocks, float scale,
                                       int prefix_len, int prefix_split, int partition_size,
                                       float* ws_out, float* ws_m, float* ws_l,
                                       unsigned* counters, int max_partitions,
                                       const int32_t* order, pa_stream_t stream);

/*
 * Paged (chunked) prefill attention ("How LLM Inference Serving Works",
 * sections "Two Phases: Prefill and Decode" and "Chunked prefill"; paging as
 * in [PA]).  Each sequence b contributes a chunk of n_b new tokens, whose
 * K/V the caller has already written into the cache (pa_reshape_and_cache);
 * with ctx_b = context_lens[b] (chunk included) the chunk holds positions
 * ctx_b - n_b .. ctx_b - 1, and the query at position p attends to keys
 * 0 .. p (causal; n_b = 1 is one decode step).
 *   q, out            : [T, Hq, head_dim] bf16, the chunks back to back;
 *                       T = total_query_tokens.
 *   query_start_loc   : [num_seqs + 1] int32 (device), sequence b's rows are
 *                       query_start_loc[b] .. query_start_loc[b+1] - 1.
 *   max_query_len     : host bound on every n_b (sizes the grid; longer
 *                       chunks are cut at it).
 *   k_cache, v_cache, block_tables, context_lens: as pa_decode.
 * Runs on the tensor cores (tcgen05, bf16 in, fp32 accumulate; the softmax
 * weights P enter the PV product as two bf16 parts, hi = P truncated to bf16
 * and lo = bf16(P - hi), one MMA each, so they keep about 16 bits).  head_dim 128, block_size 16, Hq / Hkv in
 * {1, 2, 4, 8} (else PA_ERR_UNSUPPORTED_SHAPE); num_seqs <= 65535.  Device-side
 * checks: 0 <= n_b <= ctx_b <= max_blocks_per_seq * 16 and rows within T (else
 * PA_DEVERR_CONTEXT_LEN and the sequence is skipped); bad block ids as
 * pa_decode.  Pointers 16-byte aligned.  scale > 0 (the kernel takes row
 * maxima of the unscaled scores; else PA_ERR_INVALID_ARG).  Async on
 * `stream`.
 */
int pa_prefill_supported(int head_dim, int group, int block_size);
pa_status pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, const int32_t* query_start_loc,
                     int max_query_len, int num_seqs, int total_query_tokens,
                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                     int num_blocks, float scale, pa_stream_t stream);

/*
 * Split-K partition size for a decode batch (host): the size, from {256, 384,
 * 512, 640, 768, 1024, 1280, 1536, 1792, 2048, 4096} tokens, that minimises a
 * model of the split-K launch's time -- its CTAs handed in grid order to the first free
 * CTA slot (num_sms x the kernel's CTAs per SM), each costing a time per
 * token, a fixed start-up and, for sequences of several partitions, a merge
 * share -- with ties going to the larger size; in grid order a 1-byte cache
 * (issue-bound kernels) whose batch has fewer (sequence, KV head) units than
 * CTA slots takes 512.  context_lens: host int32
 * [num_seqs]; kv_kind 0 = bf16 cache, 1 = INT8, 2 = FP8; num_sms the device's
 * multiprocessor count; ordered != 0 models the launch with the
 * longest-first order of pa_splitk_order, 0 the plain grid order.  Returns 0
 * on invalid arguments.  The result is a
 * performance choice only: any partition size gives the same attention.
 */
int pa_splitk_partition_size(const int32_t* context_lens, int num_seqs, int num_q_heads,
                             int num_kv_heads, int head_dim, int kv_kind, int num_sms,
                             int ordered);

/*
 * Longest-first work order for a split-K pa_decode_step (host): fills
 * order_out[0 .. num_seqs * max_partitions) with the items
 * item = part * num_seqs + b sorted by the tokens each covers,
 * min(partition_size, max(0, context_lens[b] - part * partition_size)), most
 * first, ties in item order.  Returns the item count, or -1 on invalid
 * arguments (including num_seqs * max_partitions > 65535).
 */
int pa_splitk_order(const int32_t* context_lens, int num_seqs, int partition_size,
                    int max_partitions, int32_t* order_out);

/*
 * Step planning for chunked prefill (host; "How LLM Inference Serving Works",
 * section "Chunked prefill").  Each step has a token budget
 * (max_num_batched_tokens): every pending decode (one token each) is taken
 * first, the remaining budget goes to the pending prefills in queue order, and
 * a prefill that does not fit is cut to what is left.  With more decodes than
 * the budget, the first `budget` decodes run and no prefill does.
 *   prefill_remaining[i]: tokens still to prefill for queued request i;
 *   chunk_out[i]: tokens of request i scheduled this step (0: none);
 *   *decodes_out: decodes scheduled.
 * PA_ERR_INVALID_ARG on a negative count or a missing pointer.
 */
pa_status pa_plan_step(int budget, int num_decodes, const int32_t* prefill_remaining,
                       int num_prefills, int32_t* chunk_out, int* decodes_out);

/* ------------------------------------------------------------------------ */
/* Host block allocator [PA], [SH], [LIFE], [OOM], [WALK].  Not thread-safe;
 * one allocator per caller thread or external locking.  Deterministic: the
 * free list is first-in first-out, seeded with initial_free_order (NULL means
 * 0, 1, ..., num_blocks-1); a sequence's freed blocks go to the tail in its
 * logical order.  Every call that fails leaves the allocator unchanged.
 * Slot of position pos of a sequence: table[pos / bs] * bs + pos % bs. */
typedef struct pa_alloc pa_alloc;

/* Creates an allocator over num_blocks blocks of block_size tokens.
 * initial_free_order, if not NULL, must be a permutation of [0, num_blocks). */
pa_status pa_alloc_create(int num_blocks, int block_size,
                          const int32_t* initial_free_order, pa_alloc** out);
void pa_alloc_destroy(pa_alloc* a);

/* Registers an empty sequence.  PA_ERR_INVALID_ARG if seq_id exists. */
pa_status pa_alloc_add_seq(pa_alloc* a, int seq_id);

/* Appends one token.  *slot_out receives its slot.  A new block is taken
 * when the token opens a block; when it lands in a partly filled block
 * shared with another sequence (reference count > 1), the sequence moves to
 * a fresh block first and *cow_src / *cow_dst receive the (old, new) block
 * ids, whose first pos % bs token rows the caller must copy; otherwise both
 * are -1.  cow_src / cow_dst may be NULL.  PA_ERR_OUT_OF_BLOCKS if a block is
 * needed and none is free. */
pa_status pa_alloc_append_slot(pa_alloc* a, int seq_id, int64_t* slot_out,
                               int32_t* cow_src, int32_t* cow_dst);

/* One append for each of n distinct sequences, all or nothing: slots_out[i],
 * cow_src[i], cow_dst[i] as pa_alloc_append_slot for seq_ids[i]
 * (cow arrays may be NULL). */
pa_status pa_alloc_append_slots(pa_alloc* a, const int* seq_ids, int n,
                                int64_t* slots_out, int32_t* cow_src,
                                int32_t* cow_dst);

/* Appends num_tokens tokens to one sequence, all or nothing (a prompt).
 * Only the first append can need a copy; its pair goes to cow_src/cow_dst. */
pa_status pa_alloc_reserve(pa_alloc* a, int seq_id, int num_tokens,
                           int32_t* cow_src, int32_t* cow_dst);

/* child_id becomes a copy of parent_id sharing all its blocks (+1 reference
 * each).  PA_ERR_INVALID_ARG if parent is unknown or child exists. */
pa_status pa_alloc_fork(pa_alloc* a, int parent_id, int child_id);

/* Drops the sequence; blocks whose count reaches 0 return to the free tail. */
pa_status pa_alloc_free_seq(pa_alloc* a, int seq_id);

/* Copies the sequence's block table (its first min(cap, length) entries) to
 * out and its length to *n_out.  out may be NULL when cap == 0. */
pa_status pa_alloc_block_table(const pa_alloc* a, int seq_id, int32_t* out,
                               int cap, int* n_out);

/* Fills a padded table [n, max_blocks] (entries past a sequence's length are
 * -1) and, if ctx_out is not NULL, its token count per sequence.
 * PA_ERR_INVALID_ARG if a table is longer than max_blocks. */
pa_status pa_alloc_block_tables(const pa_alloc* a, const int* seq_ids, int n,
                                int32_t* out, int max_blocks, int32_t* ctx_out);

/* Tokens held by a sequence, or -1 if unknown. */
int64_t pa_alloc_seq_len(const pa_alloc* a, int seq_id);
/* Reference count of a block, or -1 if out of range. */
int pa_alloc_refcount(const pa_alloc* a, int block);
int pa_alloc_num_free(const pa_alloc* a);
int pa_alloc_num_blocks(const pa_alloc* a);
/* Copies the free list, head first (at most cap entries); *n_out = its size. */
pa_status pa_alloc_free_list(const pa_alloc* a, int32_t* out, int cap, int* n_out);
/* Empty slots in the sequence's last block, or -1 if unknown [WALK]. */
int pa_alloc_tail_waste(const pa_alloc* a, int seq_id);

/* ------------------------------------------------------------------------ */
/* Automatic prefix caching [PFX] ("How LLM Inference Serving Works",
 * section "Prefix Caching and Chunked Prefill", and "Putting It Together":
 * blocks become cached-but-evictable when their counts drop).  Every full
 * block of a prompt is named by a chained hash of the tokens in it and of
 * all tokens before it; a table maps names to physical blocks, so a prompt
 * reuses the blocks of the longest cached prefix, and a block matches only
 * if the whole prefix up to it is identical.  The pages fix no hash; here a
 * block's name is SHA-256(parent name || its tokens as little-endian int32),
 * the first block's parent being 32 zero bytes, or SHA-256(cache_salt) when
 * the request carries a salt (so tenants with different salts never share).
 * A named block whose count reaches 0 is kept, cached-but-evictable, in
 * least-recently-used order; fresh blocks come from the free list first and
 * then by evicting the least recently used cached block (its name is
 * dropped).  Only prompt blocks are named; blocks filled by later appends
 * are not. */

/* Turns prefix caching on; only while the allocator holds no sequence. */
pa_status pa_alloc_enable_prefix_cache(pa_alloc* a);

/* Registers seq_id with a prompt of num_tokens tokens: the longest cached
 * prefix of whole blocks is shared (+1 reference each), the rest of the
 * prompt gets fresh blocks, and the prompt's new full blocks are named.
 * *cached_tokens (may be NULL) receives how many leading tokens already
 * have their K/V in the cache (a multiple of block_size); the caller
 * computes the rest.  salt / salt_len: optional per-request cache salt
 * (salt_len 0: none).  PA_ERR_OUT_OF_BLOCKS (state unchanged) if the free
 * and evictable blocks cannot hold the uncached part; PA_ERR_INVALID_ARG if
 * prefix caching is off or seq_id exists. */
pa_status pa_alloc_add_seq_prompt(pa_alloc* a, int seq_id, const int32_t* tokens,
                                  int num_tokens, const void* salt, int salt_len,
                                  int* cached_tokens);

/* Number of cached-but-evictable blocks (-1 if a is NULL). */
int pa_alloc_num_evictable(const pa_alloc* a);

/* Copies the cached-but-evictable blocks, least recently used first. */
pa_status pa_alloc_evictable_list(const pa_alloc* a, int32_t* out, int cap, int* n_out);

/* The names used above, exposed for callers that keep their own index:
 * out[32] = the first block's parent name for this salt (salt_len 0: none). */
pa_status pa_prefix_root_hash(const void* salt, int salt_len, uint8_t* out);
/* out[32] = SHA-256(parent[32] || tokens as little-endian int32). */
pa_status pa_prefix_block_hash(const uint8_t* parent, const int32_t* tokens, int num_tokens,
                               uint8_t* out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
