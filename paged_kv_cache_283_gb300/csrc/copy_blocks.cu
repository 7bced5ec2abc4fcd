// Copy-on-write block copy (pa_copy_blocks).
//
// "How LLM Inference Serving Works" (dev.to), section "Sharing comes for
// free": blocks are shared between sequences with reference counts and a
// block is copied only when one branch needs to write into it.  The host
// allocator (allocator.cpp) decides when: an append into a shared, partly
// filled last block moves the writer onto a fresh block and reports the
// (source, destination) pair; this kernel then copies the source block's K
// and V, in every layer, into the destination.
//
// Pure data movement: one CTA per (pair, layer, K or V) streams one whole
// block (Hkv * bs * D bf16 = 32 KiB at the Llama-8B shape) with 16-byte
// loads and stores, four in flight per thread.

#include <cuda_runtime.h>
#include <stdint.h>

#include "device.cuh"
#include "internal.h"

namespace pa {

namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyBlocksParams p) {
  griddep_wait();  // the producer of the pools / mapping is complete
  griddep_launch_dependents();
  const int pair = blockIdx.x;
  const int layer = blockIdx.y;
  const bool is_v = blockIdx.z != 0;
  const int64_t src = __ldg(p.block_mapping + 2 * static_cast<int64_t>(pair));
  const int64_t dst = __ldg(p.block_mapping + 2 * static_cast<int64_t>(pair) + 1);
  if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
    if (threadIdx.x == 0) raise_error(p.err, PA_DEVERR_BLOCK_ID);
    return;
  }
  if (src == dst) return;
  unsigned char* pool = static_cast<unsigned char*>(is_v ? p.v_caches[layer] : p.k_caches[layer]);
  const uint4* s = reinterpret_cast<const uint4*>(pool + src * p.block_bytes);
  uint4* d = reinterpret_cast<uint4*>(pool + dst * p.block_bytes);
  const int64_t n = p.block_bytes / 16;
  int64_t i = threadIdx.x;
  for (; i + 3 * kCopyThreads < n; i += 4 * kCopyThreads) {
    const uint4 a = __ldg(s + i), b = __ldg(s + i + kCopyThreads);
    const uint4 c = __ldg(s + i + 2 * kCopyThreads), e = __ldg(s + i + 3 * kCopyThreads);
    d[i] = a;
    d[i + kCopyThreads] = b;
    d[i + 2 * kCopyThreads] = c;
    d[i + 3 * kCopyThreads] = e;
  }
  for (; i < n; i += kCopyThreads) d[i] = __ldg(s + i);
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyBlocksParams& p, int num_pairs, int num_layers,
                               cudaStream_t stream) {
  if (num_pairs == 0 || num_layers == 0) return cudaSuccess;
  return launch_pdl(copy_blocks_kernel, dim3(num_pairs, num_layers, 2), dim3(kCopyThreads), 0,
                    stream, p);
}

}  // namespace pa
