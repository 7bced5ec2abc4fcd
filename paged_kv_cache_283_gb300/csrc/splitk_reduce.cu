// Split-K merge (pa_splitk_reduce): combines the per-partition statistics
// written by the partition pass by the log-sum-exp identity,
//   M = max_p m_p,  w_p = l_p exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p,
// and rounds the result to bf16.  Reads B * Hq * P * (D + 2) * 4 bytes.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "device.cuh"
#include "internal.h"

namespace pa {

namespace {

// Log-sum-exp merge of split-K partitions: one CTA of D threads per
// (sequence, query head); thread d owns output dim d.  Partition weights
// are recomputed by every thread from (m, l), which are warp-uniform loads.
// The first kSpecParts partitions' (m, l, o) are read before the context
// length is known (those workspace rows always exist), so a short sequence
// costs one memory round trip instead of three.
constexpr int kSpecParts = 4;

template <int D>
__global__ void __launch_bounds__(D) splitk_reduce_kernel(const ReduceParams p) {
  griddep_wait();  // the partition pass is complete
  griddep_launch_dependents();
  const int hq = blockIdx.x;
  const int b = blockIdx.y;
  const int d = threadIdx.x;
  const size_t row0 = (static_cast<size_t>(b) * p.num_q_heads + hq) * p.max_partitions;
  const float* m = p.ws_m + row0;
  const float* l = p.ws_l + row0;
  const float* o = p.ws_o + row0 * D + d;
  float ms[kSpecParts], ls[kSpecParts], os[kSpecParts];
#pragma unroll
  for (int i = 0; i < kSpecParts; ++i) {
    if (i < p.max_partitions) {
      ms[i] = __ldg(m + i);
      ls[i] = __ldg(l + i);
      os[i] = __ldg(o + static_cast<size_t>(i) * D);
    }
  }
  int ctx = __ldg(p.context_lens + b);
  const int64_t cap = static_cast<int64_t>(p.max_partitions) * p.partition_size;
  if (ctx < 0 || ctx > cap) {
    if (d == 0 && hq == 0) raise_error(p.err, PA_DEVERR_CONTEXT_LEN);
    ctx = ctx < 0 ? 0 : static_cast<int>(cap);
  }
  const int np = (ctx + p.partition_size - 1) / p.partition_size;
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kSpecParts; ++i)
    if (i < np) M = fmaxf(M, ms[i]);
  for (int i = kSpecParts; i < np; ++i) M = fmaxf(M, m[i]);
  float acc = 0.f, Ls = 0.f;
#pragma unroll
  for (int i = 0; i < kSpecParts; ++i) {
    if (i < np) {
      const float w = ls[i] * expf(ms[i] - M);
      Ls += w;
      acc += w * os[i];
    }
  }
  int i = kSpecParts;
  for (; i + 4 <= np; i += 4) {
    const float w0 = l[i] * expf(m[i] - M), w1 = l[i + 1] * expf(m[i + 1] - M);
    const float w2 = l[i + 2] * expf(m[i + 2] - M), w3 = l[i + 3] * expf(m[i + 3] - M);
    const float o0 = o[static_cast<size_t>(i) * D], o1 = o[static_cast<size_t>(i + 1) * D];
    const float o2 = o[static_cast<size_t>(i + 2) * D], o3 = o[static_cast<size_t>(i + 3) * D];
    Ls += (w0 + w1) + (w2 + w3);
    acc += (w0 * o0 + w1 * o1) + (w2 * o2 + w3 * o3);
  }
  for (; i < np; ++i) {
    const float w = l[i] * expf(m[i] - M);
    Ls += w;
    acc += w * o[static_cast<size_t>(i) * D];
  }
  const float r = np > 0 ? acc / Ls : 0.f;
  p.out[(static_cast<size_t>(b) * p.num_q_heads + hq) * D + d] = __float2bfloat16_rn(r);
}

}  // namespace

cudaError_t launch_splitk_reduce(const ReduceParams& p, int head_dim, cudaStream_t stream) {
  const dim3 grid(p.num_q_heads, p.num_seqs);
  if (head_dim == 128) return launch_pdl(splitk_reduce_kernel<128>, grid, dim3(128), 0, stream, p);
  if (head_dim == 64) return launch_pdl(splitk_reduce_kernel<64>, grid, dim3(64), 0, stream, p);
  return cudaErrorInvalidValue;
}

}  // namespace pa
