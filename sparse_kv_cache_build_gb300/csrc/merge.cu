// Log-sum-exp merge of split-K partials into the attention output.
//
// Source: "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding",
// abstract (split-K decode attention). Each split s holds (m_s, l_s, acc_s) with
// l_s = sum exp(x - m_s) and acc_s = sum exp(x - m_s) v over its tokens; then
//   M = max_s m_s,  L = sum_s l_s exp(m_s - M),  out = sum_s acc_s exp(m_s - M) / L,
//   lse = M + log L.
// Splits with m_s = -inf hold no tokens and carry no weight. One block per (b, h), one
// thread per output column; the S partial rows of a head are contiguous, so every read is
// coalesced.
#include <math.h>

#include "kv_internal.cuh"

namespace skv {
namespace {

__global__ void merge_kernel(const float* __restrict__ part_acc,
                             const float* __restrict__ part_ml, int S, int D,
                             float* __restrict__ out, float* __restrict__ lse) {
  const long bh = blockIdx.x;
  const int dd = threadIdx.x;
  const float* ml = part_ml + bh * S * 2;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, ml[2 * s]);
  if (M == -INFINITY) {
    out[bh * D + dd] = 0.f;
    if (dd == 0 && lse != nullptr) lse[bh] = -INFINITY;
    return;
  }
  float L = 0.f, A = 0.f;
  for (int s = 0; s < S; ++s) {
    const float m = ml[2 * s];
    if (m == -INFINITY) continue;
    const float w = expf(m - M);
    L = fmaf(ml[2 * s + 1], w, L);
    A = fmaf(part_acc[(bh * S + s) * D + dd], w, A);
  }
  out[bh * D + dd] = A / L;
  if (dd == 0 && lse != nullptr) lse[bh] = M + logf(L);
}

}  // namespace

cudaError_t launch_merge(const float* part_acc, const float* part_ml, int batch, int Hq,
                         int num_splits, int D, float* out, float* lse, cudaStream_t s) {
  merge_kernel<<<(unsigned)(batch * Hq), D, 0, s>>>(part_acc, part_ml, num_splits, D, out, lse);
  return cudaGetLastError();
}

}  // namespace skv
