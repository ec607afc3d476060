// Log-sum-exp merge of split-K partials into the attention output.
//
// Source: "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding",
// abstract (split-K decode attention). Each split s holds (m_s, l_s, acc_s) with
// l_s = sum exp(x - m_s) and acc_s = sum exp(x - m_s) v over its tokens; then
//   M = max_s m_s,  L = sum_s l_s exp(m_s - M),  out = sum_s acc_s exp(m_s - M) / L,
//   lse = M + log L.
// Splits with m_s = -inf hold no tokens and carry no weight.
//
// The work is tiny (S*(D+2) floats per head) so the kernel is built for latency: one
// block of 4*D threads per (b, h). The split weights are computed once, in parallel, into
// shared memory; then each of the four thread groups sums a quarter of the splits for its
// column with all loads independent, and the four partial sums meet in shared memory.
#include <math.h>

#include "kv_internal.cuh"

namespace skv {
namespace {

constexpr int kMergeParts = 4;
constexpr int kMergeMaxSplits = 4096;     // splits whose weights fit in shared memory

template <int D>
__global__ void __launch_bounds__(D * kMergeParts)
merge_kernel(const float* __restrict__ part_acc, const float* __restrict__ part_ml, int S,
             float* __restrict__ out, float* __restrict__ lse) {
  __shared__ float w[kMergeMaxSplits];
  __shared__ float red[D * kMergeParts / 32];
  __shared__ float partial[kMergeParts][D];
  __shared__ float sM, sL;
  pdl_trigger();
  pdl_wait();
  const long bh = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int T = D * kMergeParts;
  const float* ml = part_ml + bh * S * 2;

  float m = -INFINITY;
  for (int s = tid; s < S; s += T) m = fmaxf(m, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (tid == 0) {
    float M = -INFINITY;
    for (int i = 0; i < T / 32; ++i) M = fmaxf(M, red[i]);
    sM = M;
  }
  __syncthreads();
  const float M = sM;
  if (M == -INFINITY) {                       // every split empty
    if (tid < D) out[bh * D + tid] = 0.f;
    if (tid == 0 && lse != nullptr) lse[bh] = -INFINITY;
    return;
  }
  float l = 0.f;
  for (int s = tid; s < S; s += T) {
    const float ms = ml[2 * s];
    const float ws = ms == -INFINITY ? 0.f : expf(ms - M);
    w[s] = ws;
    l = fmaf(ml[2 * s + 1], ws, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  __syncthreads();                            // red[] reuse and w[] complete
  if (lane == 0) red[warp] = l;
  __syncthreads();
  if (tid == 0) {
    float L = 0.f;
    for (int i = 0; i < T / 32; ++i) L += red[i];
    sL = L;
  }
  const int d = tid % D, part = tid / D;
  const float* a = part_acc + bh * S * D + d;
  float acc = 0.f;
#pragma unroll 8
  for (int s = part; s < S; s += kMergeParts) acc = fmaf(a[(long)s * D], w[s], acc);
  partial[part][d] = acc;
  __syncthreads();
  if (part == 0) {
    float A = 0.f;
#pragma unroll
    for (int p = 0; p < kMergeParts; ++p) A += partial[p][d];
    out[bh * D + d] = A / sL;
    if (d == 0 && lse != nullptr) lse[bh] = M + logf(sL);
  }
}

// Up to 64 splits (the automatic split counts): every load is issued at once (each thread
// its column of a quarter of the splits, each warp every split's (m, l)), each warp finds M
// and L itself from its (m, l) with warp instructions, and one barrier joins the four
// partial sums: one dependent memory round trip and one barrier.
constexpr int kMergeShortSplits = 64;

template <int D>
__global__ void __launch_bounds__(D * kMergeParts)
merge_kernel_short(const float* __restrict__ part_acc, const float* __restrict__ part_ml,
                   int S, float* __restrict__ out, float* __restrict__ lse) {
  constexpr int PER = kMergeShortSplits / kMergeParts;   // splits per thread at most
  __shared__ float partial[kMergeParts][D];
  pdl_trigger();
  pdl_wait();
  const long bh = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int d = tid % D, part = tid / D;
  const float* ml = part_ml + bh * S * 2;
  const float* a = part_acc + bh * S * D + d;
  float av[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int sp = part + k * kMergeParts;
    av[k] = sp < S ? __ldcg(a + (long)sp * D) : 0.f;
  }
  const float m0 = lane < S ? __ldcg(ml + 2 * lane) : -INFINITY;
  const float m1 = lane + 32 < S ? __ldcg(ml + 2 * (lane + 32)) : -INFINITY;
  const float l0 = lane < S ? __ldcg(ml + 2 * lane + 1) : 0.f;
  const float l1 = lane + 32 < S ? __ldcg(ml + 2 * (lane + 32) + 1) : 0.f;
  float M = fmaxf(m0, m1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (M == -INFINITY) {                          // every split empty (block-uniform)
    if (part == 0) out[bh * D + d] = 0.f;
    if (tid == 0 && lse != nullptr) lse[bh] = -INFINITY;
    return;
  }
  const float w0 = m0 == -INFINITY ? 0.f : expf(m0 - M);
  const float w1 = m1 == -INFINITY ? 0.f : expf(m1 - M);
  float L = fmaf(l0, w0, l1 * w1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int sp = part + k * kMergeParts;                // block-uniform per k
    const float ws = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
    if (sp < S) acc = fmaf(av[k], ws, acc);
  }
  partial[part][d] = acc;
  __syncthreads();
  if (part == 0) {
    float A = 0.f;
#pragma unroll
    for (int p = 0; p < kMergeParts; ++p) A += partial[p][d];
    out[bh * D + d] = A / L;
    if (d == 0 && lse != nullptr) lse[bh] = M + logf(L);
  }
}

// Fallback for more splits than the shared weight table holds: one thread per column.
__global__ void merge_kernel_many(const float* __restrict__ part_acc,
                                  const float* __restrict__ part_ml, int S, int D,
                                  float* __restrict__ out, float* __restrict__ lse) {
  pdl_trigger();
  pdl_wait();
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
    const float ms = ml[2 * s];
    const float ws = ms == -INFINITY ? 0.f : expf(ms - M);
    L = fmaf(ml[2 * s + 1], ws, L);
    A = fmaf(part_acc[(bh * S + s) * D + dd], ws, A);
  }
  out[bh * D + dd] = A / L;
  if (dd == 0 && lse != nullptr) lse[bh] = M + logf(L);
}

}  // namespace

cudaError_t launch_merge(const float* part_acc, const float* part_ml, int batch, int Hq,
                         int num_splits, int D, float* out, float* lse, cudaStream_t s) {
  const unsigned blocks = (unsigned)(batch * Hq);
  if (num_splits > kMergeMaxSplits)
    return launch_pdl(merge_kernel_many, dim3(blocks), dim3(D), 0, s, part_acc, part_ml,
                      num_splits, D, out, lse);
  if (num_splits <= kMergeShortSplits) {
    if (D == 128)
      return launch_pdl(merge_kernel_short<128>, dim3(blocks), dim3(128 * kMergeParts), 0, s,
                        part_acc, part_ml, num_splits, out, lse);
    return launch_pdl(merge_kernel_short<64>, dim3(blocks), dim3(64 * kMergeParts), 0, s,
                      part_acc, part_ml, num_splits, out, lse);
  }
  if (D == 128)
    return launch_pdl(merge_kernel<128>, dim3(blocks), dim3(128 * kMergeParts), 0, s,
                      part_acc, part_ml, num_splits, out, lse);
  return launch_pdl(merge_kernel<64>, dim3(blocks), dim3(64 * kMergeParts), 0, s, part_acc,
                    part_ml, num_splits, out, lse);
}

}  // namespace skv
