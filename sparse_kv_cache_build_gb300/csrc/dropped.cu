// Dropped attention mass probe (diagnostic; not part of a decode step).
//
//   delta[b][h] = sum over valid tokens of unselected pages of exp(x_t - M)
//                 / sum over all valid tokens of exp(x_t - M),   x_t = sm_scale * q.k_t
//
// Sources: "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference",
// abstract (delta, the attention mass of the discarded entries); "EntmaxKV: Support-Aware
// Decoding for Entmax Attention", abstract (the sparse output error is governed by delta).
//
// Pass 1: one CTA per (page range s, KV head g, sequence b). The selected list of the
// group is turned into a bitmap over the CTA's page range in shared memory; each warp walks
// its pages token by token (one coalesced row read per token, a butterfly sum per query
// head) and keeps a running (max, total mass, dropped mass) per head in base 2. The warps
// are merged and the CTA writes one triple per head. Pass 2 merges the triples of the
// ranges. The probe reads every key once; it favours plainness over speed.
#include <math.h>

#include "kv_internal.cuh"

namespace skv {
namespace {

constexpr int kDmWarps = 8;
constexpr int kDmMaxRange = 1 << 16;      // pages of one range (bitmap of 8 KB)

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDmWarps * 32)
dropped_partial_kernel(kv_cache_desc d, const T* __restrict__ q, float qk_scale_log2,
                       const int32_t* __restrict__ sel_idx, const int32_t* __restrict__ sel_cnt,
                       int sel_stride, int S, float* __restrict__ partials, DevCtx ctx) {
  constexpr int EPV = D / 32;
  __shared__ uint32_t bitmap[kDmMaxRange / 32];
  __shared__ float wst[kDmWarps][G][3];

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, PS = d.page_size;
  const int len = checked_len(ctx, d, b);
  const int n = ceil_div(len, PS);
  const int c = n > 0 ? ceil_div(n, S) : 0;
  const int pa = min(n, s * c);
  const int pb = min(n, pa + min(c, kDmMaxRange));
  const long grp = (long)b * Hkv + g;

  for (int i = tid; i < kDmMaxRange / 32; i += kDmWarps * 32) bitmap[i] = 0u;
  __syncthreads();
  int cnt = sel_cnt[grp];
  if (cnt < 0 || cnt > sel_stride) {
    if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
    cnt = cnt < 0 ? 0 : sel_stride;
  }
  for (int i = tid; i < cnt; i += kDmWarps * 32) {
    const int p = sel_idx[grp * sel_stride + i];
    if (p < 0 || p >= n) {
      flag(ctx, KV_DEVERR_BAD_SEL);
    } else if (p >= pa && p < pb) {
      atomicOr(&bitmap[(p - pa) >> 5], 1u << ((p - pa) & 31));
    }
  }
  __syncthreads();

  float qv[G][EPV];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < EPV; ++e)
      qv[h][e] = load_elem<T>(q, ((long)b * Hq + g * G + h) * D + lane * EPV + e);

  float m[G], la[G], ld[G];
#pragma unroll
  for (int h = 0; h < G; ++h) { m[h] = -INFINITY; la[h] = 0.f; ld[h] = 0.f; }

  const T* kp = static_cast<const T*>(d.k_pool);
  const int32_t* table = d.page_table + (long)b * d.page_table_stride;
  for (int p = pa + warp; p < pb; p += kDmWarps) {
    const int P = table[p];
    if (P < 0 || P >= d.num_phys_pages) {
      if (lane == 0) flag(ctx, KV_DEVERR_BAD_PAGE);
      continue;
    }
    const bool kept = (bitmap[(p - pa) >> 5] >> ((p - pa) & 31)) & 1u;
    const int valid = min(PS, len - p * PS);
    const T* page = kp + (((long)P * Hkv + g) * PS) * D + lane * EPV;
    for (int t = 0; t < valid; ++t) {
      float kf[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) kf[e] = load_elem<T>(page, (long)t * D + e);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) dot = fmaf(qv[h][e], kf[e], dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const float x = dot * qk_scale_log2;
        if (x > m[h]) {
          const float sc = m[h] == -INFINITY ? 0.f : exp2f(m[h] - x);
          la[h] *= sc;
          ld[h] *= sc;
          m[h] = x;
        }
        const float w = exp2f(x - m[h]);
        la[h] += w;
        if (!kept) ld[h] += w;
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      wst[warp][h][0] = m[h];
      wst[warp][h][1] = la[h];
      wst[warp][h][2] = ld[h];
    }
  }
  __syncthreads();
  if (tid < G) {
    const int h = tid;
    float M = -INFINITY;
    for (int w = 0; w < kDmWarps; ++w) M = fmaxf(M, wst[w][h][0]);
    float LA = 0.f, LD = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kDmWarps; ++w) {
        const float mw = wst[w][h][0];
        if (mw == -INFINITY) continue;
        const float sc = exp2f(mw - M);
        LA = fmaf(wst[w][h][1], sc, LA);
        LD = fmaf(wst[w][h][2], sc, LD);
      }
    }
    float* dst = partials + (((long)b * Hq + g * G + h) * S + s) * 3;
    dst[0] = M;
    dst[1] = LA;
    dst[2] = LD;
  }
}

__global__ void dropped_merge_kernel(const float* __restrict__ partials, int BH, int S,
                                     float* __restrict__ delta) {
  const int bh = blockIdx.x * blockDim.x + threadIdx.x;
  if (bh >= BH) return;
  const float* pr = partials + (long)bh * S * 3;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, pr[3 * s]);
  float LA = 0.f, LD = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      if (pr[3 * s] == -INFINITY) continue;
      const float sc = exp2f(pr[3 * s] - M);
      LA = fmaf(pr[3 * s + 1], sc, LA);
      LD = fmaf(pr[3 * s + 2], sc, LD);
    }
  }
  delta[bh] = LA > 0.f ? LD / LA : 0.f;
}

template <typename T, int D>
cudaError_t launch_partial_d(const kv_cache_desc& d, const void* q, int G, float scale_log2,
                             const int32_t* sel_idx, const int32_t* sel_cnt, int sel_stride,
                             int S, float* partials, DevCtx ctx, cudaStream_t st) {
  dim3 grid(S, d.num_kv_heads, d.batch);
  const T* qt = static_cast<const T*>(q);
  switch (G) {
    case 1: dropped_partial_kernel<T, D, 1><<<grid, kDmWarps * 32, 0, st>>>(d, qt, scale_log2, sel_idx, sel_cnt, sel_stride, S, partials, ctx); break;
    case 2: dropped_partial_kernel<T, D, 2><<<grid, kDmWarps * 32, 0, st>>>(d, qt, scale_log2, sel_idx, sel_cnt, sel_stride, S, partials, ctx); break;
    case 4: dropped_partial_kernel<T, D, 4><<<grid, kDmWarps * 32, 0, st>>>(d, qt, scale_log2, sel_idx, sel_cnt, sel_stride, S, partials, ctx); break;
    case 8: dropped_partial_kernel<T, D, 8><<<grid, kDmWarps * 32, 0, st>>>(d, qt, scale_log2, sel_idx, sel_cnt, sel_stride, S, partials, ctx); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dropped_mass(const kv_cache_desc& d, const void* q, int Hq,
                                float sm_scale, const int32_t* sel_idx,
                                const int32_t* sel_cnt, int sel_stride, int num_splits,
                                float* partials, float* delta, DevCtx ctx, cudaStream_t st) {
  const int G = Hq / d.num_kv_heads;
  const float sl2 = sm_scale * kLog2e;
  cudaError_t e;
  const bool bf = d.dtype == KV_BF16;
  if (d.head_dim == 128)
    e = bf ? launch_partial_d<bf16_t, 128>(d, q, G, sl2, sel_idx, sel_cnt, sel_stride, num_splits, partials, ctx, st)
           : launch_partial_d<float, 128>(d, q, G, sl2, sel_idx, sel_cnt, sel_stride, num_splits, partials, ctx, st);
  else
    e = bf ? launch_partial_d<bf16_t, 64>(d, q, G, sl2, sel_idx, sel_cnt, sel_stride, num_splits, partials, ctx, st)
           : launch_partial_d<float, 64>(d, q, G, sl2, sel_idx, sel_cnt, sel_stride, num_splits, partials, ctx, st);
  if (e != cudaSuccess) return e;
  const int BH = d.batch * Hq;
  dropped_merge_kernel<<<(BH + 127) / 128, 128, 0, st>>>(partials, BH, num_splits, delta);
  return cudaGetLastError();
}

}  // namespace skv
