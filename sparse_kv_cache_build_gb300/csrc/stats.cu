// Per-page key statistics: element-wise min and max of the keys of each mapped page, per
// KV head, over the page's valid tokens.
//
// Source: "EntmaxKV: Support-Aware Decoding for Entmax Attention", abstract -- pages are
// scored against the query from cheap per-page statistics before the page itself is read.
// The statistic kept here is the coordinate-wise [min, max] box of the page's keys, which
// makes the page score an exact upper bound of q.k (see score.cu).
//
// Subset builds: given a strictly ascending list of physical pages, only mapped pages whose
// physical index is in the list are (re)built (a binary search per page; the rest of the
// table costs one int32 read per page). Block (0, 0) checks that the list is ascending and
// inside the pool, and flags it otherwise.
//
// Layout: one warp per (physical page, KV head) chunk. The chunk is PS rows of D
// contiguous elements; lane l owns D/32 consecutive columns, so every row read by the warp
// is one coalesced 128- or 256-byte access. Values are compared as floats and written back
// bit for bit in the storage dtype (min and max of exact values are exact), or, in the FP8
// form (fp8_stats.cuh), as E4M3 bytes rounded outward under the row's power-of-two exponent
// (the warp finds the row's largest magnitude with one reduction).
#include "fp8_stats.cuh"
#include "kv_internal.cuh"

namespace skv {
namespace {

constexpr int kStatsWarps = 8;
constexpr int kStatsPagesPerBlock = 8;

template <typename T, int EPL>
__device__ __forceinline__ void load_row(const T* p, float* f) {
  if constexpr (sizeof(T) == 2) {
    if constexpr (EPL == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
      f[0] = bf16_lo(v); f[1] = bf16_hi(v);
    }
  } else {
    if constexpr (EPL == 4) {
      const float4 v = *reinterpret_cast<const float4*>(p);
      f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(p);
      f[0] = v.x; f[1] = v.y;
    }
  }
}

template <typename T, int EPL>
__device__ __forceinline__ void store_row(T* p, const float* f) {
  if constexpr (sizeof(T) == 2) {
    // the floats hold bf16 values exactly: their upper halves are the bf16 bits
    uint32_t w[EPL / 2];
#pragma unroll
    for (int i = 0; i < EPL / 2; ++i)
      w[i] = (__float_as_uint(f[2 * i]) >> 16) | (__float_as_uint(f[2 * i + 1]) & 0xffff0000u);
    if constexpr (EPL == 4) *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
    else *reinterpret_cast<uint32_t*>(p) = w[0];
  } else {
    if constexpr (EPL == 4) *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    else *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
  }
}

// Whether P is one of list[0, n) (strictly ascending): lower bound by bisection. Every lane of
// a warp reads the same entries (broadcast loads).
__device__ __forceinline__ bool in_sorted(const int32_t* __restrict__ list, int n, int P) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(list + mid) < P) lo = mid + 1;
    else hi = mid;
  }
  return lo < n && __ldg(list + lo) == P;
}

template <typename T, int D, bool F8>
__global__ void __launch_bounds__(kStatsWarps * 32)
page_stats_kernel(kv_cache_desc d, T* __restrict__ stats, uint8_t* __restrict__ codes,
                  int8_t* __restrict__ exps, const int32_t* __restrict__ subset, int n_subset,
                  DevCtx ctx) {
  constexpr int EPL = D / 32;
  const int b = blockIdx.y;
  if (subset != nullptr && blockIdx.x == 0 && b == 0) {
    for (int i = threadIdx.x; i < n_subset; i += blockDim.x) {
      const int P = __ldg(subset + i);
      if (P < 0 || P >= d.num_phys_pages || (i + 1 < n_subset && __ldg(subset + i + 1) <= P))
        flag(ctx, KV_DEVERR_BAD_PAGE);
    }
  }
  const int len = checked_len(ctx, d, b);
  const int PS = d.page_size, Hkv = d.num_kv_heads;
  const int n_pages = ceil_div(len, PS);
  const int p0 = blockIdx.x * kStatsPagesPerBlock;
  if (p0 >= n_pages) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = kStatsPagesPerBlock * Hkv;
  const T* __restrict__ kp = static_cast<const T*>(d.k_pool);

  for (int it = warp; it < items; it += kStatsWarps) {
    const int p = p0 + it / Hkv;
    const int g = it % Hkv;
    if (p >= n_pages) break;
    const int P = d.page_table[(long)b * d.page_table_stride + p];
    if (P < 0 || P >= d.num_phys_pages) {
      if (lane == 0) flag(ctx, KV_DEVERR_BAD_PAGE);
      continue;
    }
    if (subset != nullptr && !in_sorted(subset, n_subset, P)) continue;
    const int valid = min(PS, len - p * PS);
    const T* src = kp + (((long)P * Hkv + g) * PS) * D + lane * EPL;
    float mn[EPL], mx[EPL], v[EPL];
    load_row<T, EPL>(src, mn);
#pragma unroll
    for (int e = 0; e < EPL; ++e) mx[e] = mn[e];
    for (int t = 1; t < valid; ++t) {
      load_row<T, EPL>(src + (long)t * D, v);
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        mn[e] = v[e] < mn[e] ? v[e] : mn[e];
        mx[e] = v[e] > mx[e] ? v[e] : mx[e];
      }
    }
    if constexpr (F8) {
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) m = fmaxf(m, fmaxf(fabsf(mn[e]), fabsf(mx[e])));
      const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
      const int ex = fp8::row_exponent(__uint_as_float(mb));
      const float inv = fp8::pow2(-ex);
      uint32_t lo = 0u, hi = 0u;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        lo |= fp8::quantize_down(mn[e], inv) << (8 * e);
        hi |= fp8::quantize_up(mx[e], inv) << (8 * e);
      }
      uint8_t* dst = codes + (((long)P * Hkv + g) * 2) * D + lane * EPL;
      if constexpr (EPL == 4) {
        *reinterpret_cast<uint32_t*>(dst) = lo;
        *reinterpret_cast<uint32_t*>(dst + D) = hi;
      } else {
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)lo;
        *reinterpret_cast<uint16_t*>(dst + D) = (uint16_t)hi;
      }
      if (lane == 0) exps[(long)P * Hkv + g] = (int8_t)ex;
    } else {
      T* dst = stats + (((long)P * Hkv + g) * 2) * D + lane * EPL;
      store_row<T, EPL>(dst, mn);
      store_row<T, EPL>(dst + D, mx);
    }
  }
}

template <typename T, int D>
cudaError_t launch_t(const kv_cache_desc& d, void* stats, int8_t* exps, const int32_t* subset,
                     int n_subset, DevCtx ctx, cudaStream_t s) {
  dim3 grid(ceil_div(d.page_table_stride, kStatsPagesPerBlock), d.batch);
  if (exps != nullptr)
    page_stats_kernel<T, D, true><<<grid, kStatsWarps * 32, 0, s>>>(
        d, nullptr, static_cast<uint8_t*>(stats), exps, subset, n_subset, ctx);
  else
    page_stats_kernel<T, D, false><<<grid, kStatsWarps * 32, 0, s>>>(
        d, static_cast<T*>(stats), nullptr, nullptr, subset, n_subset, ctx);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_page_stats(const kv_cache_desc& d, void* stats, int8_t* stats_exp,
                              const int32_t* subset, int n_subset, DevCtx ctx,
                              cudaStream_t s) {
  const bool bf = d.dtype == KV_BF16;
  if (d.head_dim == 128)
    return bf ? launch_t<bf16_t, 128>(d, stats, stats_exp, subset, n_subset, ctx, s)
              : launch_t<float, 128>(d, stats, stats_exp, subset, n_subset, ctx, s);
  return bf ? launch_t<bf16_t, 64>(d, stats, stats_exp, subset, n_subset, ctx, s)
            : launch_t<float, 64>(d, stats, stats_exp, subset, n_subset, ctx, s);
}

}  // namespace skv
