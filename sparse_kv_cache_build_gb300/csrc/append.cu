// Token append with incremental page statistics.
//
// Source: "EntmaxKV: Support-Aware Decoding for Entmax Attention", abstract -- the cache
// grows by one token per decode step and pages are scored from per-page statistics; keeping
// those statistics current must not cost a re-read of the cache. Appending token t of
// sequence b writes its key and value at slot t % PS of logical page t / PS and folds the key
// into that page's element-wise [min, max] (a page's first token resets them). Min and max
// are exact, so the result equals kv_build_page_stats of the grown cache bit for bit: a key
// replaces the running min (max) only when strictly smaller (larger), the same rule, in the
// same token order, as the full build.
//
// One block per (KV head, sequence), one thread per column: the new token's 2*D elements
// and the page's 2*D statistics are the only bytes touched.
#include "kv_internal.cuh"

namespace skv {
namespace {

template <typename T>
__device__ __forceinline__ void store_elem(void* base, long i, float v);
template <>
__device__ __forceinline__ void store_elem<bf16_t>(void* base, long i, float v) {
  reinterpret_cast<uint16_t*>(base)[i] = static_cast<uint16_t>(__float_as_uint(v) >> 16);
}
template <>
__device__ __forceinline__ void store_elem<float>(void* base, long i, float v) {
  reinterpret_cast<float*>(base)[i] = v;
}

template <typename T>
__global__ void append_kernel(kv_cache_desc d, const T* __restrict__ k_new,
                              const T* __restrict__ v_new, T* __restrict__ stats, DevCtx ctx) {
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.x, b = blockIdx.y;
  const int D = d.head_dim, Hkv = d.num_kv_heads, PS = d.page_size;
  int len = d.seq_lens[b];
  if (len <= 0) return;                                   // nothing to append
  if (len > d.page_table_stride * PS) {
    if (threadIdx.x == 0) flag(ctx, KV_DEVERR_BAD_LEN);
    return;
  }
  const int t = len - 1, p = t / PS, slot = t % PS;
  const int P = d.page_table[(long)b * d.page_table_stride + p];
  if (P < 0 || P >= d.num_phys_pages) {
    if (threadIdx.x == 0) flag(ctx, KV_DEVERR_BAD_PAGE);
    return;
  }
  void* kp = const_cast<void*>(d.k_pool);
  void* vp = const_cast<void*>(d.v_pool);
  const long src = ((long)b * Hkv + g) * D;
  const long row = (((long)P * Hkv + g) * PS + slot) * D;
  const long srow = ((long)P * Hkv + g) * 2 * D;
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    const float k = load_elem<T>(k_new, src + i);
    const float v = load_elem<T>(v_new, src + i);
    store_elem<T>(kp, row + i, k);
    store_elem<T>(vp, row + i, v);
    float mn = k, mx = k;
    if (slot > 0) {
      const float omn = load_elem<T>(stats, srow + i);
      const float omx = load_elem<T>(stats, srow + D + i);
      mn = k < omn ? k : omn;
      mx = k > omx ? k : omx;
    }
    store_elem<T>(stats, srow + i, mn);
    store_elem<T>(stats, srow + D + i, mx);
  }
}

}  // namespace

cudaError_t launch_append(const kv_cache_desc& d, const void* k_new, const void* v_new,
                          void* stats, DevCtx ctx, cudaStream_t s) {
  dim3 grid(d.num_kv_heads, d.batch);
  if (d.dtype == KV_BF16)
    return launch_pdl(append_kernel<bf16_t>, grid, dim3(d.head_dim), 0, s, d,
                      static_cast<const bf16_t*>(k_new), static_cast<const bf16_t*>(v_new),
                      static_cast<bf16_t*>(stats), ctx);
  return launch_pdl(append_kernel<float>, grid, dim3(d.head_dim), 0, s, d,
                    static_cast<const float*>(k_new), static_cast<const float*>(v_new),
                    static_cast<float*>(stats), ctx);
}

}  // namespace skv
