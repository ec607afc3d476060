// Query-aware page score: for each (sequence b, KV head g, logical page p)
//
//   s[b][g][p] = sum over query heads h of group g, over d, of
//                max(q[h][d] * mn[P][g][d], q[h][d] * mx[P][g][d]),   P = page_table[b][p]
//
// Sources: "EntmaxKV: Support-Aware Decoding for Entmax Attention", abstract (pages scored
// against the query from per-page statistics); "SparDA: Sparse Decoupled Attention for
// Efficient Long-Context LLM Inference", section 3.1 (per-head relevance summed inside a
// GQA group into one shared score).
//
// Because mn <= mx, max(q*mn, q*mx) = max(q, 0) * mx + min(q, 0) * mn exactly. Summed over
// the group's heads this is  sum_d  Pos[d] * mx[d] + Neg[d] * mn[d]  with
// Pos[d] = sum_h max(q[h][d], 0) and Neg[d] = sum_h min(q[h][d], 0): one dot product of
// length 2D per page whatever the group size. Pos/Neg are built once per block in shared
// memory in the [mn | mx] order of a stats row, so a page's score is the dot product of
// its contiguous stats row with that vector.
//
// The pass streams the stats array (2*D elements per page and KV head) once: it is
// HBM-bound, and short, so it is built to put every load in flight in one wave. Eight lanes
// own one page (16-byte chunks j, j+8, ... of the row), a 128-thread block covers 16 pages,
// and the grid covers every page of every group. Each block issues its page-table and
// statistics loads first and only then builds Pos/Neg from q, so the two latency chains
// overlap.
#include "kv_internal.cuh"

namespace skv {
namespace {

constexpr int kScoreWarps = 4;
constexpr int kScorePagesPerBlock = kScoreWarps * 4;   // 16

template <typename T, int D>
__global__ void __launch_bounds__(kScoreWarps * 32)
score_kernel(kv_cache_desc d, const T* __restrict__ q, int G, const T* __restrict__ stats,
             float* __restrict__ scores, int scores_stride, DevCtx ctx) {
  constexpr int EB = ElemTraits<T>::bytes;
  constexpr int EPC = 16 / EB;                // elements per 16-byte chunk
  constexpr int CPL = (2 * D * EB / 16) / 8;  // chunks per lane per stats row
  __shared__ __align__(16) float w[2 * D];    // [Neg | Pos], matching a row's [mn | mx]
  pdl_trigger();
  pdl_wait();

  const int b = blockIdx.z, g = blockIdx.y;
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, d.page_size);
  const int p_block = blockIdx.x * kScorePagesPerBlock;
  if (p_block >= n_pages) return;

  const int Hkv = d.num_kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 3, j = lane & 7;
  const int p = p_block + warp * 4 + grp;
  uint4 raw[CPL];
  bool ok = false;
  if (p < n_pages) {
    const int P = d.page_table[(long)b * d.page_table_stride + p];
    if (P >= 0 && P < d.num_phys_pages) {
      ok = true;
      const uint4* row = reinterpret_cast<const uint4*>(
          reinterpret_cast<const char*>(stats) + (((long)P * Hkv + g) * 2 * D) * EB);
#pragma unroll
      for (int u = 0; u < CPL; ++u) raw[u] = __ldg(row + j + 8 * u);
    } else if (j == 0) {
      flag(ctx, KV_DEVERR_BAD_PAGE);
    }
  }

  const int Hq = Hkv * G;
  for (int t = threadIdx.x; t < D; t += kScoreWarps * 32) {
    float pos = 0.f, neg = 0.f;
    for (int h = g * G; h < (g + 1) * G; ++h) {
      const float x = load_elem<T>(q, ((long)b * Hq + h) * D + t);
      pos += fmaxf(x, 0.f);
      neg += fminf(x, 0.f);
    }
    w[t] = neg;
    w[D + t] = pos;
  }
  __syncthreads();

  float acc = 0.f;
  if (ok) {
#pragma unroll
    for (int u = 0; u < CPL; ++u) {
      float f[EPC];
      chunk_to_f32<T>(raw[u], f);
      const float* wc = w + (j + 8 * u) * EPC;
#pragma unroll
      for (int e = 0; e < EPC; ++e) acc = fmaf(wc[e], f[e], acc);
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (j == 0 && ok) scores[((long)b * Hkv + g) * scores_stride + p] = acc;
}

template <typename T, int D>
cudaError_t launch_t(const kv_cache_desc& d, const void* q, int Hq, const void* stats,
                     float* scores, int scores_stride, DevCtx ctx, cudaStream_t s) {
  dim3 grid(ceil_div(d.page_table_stride, kScorePagesPerBlock), d.num_kv_heads, d.batch);
  return launch_pdl(score_kernel<T, D>, grid, dim3(kScoreWarps * 32), 0, s, d,
                    static_cast<const T*>(q), Hq / d.num_kv_heads,
                    static_cast<const T*>(stats), scores, scores_stride, ctx);
}

}  // namespace

cudaError_t launch_score_pages(const kv_cache_desc& d, const void* q, int Hq,
                               const void* stats, float* scores, int scores_stride,
                               DevCtx ctx, cudaStream_t s) {
  const bool bf = d.dtype == KV_BF16;
  if (d.head_dim == 128)
    return bf ? launch_t<bf16_t, 128>(d, q, Hq, stats, scores, scores_stride, ctx, s)
              : launch_t<float, 128>(d, q, Hq, stats, scores, scores_stride, ctx, s);
  return bf ? launch_t<bf16_t, 64>(d, q, Hq, stats, scores, scores_stride, ctx, s)
            : launch_t<float, 64>(d, q, Hq, stats, scores, scores_stride, ctx, s);
}

}  // namespace skv
