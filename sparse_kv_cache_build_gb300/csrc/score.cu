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
// HBM-bound, and short, so it is built to put every load in flight in about one wave. Eight
// lanes own one page (16-byte chunks j, j+8, ... of the row), a 128-thread block covers runs
// of 16 pages (one run, or as many as keep the grid to about 8 blocks per SM, the next run's
// loads in flight while a run is summed), and the grid covers every page of every group.
// Each block issues its first page-table load before the sequence length, then its
// statistics loads, and only then builds Pos/Neg from q, so the latency chains overlap.
//
// score_select_kernel is the same pass followed by the group's top-k (the rule of
// select.cu): 512-thread blocks of 64 pages each; the block of a group that finishes last
// (a per-group arrival counter, returned to zero) reads the group's scores back from L2
// and runs the block-wide selection of cta_topk.cuh, so the selection costs no launch of
// its own and runs once per group.
//
// FP8 statistics (fp8_stats.cuh): a row is 2*D E4M3 bytes plus the row's exponent e. Four
// lanes own a row (each keeps the same 64 bytes in flight as a lane of a bf16 row, so a warp
// covers twice the rows), the bytes convert exactly to half precision two at a time and then
// to float, and the row's dot product is scaled by 2^e once at the end (a power-of-two
// scaling commutes with the fp32 rounding of the sum, so this equals summing the decoded
// values times 2^e).
#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>

#include "cta_topk.cuh"
#include "fp8_stats.cuh"
#include "kv_internal.cuh"

namespace skv {
namespace {

constexpr int kScoreWarps = 4;
constexpr int kScoreMaxRuns = 8;              // 16-page runs per score block at most
// rows (pages) per warp: eight lanes per row, four for FP8 rows
template <bool F8>
constexpr int rows_per_warp() { return F8 ? 8 : 4; }

// The 16 values of a 16-byte chunk of E4M3 bytes, in byte order (exact).
__device__ __forceinline__ void fp8_chunk_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)((w[i] >> (16 * j)) & 0xffffu), __NV_E4M3);
      const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&h));
      f[4 * i + 2 * j] = x.x;
      f[4 * i + 2 * j + 1] = x.y;
    }
  }
}
constexpr int kSelWarps = 16;                          // score + select blocks: 512 threads
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kSelCandWords = 4096;                    // gathered keys of the threshold bin

// This lane's first page of block `chunk` (a block takes `rounds` runs of WARPS * RPW pages;
// the page lies in the table's row whatever the length).
template <int WARPS, bool F8>
__device__ __forceinline__ int score_page(int chunk, int rounds) {
  constexpr int RPW = rows_per_warp<F8>();
  return chunk * WARPS * RPW * rounds + (threadIdx.x >> 5) * RPW + (threadIdx.x & 31) / (32 / RPW);
}

// The page-table entry of this lane's first page, loaded before the sequence length is known
// (the entry lies in the table's row whatever the length; it is used only below the length),
// so the two loads are in flight together.
template <int WARPS, bool F8>
__device__ __forceinline__ int score_table_entry(const kv_cache_desc& d, int b, int chunk,
                                                 int rounds) {
  const int p = score_page<WARPS, F8>(chunk, rounds);
  return p < d.page_table_stride ? __ldg(d.page_table + (long)b * d.page_table_stride + p) : -1;
}

// Scores of this block's pages for group (b, g) into scores: `rounds` runs of WARPS * RPW
// pages, the next run's loads in flight while a run is summed. Returns false (block-uniform)
// if the block has no page of the sequence. P_lane: this lane's first page-table entry
// (score_table_entry). F8: stats are E4M3 bytes with one exponent per row in stats_exp;
// otherwise stats are of the query's type T.
template <typename T, int D, int WARPS, bool F8>
__device__ __forceinline__ bool score_block(const kv_cache_desc& d, const T* __restrict__ q,
                                            int G, const void* __restrict__ stats,
                                            const int8_t* __restrict__ stats_exp, float* w,
                                            float* __restrict__ scores, int scores_stride,
                                            int b, int g, int chunk, int rounds, int n_pages,
                                            int P_lane, const DevCtx& ctx) {
  constexpr int EB = F8 ? 1 : ElemTraits<T>::bytes;   // bytes per statistic
  constexpr int EPC = 16 / EB;                // elements per 16-byte chunk
  constexpr int RPW = rows_per_warp<F8>();
  constexpr int LPR = 32 / RPW;               // lanes per row
  constexpr int CPL = (2 * D * EB / 16) / LPR;  // chunks per lane per stats row
  constexpr int SPAN = WARPS * RPW;           // pages of one run
  const int p_block = chunk * SPAN * rounds;
  if (p_block >= n_pages) return false;

  const int Hkv = d.num_kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, j = lane % LPR;
  const int p0 = p_block + warp * RPW + grp;
  const int32_t* trow = d.page_table + (long)b * d.page_table_stride;
  auto load = [&](int r, uint4 (&raw)[CPL], int& row_exp) -> bool {
    const int p = p0 + r * SPAN;
    if (r >= rounds || p >= n_pages) return false;
    const int P = r == 0 ? P_lane : trow[p];
    if (P < 0 || P >= d.num_phys_pages) {
      if (j == 0) flag(ctx, KV_DEVERR_BAD_PAGE);
      return false;
    }
    const uint4* row = reinterpret_cast<const uint4*>(
        reinterpret_cast<const char*>(stats) + (((long)P * Hkv + g) * 2 * D) * EB);
#pragma unroll
    for (int u = 0; u < CPL; ++u) raw[u] = __ldg(row + j + LPR * u);
    if constexpr (F8) row_exp = __ldg(stats_exp + (long)P * Hkv + g);
    return true;
  };
  uint4 raw[CPL], nraw[CPL];
  int row_exp = 0, nrow_exp = 0;
  bool ok = load(0, raw, row_exp);

  const int Hq = Hkv * G;
  for (int t = threadIdx.x; t < D; t += WARPS * 32) {
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

  for (int r = 0; r < rounds && p_block + r * SPAN < n_pages; ++r) {   // block-uniform
    const bool nok = load(r + 1, nraw, nrow_exp);
    float acc = 0.f;
    if (ok) {
#pragma unroll
      for (int u = 0; u < CPL; ++u) {
        float f[EPC];
        if constexpr (F8) fp8_chunk_to_f32(raw[u], f);
        else chunk_to_f32<T>(raw[u], f);
        const float* wc = w + (j + LPR * u) * EPC;
#pragma unroll
        for (int e = 0; e < EPC; ++e) acc = fmaf(wc[e], f[e], acc);
      }
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if constexpr (F8) acc *= fp8::pow2(row_exp);
    if (j == 0 && ok) scores[((long)b * Hkv + g) * scores_stride + p0 + r * SPAN] = acc;
#pragma unroll
    for (int u = 0; u < CPL; ++u) raw[u] = nraw[u];
    row_exp = nrow_exp;
    ok = nok;
  }
  return true;
}

template <typename T, int D, bool F8>
__global__ void __launch_bounds__(kScoreWarps * 32)
score_kernel(kv_cache_desc d, const T* __restrict__ q, int G, const void* __restrict__ stats,
             const int8_t* __restrict__ stats_exp, float* __restrict__ scores,
             int scores_stride, int rounds, DevCtx ctx) {
  __shared__ __align__(16) float w[2 * D];    // [Neg | Pos], matching a row's [mn | mx]
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.z, g = blockIdx.y, chunk = blockIdx.x;
  const int P_lane = score_table_entry<kScoreWarps, F8>(d, b, chunk, rounds);
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, d.page_size);
  score_block<T, D, kScoreWarps, F8>(d, q, G, stats, stats_exp, w, scores, scores_stride, b, g,
                                     chunk, rounds, n_pages, P_lane, ctx);
}

// Shared words for the keys of a group of up to max_pages pages (cta_topk.cuh).
__host__ __device__ constexpr size_t select_key_words(int max_pages) {
  return (size_t)cta_key_words(max_pages);
}

template <typename T, int D, bool F8>
__global__ void __launch_bounds__(kSelThreads)
score_select_kernel(kv_cache_desc d, const T* __restrict__ q, int G,
                    const void* __restrict__ stats, const int8_t* __restrict__ stats_exp,
                    float* __restrict__ scores, int scores_stride,
                    double keep_ratio, int budget, int k_max, int32_t* __restrict__ counters,
                    int32_t* __restrict__ sel_idx, int32_t* __restrict__ sel_cnt,
                    int key_words, DevCtx ctx) {
  extern __shared__ __align__(16) uint32_t dyn_words[];     // keys, then candidates
  __shared__ __align__(16) float w[2 * D];
  __shared__ uint32_t hist[kHistWords];
  __shared__ uint32_t misc[8 + kSelWarps];
  __shared__ uint32_t red[cta_red_words<kSelThreads>()];
  __shared__ uint64_t wtot[kSelWarps];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.z, tid = threadIdx.x;
  const int g = blockIdx.y, chunk = blockIdx.x;
  const int P_lane = score_table_entry<kSelWarps, F8>(d, b, chunk, 1);
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, d.page_size);
  const long grp = (long)b * d.num_kv_heads + g;
  if (n_pages == 0) {                         // nothing to score or keep
    if (chunk == 0 && tid == 0) sel_cnt[grp] = 0;
    return;
  }
  if (!score_block<T, D, kSelWarps, F8>(d, q, G, stats, stats_exp, w, scores, scores_stride, b,
                                        g, chunk, 1, n_pages, P_lane, ctx))
    return;

  // ---- the group's last block selects -----------------------------------------------------
  const int blocks = ceil_div(n_pages, kSelWarps * rows_per_warp<F8>());
  __syncthreads();                            // this block's scores are written
  if (tid == 0) {
    __threadfence();                          // release: this block's scores first
    s_last = atomicAdd(&counters[grp], 1) == blocks - 1;
    __threadfence();                          // acquire: the other blocks' scores
  }
  __syncthreads();                            // orders every thread after it
  if (!s_last) return;
  if (tid == 0) counters[grp] = 0;            // ready for the next step
  int k = keep_rule(n_pages, nullptr, b, keep_ratio, budget);
  if (k > k_max) {
    if (tid == 0) flag(ctx, KV_DEVERR_KEEP);
    k = k_max;
  }
  int32_t* out = sel_idx + grp * k_max;
  if (tid == 0) sel_cnt[grp] = k;
  if (k >= n_pages) {                         // every page kept
    for (int i = tid; i < n_pages; i += kSelThreads) out[i] = i;
    return;
  }
  // the group's scores into shared memory: one bulk copy where the row allows it (the other
  // blocks' stores were made visible by the acquire above; the proxy fence orders them before
  // the asynchronous copy), else loads
  const float* srow = scores + grp * scores_stride;
  if (cta_row_bulk_ok(srow, scores_stride)) {
    if (tid == 0) {
      mbar_init(&s_bar, 1);
      fence_mbar_init();
      asm volatile("fence.proxy.async.global;" ::: "memory");
      cta_fill_bulk_issue(dyn_words, srow, n_pages, &s_bar);
    }
    __syncthreads();
    if (!mbar_wait_bounded(&s_bar, 0u, ctx.wait_ns) && tid == 0) flag(ctx, KV_DEVERR_TIMEOUT);
  } else {
    cta_fill_loads<kSelThreads>(dyn_words, srow, n_pages);
  }
  const CtaKeys K = cta_keys_finish<kSelThreads>(dyn_words, n_pages, red);
  uint32_t thr, take_eq;
  cta_threshold<kSelThreads>(K, k, hist, misc, dyn_words + key_words, kSelCandWords, thr,
                             take_eq);
  cta_compact<kSelThreads>(K, thr, take_eq, wtot, 0, k, [&](int p, int pos) { out[pos] = p; });
}

// Multiprocessors of the current device (cached per device).
int device_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <typename T, int D, bool F8>
cudaError_t launch_t(const kv_cache_desc& d, const void* q, int Hq, const void* stats,
                     const int8_t* stats_exp, float* scores, int scores_stride, DevCtx ctx,
                     cudaStream_t s) {
  // runs per block: one, or enough that the grid is about one wave of 8 blocks per SM, but
  // at most kScoreMaxRuns: the grid is sized by the longest sequence, so with sequences of
  // mixed lengths longer blocks would leave the short sequences' SMs idle; several waves of
  // short blocks balance instead
  constexpr int SPAN = kScoreWarps * rows_per_warp<F8>();
  const long rows = (long)d.page_table_stride * d.num_kv_heads * d.batch;
  const long per_run = 8L * device_sms() * SPAN;
  const int rounds = (int)std::min((long)kScoreMaxRuns, std::max(1L, (rows + per_run - 1) / per_run));
  dim3 grid(ceil_div(d.page_table_stride, SPAN * rounds), d.num_kv_heads, d.batch);
  return launch_pdl(score_kernel<T, D, F8>, grid, dim3(kScoreWarps * 32), 0, s, d,
                    static_cast<const T*>(q), Hq / d.num_kv_heads, stats, stats_exp, scores,
                    scores_stride, rounds, ctx);
}

template <typename T, int D, bool F8>
cudaError_t launch_sel_t(const kv_cache_desc& d, const void* q, int Hq, const void* stats,
                         const int8_t* stats_exp, float* scores, int scores_stride,
                         double keep_ratio, int budget, int k_max, int32_t* counters,
                         int32_t* sel_idx, int32_t* sel_cnt, DevCtx ctx, cudaStream_t s) {
  const int key_words = (int)select_key_words(d.page_table_stride);
  const size_t smem = 4 * ((size_t)key_words + kSelCandWords);
  auto kern = score_select_kernel<T, D, F8>;
  // always: the kernel's static shared memory counts against the 48 KB default too
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(ceil_div(d.page_table_stride, kSelWarps * rows_per_warp<F8>()), d.num_kv_heads,
            d.batch);
  return launch_pdl(kern, grid, dim3(kSelThreads), smem, s, d, static_cast<const T*>(q),
                    Hq / d.num_kv_heads, stats, stats_exp, scores, scores_stride, keep_ratio,
                    budget, k_max, counters, sel_idx, sel_cnt, key_words, ctx);
}

}  // namespace

size_t score_select_smem(int page_table_stride) {
  return 4 * (select_key_words(page_table_stride) + kSelCandWords);
}

cudaError_t launch_score_select(const kv_cache_desc& d, const void* q, int Hq,
                                const void* stats, const int8_t* stats_exp, float* scores,
                                int scores_stride, double keep_ratio, int budget, int k_max,
                                int32_t* counters, int32_t* sel_idx, int32_t* sel_cnt,
                                DevCtx ctx, cudaStream_t s) {
#define SKV_SEL(T, D, F8)                                                                   \
  return launch_sel_t<T, D, F8>(d, q, Hq, stats, stats_exp, scores, scores_stride, keep_ratio, \
                                budget, k_max, counters, sel_idx, sel_cnt, ctx, s)
  const bool bf = d.dtype == KV_BF16, f8 = stats_exp != nullptr, wide = d.head_dim == 128;
  if (bf && wide) { if (f8) SKV_SEL(bf16_t, 128, true); SKV_SEL(bf16_t, 128, false); }
  if (bf) { if (f8) SKV_SEL(bf16_t, 64, true); SKV_SEL(bf16_t, 64, false); }
  if (wide) { if (f8) SKV_SEL(float, 128, true); SKV_SEL(float, 128, false); }
  if (f8) SKV_SEL(float, 64, true);
  SKV_SEL(float, 64, false);
#undef SKV_SEL
}

cudaError_t launch_score_pages(const kv_cache_desc& d, const void* q, int Hq,
                               const void* stats, const int8_t* stats_exp, float* scores,
                               int scores_stride, DevCtx ctx, cudaStream_t s) {
#define SKV_SC(T, D, F8) \
  return launch_t<T, D, F8>(d, q, Hq, stats, stats_exp, scores, scores_stride, ctx, s)
  const bool bf = d.dtype == KV_BF16, f8 = stats_exp != nullptr, wide = d.head_dim == 128;
  if (bf && wide) { if (f8) SKV_SC(bf16_t, 128, true); SKV_SC(bf16_t, 128, false); }
  if (bf) { if (f8) SKV_SC(bf16_t, 64, true); SKV_SC(bf16_t, 64, false); }
  if (wide) { if (f8) SKV_SC(float, 128, true); SKV_SC(float, 128, false); }
  if (f8) SKV_SC(float, 64, true);
  SKV_SC(float, 64, false);
#undef SKV_SC
}

}  // namespace skv
