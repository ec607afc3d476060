// Top-k page selection per (sequence, KV head) group.
//
// Sources: "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference",
// abstract (top-k selection of KV entries); "SparDA: Sparse Decoupled Attention for
// Efficient Long-Context LLM Inference", appendix A (the top-k operator over block scores)
// and appendix C (a fixed block budget); "Where Activation Sparsity and KV-Cache Sparsity
// Cross in LLM Decoding", Tables 16-17 (keep ratios r_KV).
//
// Order: score descending, then page index ascending. Output: the kept pages in ascending
// page order.
//
// Structured selection (SparDA section 3.1 and appendix A: initial blocks, a local window
// of recent blocks and top-k blocks joined): the first `sink` and the last `local` pages of
// a group are forced in by giving them the largest key (no finite score maps to it), and
// the keep count becomes max(k, forced). Without scores every other page gets the smallest
// key, which with sink = 0 and local = k is the KV-window baseline ("Where Activation
// Sparsity and KV-Cache Sparsity Cross in LLM Decoding", Tables 3 and 11).
//
// One block per group (512 threads for the block top-k, 1024 for the original form). Scores
// are mapped to unsigned keys whose integer order is the float order. Groups whose keys fit
// in shared memory (up to ~48K pages) take the block top-k of cta_topk.cuh: the score row arrives in shared memory by one bulk copy
// (loads where the row is not 16-byte aligned), the first radix digit starts at the highest
// bit on which the keys differ, the threshold bin's keys are gathered and ranked, and the
// kept pages are written in order by warp ballots after one scan of per-warp counts.
// Longer groups take the original form below: a most-significant-digit radix select (up to
// four 8-bit passes,
// histograms in shared memory with warp-aggregated atomics) finds the k-th largest key T
// and how many keys equal to T are kept (the lowest-indexed ones). Groups of up to 16384
// pages keep their keys in registers (16 per thread) for every pass, so the scores are read
// from memory once; a pass that finds a digit bin holding exactly the keys still needed
// ends the search early (every key at or above that bin is kept). The ordered compaction
// then runs one block-wide exclusive scan of packed (greater-than-T, equal-to-T) counts per
// 1024 consecutive pages, which gives each kept page its output slot, so the output is
// ascending by construction. Longer groups take the same steps reading keys from L2.
#include "cta_topk.cuh"
#include "kv_internal.cuh"

namespace skv {
namespace {

constexpr int kSelCand = 4096;               // gathered keys of the threshold's bin
constexpr int kSelectCtaThreads = 512;       // threads of the block top-k kernel
constexpr size_t kSelectCtaSmemLimit = 227 * 1024;   // shared memory a block may opt into

// Shared words of the block top-k for groups of up to max_pages pages: keys, then candidates.
constexpr size_t select_cta_words(int max_pages) {
  return (size_t)cta_key_words(max_pages) + kSelCand;
}

// Keep count of group (b, g) and its page count n; flags a bad length or keep count.
__device__ __forceinline__ int select_count(const int32_t* seq_lens, int PS, int table_stride,
                                            const int32_t* keep, double keep_ratio, int budget,
                                            int k_max, int sink, int local, int b, int& n,
                                            const DevCtx& ctx) {
  int len = seq_lens[b];
  if (len < 0 || len > table_stride * PS) {
    if (threadIdx.x == 0) flag(ctx, KV_DEVERR_BAD_LEN);
    len = len < 0 ? 0 : table_stride * PS;
  }
  n = ceil_div(len, PS);
  int k = keep_rule(n, keep, b, keep_ratio, budget);
  const int forced = min(n, max(0, sink) + max(0, local));   // [0, sink) and [n - local, n)
  k = max(k, forced);
  if (k > k_max) {
    if (threadIdx.x == 0) flag(ctx, KV_DEVERR_KEEP);
    k = k_max;
  }
  return k;
}

__global__ void __launch_bounds__(kSelectCtaThreads)
select_cta_kernel(const float* __restrict__ scores, int scores_stride,
                  const int32_t* __restrict__ seq_lens, int PS, int Hkv,
                  const int32_t* __restrict__ keep, double keep_ratio, int budget, int k_max,
                  int sink, int local, int32_t* __restrict__ sel_idx,
                  int32_t* __restrict__ sel_cnt, int table_stride, int key_words, DevCtx ctx) {
  extern __shared__ __align__(16) uint32_t words[];           // keys, then candidates
  __shared__ uint32_t hist[kHistWords];
  __shared__ uint32_t misc[8 + kSelectCtaThreads / 32];
  __shared__ uint32_t red[cta_red_words<kSelectCtaThreads>()];
  __shared__ uint64_t wtot[kSelectCtaThreads / 32];
  __shared__ __align__(8) uint64_t s_bar;
  pdl_trigger();
  if (threadIdx.x == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  const int g = blockIdx.x, b = blockIdx.y;
  int n = 0;
  const int k = select_count(seq_lens, PS, table_stride, keep, keep_ratio, budget, k_max, sink,
                             local, b, n, ctx);
  const long grp = (long)b * Hkv + g;
  int32_t* out = sel_idx + grp * k_max;
  if (threadIdx.x == 0) sel_cnt[grp] = k;
  if (k >= n) {                              // keep every page (also n == 0)
    for (int i = threadIdx.x; i < n; i += kSelectCtaThreads) out[i] = i;
    return;
  }
  if (k == 0) return;
  const float* row = scores != nullptr ? scores + grp * scores_stride : nullptr;
  const bool have_row = row != nullptr;
  if (have_row && cta_row_bulk_ok(row, scores_stride)) {   // one bulk copy of the row
    if (threadIdx.x == 0) cta_fill_bulk_issue(words, row, n, &s_bar);
    if (!mbar_wait_bounded(&s_bar, 0u, ctx.wait_ns) && threadIdx.x == 0)
      flag(ctx, KV_DEVERR_TIMEOUT);
  } else if (have_row) {
    cta_fill_loads<kSelectCtaThreads>(words, row, n);
  }
  const CtaKeys K = cta_keys_finish<kSelectCtaThreads, true>(
      words, n, red, [&](int i, uint32_t key) -> uint32_t {
        if (i < sink || i >= n - local) return 0xffffffffu;   // forced in
        return have_row ? key : 0u;
      });
  uint32_t T, take_eq;
  cta_threshold<kSelectCtaThreads>(K, k, hist, misc, words + key_words, kSelCand, T, take_eq);
  cta_compact<kSelectCtaThreads>(K, T, take_eq, wtot, 0, k, [&](int p, int pos) { out[pos] = p; });
}

// Block-wide exclusive scan of a 64-bit value (two packed 32-bit counters).
__device__ __forceinline__ uint64_t block_exclusive_scan(uint64_t v, uint64_t* warp_tot,
                                                         uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint64_t t = warp_tot[lane];
    uint64_t ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += y;
    }
    warp_tot[lane] = ti - t;                 // exclusive prefix of warp totals
    if (lane == 31) *total = ti;
  }
  __syncthreads();
  return warp_tot[warp] + incl - v;
}

constexpr int kRegKeys = 16;                 // keys per thread kept in registers

// REG: keys live in registers (n <= kRegKeys * kSelectThreads); otherwise each pass
// re-reads them from the score row (L2-resident).
template <bool REG>
__global__ void __launch_bounds__(kSelectThreads)
select_kernel(const float* __restrict__ scores, int scores_stride,
              const int32_t* __restrict__ seq_lens, int PS, int Hkv,
              const int32_t* __restrict__ keep, double keep_ratio, int budget, int k_max,
              int sink, int local, int32_t* __restrict__ sel_idx,
              int32_t* __restrict__ sel_cnt, int table_stride, DevCtx ctx) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_remaining, s_exact;
  __shared__ uint64_t warp_tot[32];
  __shared__ uint64_t s_total;
  pdl_trigger();
  pdl_wait();

  const int g = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int len = seq_lens[b];
  if (len < 0 || len > table_stride * PS) {
    if (tid == 0) flag(ctx, KV_DEVERR_BAD_LEN);
    len = len < 0 ? 0 : table_stride * PS;
  }
  const int n = ceil_div(len, PS);
  int k = keep_rule(n, keep, b, keep_ratio, budget);
  const int forced = min(n, max(0, sink) + max(0, local));   // [0, sink) and [n - local, n)
  k = max(k, forced);
  if (k > k_max) {
    if (tid == 0) flag(ctx, KV_DEVERR_KEEP);
    k = k_max;
  }
  const long grp = (long)b * Hkv + g;
  const float* row = scores != nullptr ? scores + grp * scores_stride : nullptr;
  auto key_at = [&](int i) -> uint32_t {
    if (i < sink || i >= n - local) return 0xffffffffu;   // forced in
    return row != nullptr ? score_order_key(row[i]) : 0u;
  };
  int32_t* out = sel_idx + grp * k_max;
  if (tid == 0) sel_cnt[grp] = k;

  if (k >= n) {                              // keep every page (also n == 0)
    for (int i = tid; i < n; i += kSelectThreads) out[i] = i;
    return;
  }
  if (k == 0) return;

  const int nj = ceil_div(n, kSelectThreads);   // key slices of 1024 consecutive pages
  uint32_t rk[REG ? kRegKeys : 1];
  if constexpr (REG) {
#pragma unroll
    for (int j = 0; j < kRegKeys; ++j) {
      const int i = j * kSelectThreads + tid;
      rk[j] = i < n ? key_at(i) : 0u;
    }
  }
  auto key_of = [&](int j) -> uint32_t {
    if constexpr (REG) return rk[j];
    else return key_at(j * kSelectThreads + tid);
  };

  // ---- radix select of the k-th largest key -------------------------------------------
  uint32_t prefix = 0, mask = 0, remaining = (uint32_t)k;
  bool exact = false;
  for (int shift = 24; shift >= 0 && !exact; shift -= 8) {
    for (int i = tid; i < 256; i += kSelectThreads) hist[i] = 0;
    if (tid == 0) s_exact = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < (REG ? kRegKeys : 1); ++j) {
      for (int jj = j; jj < (REG ? j + 1 : nj); ++jj) {
        if (REG && jj >= nj) break;
        const int i = jj * kSelectThreads + tid;
        uint32_t digit = 256;                // 256 = not counted in this pass
        if (i < n) {
          const uint32_t key = key_of(jj);
          if ((key & mask) == prefix) digit = (key >> shift) & 255u;
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        if (digit < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t c[8], lane_sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) { c[e] = hist[lane * 8 + e]; lane_sum += c[e]; }
      uint32_t incl = lane_sum;             // keys in digits >= this lane's lowest bin
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      uint32_t above = incl - lane_sum;     // keys in digits above this lane's bins
      if (above < remaining && remaining <= incl) {
#pragma unroll
        for (int e = 7; e >= 0; --e) {
          if (above + c[e] >= remaining) {
            s_prefix = prefix | ((uint32_t)(lane * 8 + e) << shift);
            s_remaining = remaining - above;
            s_exact = (above + c[e] == remaining) ? 1u : 0u;
            break;
          }
          above += c[e];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    exact = s_exact != 0;
    mask |= 255u << shift;
  }
  // Keep key > T, and the first take_eq keys equal to T in page order. When a bin held
  // exactly the keys still needed, every key >= its (zero-extended) prefix is kept.
  const uint32_t T = prefix;
  const uint32_t take_eq = exact ? 0xffffffffu : remaining;

  // ---- ordered compaction, one slice of 1024 pages at a time ------------------------------
  uint32_t carry_gt = 0, carry_eq = 0;
  for (int j = 0; j < nj; ++j) {
    const int i = j * kSelectThreads + tid;
    uint32_t key = 0;
    bool valid = i < n;
    if constexpr (REG) {
#pragma unroll
      for (int jj = 0; jj < kRegKeys; ++jj) key = (jj == j) ? rk[jj] : key;
    } else {
      if (valid) key = key_at(i);
    }
    const uint32_t gt = valid && key > T;
    const uint32_t eq = valid && key == T;
    const uint64_t ex = block_exclusive_scan(((uint64_t)gt << 32) | eq, warp_tot, &s_total);
    const uint32_t gt_before = carry_gt + (uint32_t)(ex >> 32);
    const uint32_t eq_before = carry_eq + (uint32_t)(ex & 0xffffffffu);
    if (gt) out[gt_before + min(eq_before, take_eq)] = i;
    else if (eq && eq_before < take_eq) out[gt_before + eq_before] = i;
    carry_gt += (uint32_t)(s_total >> 32);
    carry_eq += (uint32_t)(s_total & 0xffffffffu);
    __syncthreads();                         // warp_tot / s_total are rewritten next slice
  }
}

}  // namespace

cudaError_t launch_select_topk(const float* scores, int scores_stride, const int32_t* seq_lens,
                               int page_size, int batch, int Hkv, const int32_t* keep,
                               double keep_ratio, int budget_pages, int k_max, int sink,
                               int local, int32_t* sel_idx, int32_t* sel_cnt,
                               int page_table_stride, DevCtx ctx, cudaStream_t s) {
  dim3 grid(Hkv, batch);
  const size_t words = select_cta_words(page_table_stride);
  const size_t smem = 4 * words;
  if (smem + 4 * (kHistWords + 8 + kSelectCtaThreads / 32) + 8 * (kSelectCtaThreads / 32) +
          1024 <= kSelectCtaSmemLimit) {
    // always: the kernel's static shared memory counts against the 48 KB default too
    cudaError_t e = cudaFuncSetAttribute(select_cta_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(select_cta_kernel, grid, dim3(kSelectCtaThreads), smem, s, scores,
                      scores_stride, seq_lens, page_size, Hkv, keep, keep_ratio, budget_pages,
                      k_max, sink, local, sel_idx, sel_cnt, page_table_stride,
                      (int)(words - kSelCand), ctx);
  }
  auto kern = page_table_stride <= kRegKeys * kSelectThreads ? select_kernel<true>
                                                              : select_kernel<false>;
  return launch_pdl(kern, grid, dim3(kSelectThreads), 0, s, scores, scores_stride, seq_lens,
                    page_size, Hkv, keep, keep_ratio, budget_pages, k_max, sink, local, sel_idx,
                    sel_cnt, page_table_stride, ctx);
}

}  // namespace skv
