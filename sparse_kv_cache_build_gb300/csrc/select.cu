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
// One 1024-thread block per group. Scores are mapped to unsigned keys whose integer order
// is the float order, and a most-significant-digit radix select (four 8-bit passes over
// the group's scores, histograms in shared memory with warp-aggregated atomics) finds the
// k-th largest key T and how many keys equal to T are kept (the lowest-indexed ones). A
// final ordered pass stages 8192 keys at a time in shared memory, each thread scanning 8
// consecutive keys; one block-wide exclusive scan of (greater-than-T, equal-to-T) counts
// gives each kept page its output slot, so the output is ascending by construction. The
// score rows are small (4 bytes per page) and stay in L2 across the passes.
#include "kv_internal.cuh"

namespace skv {
namespace {

constexpr int kItems = kSelectChunk / kSelectThreads;   // 8 keys per thread per chunk

__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t u = __float_as_uint(s + 0.0f);          // -0 -> +0: equal scores, equal keys
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int keep_count(int n, const int32_t* keep, int b, double ratio,
                                          int budget) {
  if (n <= 0) return 0;
  if (keep != nullptr) {
    const int k = keep[b];
    return k < 0 ? 0 : (k > n ? n : k);
  }
  if (budget > 0) return budget < n ? budget : n;
  if (ratio >= 1.0) return n;
  double c = ceil(ratio * (double)n - 1e-9);
  int k = (int)c;
  k = k < 1 ? 1 : k;
  return k < n ? k : n;
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

__global__ void __launch_bounds__(kSelectThreads)
select_kernel(const float* __restrict__ scores, int scores_stride,
              const int32_t* __restrict__ seq_lens, int PS, int Hkv,
              const int32_t* __restrict__ keep, double keep_ratio, int budget, int k_max,
              int32_t* __restrict__ sel_idx, int32_t* __restrict__ sel_cnt, int table_stride,
              DevCtx ctx) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_remaining;
  __shared__ uint64_t warp_tot[32];
  __shared__ uint64_t s_total;
  __shared__ uint32_t keys[kSelectChunk];

  const int g = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int len = seq_lens[b];
  if (len < 0 || len > table_stride * PS) {
    if (tid == 0) flag(ctx, KV_DEVERR_BAD_LEN);
    len = len < 0 ? 0 : table_stride * PS;
  }
  const int n = ceil_div(len, PS);
  int k = keep_count(n, keep, b, keep_ratio, budget);
  if (k > k_max) {
    if (tid == 0) flag(ctx, KV_DEVERR_KEEP);
    k = k_max;
  }
  const long grp = (long)b * Hkv + g;
  const float* row = scores + grp * scores_stride;
  int32_t* out = sel_idx + grp * k_max;
  if (tid == 0) sel_cnt[grp] = k;

  if (k >= n) {                              // keep every page (also n == 0)
    for (int i = tid; i < n; i += kSelectThreads) out[i] = i;
    return;
  }
  if (k == 0) return;

  // ---- radix select of the k-th largest key -------------------------------------------
  uint32_t prefix = 0, mask = 0, remaining = (uint32_t)k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelectThreads) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kSelectThreads) {
      const int i = base + tid;
      uint32_t digit = 256;                  // 256 = not counted in this pass
      if (i < n) {
        const uint32_t key = order_key(row[i]);
        if ((key & mask) == prefix) digit = (key >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (digit < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
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
            break;
          }
          above += c[e];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;                 // the k-th largest key
  const uint32_t take_eq = remaining;        // keys equal to T that are kept (>= 1)

  // ---- ordered compaction ---------------------------------------------------------------
  uint32_t carry_gt = 0, carry_eq = 0;
  for (int c0 = 0; c0 < n; c0 += kSelectChunk) {
    for (int i = tid; i < kSelectChunk; i += kSelectThreads)
      keys[i] = (c0 + i < n) ? order_key(row[c0 + i]) : 0u;
    __syncthreads();
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int e = 0; e < kItems; ++e) {
      const int idx = tid * kItems + e;
      if (c0 + idx < n) {
        const uint32_t key = keys[idx];
        gt += key > T;
        eq += key == T;
      }
    }
    const uint64_t ex = block_exclusive_scan(((uint64_t)gt << 32) | eq, warp_tot, &s_total);
    uint32_t gt_before = carry_gt + (uint32_t)(ex >> 32);
    uint32_t eq_before = carry_eq + (uint32_t)(ex & 0xffffffffu);
#pragma unroll
    for (int e = 0; e < kItems; ++e) {
      const int idx = tid * kItems + e;
      if (c0 + idx < n) {
        const uint32_t key = keys[idx];
        if (key > T) {
          out[gt_before + min(eq_before, take_eq)] = c0 + idx;
          ++gt_before;
        } else if (key == T) {
          if (eq_before < take_eq) out[gt_before + eq_before] = c0 + idx;
          ++eq_before;
        }
      }
    }
    carry_gt += (uint32_t)(s_total >> 32);
    carry_eq += (uint32_t)(s_total & 0xffffffffu);
    __syncthreads();                         // keys[] and s_total are reused next chunk
  }
}

}  // namespace

cudaError_t launch_select_topk(const float* scores, int scores_stride, const int32_t* seq_lens,
                               int page_size, int batch, int Hkv, const int32_t* keep,
                               double keep_ratio, int budget_pages, int k_max,
                               int32_t* sel_idx, int32_t* sel_cnt, int page_table_stride,
                               DevCtx ctx, cudaStream_t s) {
  dim3 grid(Hkv, batch);
  select_kernel<<<grid, kSelectThreads, 0, s>>>(scores, scores_stride, seq_lens, page_size,
                                                Hkv, keep, keep_ratio, budget_pages, k_max,
                                                sel_idx, sel_cnt, page_table_stride, ctx);
  return cudaGetLastError();
}

}  // namespace skv
