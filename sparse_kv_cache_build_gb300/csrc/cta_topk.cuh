// Top-k selection by one thread block over a group's page scores held in shared memory:
// the rule of select.cu (score descending, page index ascending), reshaped so that every
// split CTA of the attention kernel can pick its own run of the selected list without a
// separate launch. The scores of a group are small (4 B per page) and L2-resident after the
// score pass, so each of the group's S CTAs redoing this work costs less than a kernel
// boundary, provided the work is latency-lean:
//
//   * keys are loaded in batches of sixteen independent loads per thread;
//   * the load also ORs (key ^ key of page 0), so the bits above the highest differing
//     bit are known to be common and the first radix digit starts there;
//   * after one 8-bit pass the keys of the threshold's bin are gathered (order does not
//     matter for the threshold), and if they are at most one per thread each finds its
//     exact rank among them directly; larger bins take further radix passes over the
//     gathered keys only;
//   * histograms take plain shared-memory atomics into a bank-padded array (warp-wide
//     match instructions cost hundreds of cycles when a warp holds many distinct digits),
//     and the gather writes through a block scan of per-thread counts, with no atomic whose
//     result a thread waits on.
//
// Layout: thread t owns the contiguous pages [t*ipt, (t+1)*ipt) (ipt = ceil(n / NT)), stored
// at word offset t*stride with an odd stride, so that the NT threads walking their own
// chunks in step hit NT different banks.
#pragma once

#include "kv_internal.cuh"

namespace skv {

struct CtaKeys {
  uint32_t* keys;   // shared, NT * stride words
  int n, ipt, stride;
  uint32_t key0;    // key of page 0
  uint32_t diff;    // OR over the pages of (key ^ key0): the bits on which the keys differ
  // word index of page i
  __device__ __forceinline__ int slot(int i) const {
    const int t = i / ipt;
    return t * stride + (i - t * ipt);
  }
};

// The padded layout of n keys over NT threads (keys not loaded).
template <int NT>
__device__ __forceinline__ CtaKeys cta_key_layout(uint32_t* smem_words, int n) {
  CtaKeys K;
  K.keys = smem_words;
  K.n = n;
  K.ipt = ceil_div(n, NT);
  K.stride = K.ipt | 1;
  K.key0 = 0u;
  K.diff = 0u;
  return K;
}

// Shared words the layout of n keys over NT threads spans.
template <int NT>
__host__ __device__ constexpr int cta_key_words(int n) {
  return NT * (((n + NT - 1) / NT) | 1);
}

// Fill K.key0 and K.diff from keys already in the layout (visible to every thread); red:
// NT/32 words of scratch. Ends with __syncthreads.
template <int NT>
__device__ __forceinline__ void cta_key_diff(CtaKeys& K, uint32_t* red) {
  const int tid = threadIdx.x;
  const uint32_t k0 = K.keys[0];
  const int a0 = min(K.n, tid * K.ipt), a1 = min(K.n, a0 + K.ipt);
  uint32_t orv = 0u;
#pragma unroll 4
  for (int i = a0; i < a1; ++i) orv |= K.keys[tid * K.stride + (i - a0)] ^ k0;
  orv = __reduce_or_sync(0xffffffffu, orv);
  if ((tid & 31) == 0) red[tid >> 5] = orv;
  __syncthreads();
  uint32_t diff = 0u;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) diff |= red[w];
  K.key0 = k0;
  K.diff = diff;
}

// Load the n scores of a row as order keys into the padded layout; red: NT/32 words of
// scratch. Ends with __syncthreads (the keys and K.diff are then visible to every thread).
template <int NT>
__device__ __forceinline__ CtaKeys cta_load_keys(const float* row, int n, uint32_t* smem_words,
                                                 uint32_t* red) {
  constexpr int kBatch = 16;
  CtaKeys K = cta_key_layout<NT>(smem_words, n);
  const int tid = threadIdx.x;
  const uint32_t k0 = score_order_key(__ldcg(row));
  uint32_t orv = 0u;
  for (int base = 0; base < n; base += NT * kBatch) {
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * NT + tid;
      v[u] = i < n ? __ldcg(row + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * NT + tid;
      if (i < n) {
        const uint32_t key = score_order_key(v[u]);
        K.keys[K.slot(i)] = key;
        orv |= key ^ k0;
      }
    }
  }
  orv = __reduce_or_sync(0xffffffffu, orv);
  if ((tid & 31) == 0) red[tid >> 5] = orv;
  __syncthreads();
  uint32_t diff = 0u;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) diff |= red[w];
  K.key0 = k0;
  K.diff = diff;
  return K;
}

// Histogram words: 256 bins, one pad word after every 32 (conflict-free reads of eight
// consecutive bins per lane).
constexpr int kHistWords = 256 + 8;

namespace topk_detail {

__device__ __forceinline__ int hslot(uint32_t bin) { return (int)(bin + (bin >> 5)); }

// Exclusive block scan of one count per thread; wsum: NT/32 words. Every thread gets the
// total. Ends with the block synchronised once (wsum is not reused before the next sync).
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t before = 0u, all = 0u;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const uint32_t x = wsum[w];
    before += w < warp ? x : 0u;
    all += x;
  }
  total = all;
  return before + incl - v;
}

// Warp 0: from the top bin down, the bin holding the remaining-th largest key.
// misc[0] = bin, misc[1] = rank still needed inside it, misc[2] = the bin's count.
__device__ __forceinline__ void pick_bin(const uint32_t* hist, uint32_t remaining,
                                         uint32_t* misc) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8], lane_sum = 0u;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    c[e] = hist[hslot((uint32_t)(lane * 8 + e))];
    lane_sum += c[e];
  }
  uint32_t incl = lane_sum;                 // this lane's bins and every higher lane's
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  uint32_t above = incl - lane_sum;
  if (above < remaining && remaining <= incl) {
#pragma unroll
    for (int e = 7; e >= 0; --e) {
      if (above + c[e] >= remaining) {
        misc[0] = (uint32_t)(lane * 8 + e);
        misc[1] = remaining - above;
        misc[2] = c[e];
        break;
      }
      above += c[e];
    }
  }
}

}  // namespace topk_detail

// Threshold of the top k keys (0 < k < n). On return (block-uniform) the kept keys are those
// > T and the first take_eq keys == T in page order. hist: kHistWords words; misc: 8 +
// NT/32 words; cand: cand_cap words of 16-byte aligned scratch for the gathered keys of
// the threshold's bin.
template <int NT>
__device__ void cta_threshold(const CtaKeys& K, int k, uint32_t* hist, uint32_t* misc,
                              uint32_t* cand, int cand_cap, uint32_t& T, uint32_t& take_eq) {
  using namespace topk_detail;
  const int tid = threadIdx.x;
  if (K.diff == 0u) {                        // every key equal: the first k pages
    T = K.key0;
    take_eq = (uint32_t)k;
    return;
  }
  int top = 31 - __clz(K.diff);              // highest bit on which keys differ
  uint32_t mask = top == 31 ? 0u : ~((2u << top) - 1u);
  uint32_t prefix = K.key0 & mask;           // the bits every key shares
  uint32_t remaining = (uint32_t)k;
  int ncand = -1;                            // -1: histogram the chunks, else cand[0, ncand)
  const int a0 = min(K.n, tid * K.ipt), a1 = min(K.n, a0 + K.ipt);
  for (;;) {
    const int lo = top >= 7 ? top - 7 : 0;
    const uint32_t dmask = (2u << (top - lo)) - 1u;      // digit bits [lo, top]
    for (int i = tid; i < kHistWords; i += NT) hist[i] = 0u;
    __syncthreads();
    if (ncand < 0) {
#pragma unroll 4
      for (int i = a0; i < a1; ++i) {
        const uint32_t key = K.keys[tid * K.stride + (i - a0)];
        if ((key & mask) == prefix) atomicAdd(&hist[hslot((key >> lo) & dmask)], 1u);
      }
    } else {
      for (int i = tid; i < ncand; i += NT) {
        const uint32_t key = cand[i];
        if ((key & mask) == prefix) atomicAdd(&hist[hslot((key >> lo) & dmask)], 1u);
      }
    }
    __syncthreads();
    if (tid < 32) pick_bin(hist, remaining, misc);
    __syncthreads();
    const uint32_t bin = misc[0];
    remaining = misc[1];
    const uint32_t bin_count = misc[2];
    __syncthreads();                         // misc is rewritten below
    prefix |= bin << lo;
    mask |= dmask << lo;
    if (remaining == bin_count || lo == 0) { // the whole bin is kept, or the key is complete
      T = prefix;
      take_eq = remaining == bin_count ? 0xffffffffu : remaining;
      return;
    }
    top = lo - 1;
    if (ncand < 0 && (int)bin_count <= cand_cap) {
      // gather the bin's keys (page order, through a scan of per-thread counts)
      uint32_t mine = 0u, total = 0u;
#pragma unroll 4
      for (int i = a0; i < a1; ++i) mine += (K.keys[tid * K.stride + (i - a0)] & mask) == prefix;
      uint32_t at = block_excl_scan<NT>(mine, misc + 8, total);
      for (int i = a0; i < a1 && mine != 0u; ++i) {
        const uint32_t key = K.keys[tid * K.stride + (i - a0)];
        if ((key & mask) == prefix) {
          cand[at++] = key;
          --mine;
        }
      }
      __syncthreads();
      ncand = (int)bin_count;
      if (ncand <= NT) {
        // exact rank of each gathered key among the others (cand is 16-byte aligned;
        // four keys per broadcast load)
        if (tid < ncand) {
          const uint32_t c = cand[tid];
          uint32_t gt = 0u, eq = 0u;
          int j = 0;
          for (; j + 4 <= ncand; j += 4) {
            const uint4 o = *reinterpret_cast<const uint4*>(cand + j);
            gt += (o.x > c) + (o.y > c) + (o.z > c) + (o.w > c);
            eq += (o.x == c) + (o.y == c) + (o.z == c) + (o.w == c);
          }
          for (; j < ncand; ++j) {
            const uint32_t o = cand[j];
            gt += o > c;
            eq += o == c;
          }
          if (gt < remaining && remaining <= gt + eq) {   // equal keys write equal values
            misc[5] = c;
            misc[6] = remaining - gt;
          }
        }
        __syncthreads();
        T = misc[5];
        take_eq = misc[6];
        return;
      }
    }
  }
}

// Ordered compaction: calls emit(page, pos) for every kept page, pos = its position in the
// ascending kept list. wtot: NT/32 doublewords of scratch.
template <int NT, typename F>
__device__ void cta_compact(const CtaKeys& K, uint32_t T, uint32_t take_eq, uint64_t* wtot,
                            F&& emit) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int a0 = min(K.n, tid * K.ipt), a1 = min(K.n, a0 + K.ipt);
  uint32_t gt = 0, eq = 0;
#pragma unroll 4
  for (int i = a0; i < a1; ++i) {
    const uint32_t key = K.keys[tid * K.stride + (i - a0)];
    gt += key > T;
    eq += key == T;
  }
  const uint64_t v = ((uint64_t)gt << 32) | eq;
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  uint64_t before = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) before += (w < warp) ? wtot[w] : 0ull;
  __syncthreads();
  const uint64_t ex = before + incl - v;
  uint32_t gt_before = (uint32_t)(ex >> 32), eq_before = (uint32_t)(ex & 0xffffffffu);
#pragma unroll 4
  for (int i = a0; i < a1; ++i) {
    const uint32_t key = K.keys[tid * K.stride + (i - a0)];
    if (key > T) {
      emit(i, (int)(gt_before + min(eq_before, take_eq)));
      ++gt_before;
    } else if (key == T) {
      if (eq_before < take_eq) emit(i, (int)(gt_before + eq_before));
      ++eq_before;
    }
  }
}

}  // namespace skv
