// Top-k selection by one thread block over a group's page scores held in shared memory:
// the rule of select.cu (score descending, page index ascending), reshaped so that every
// split CTA of the attention kernel can pick its own run of the selected list without a
// separate launch. The scores of a group are small (4 B per page) and L2-resident after the
// score pass, so each of the group's S CTAs redoing this work costs less than a kernel
// boundary, provided the work is latency-lean. Measured on this part, what costs is the
// number of dependent steps, not the arithmetic:
//
//   * the keys arrive by one bulk asynchronous copy of the score row into shared memory
//     where the row allows it (16-byte aligned, a multiple of four floats per row): one
//     request instead of n/NT load instructions per thread (a 16K-page row lands in
//     ~0.7 us, against ~5.7 us for per-thread loads from 128 threads); otherwise by
//     per-thread loads, sixteen in flight;
//   * keys are stored contiguously in page order; a pass has thread t read the 16-byte
//     groups t, t + NT, ... of four keys (conflict-free), a batch of four groups into
//     registers before any shared store or atomic, so no shared-memory load waits behind a
//     store or atomic it might alias;
//   * the bits on which keys differ are OR ^ AND over the keys, so the first radix digit
//     starts at the highest of them; digits are 11 bits wide, so that after the first pass
//     the threshold's bin usually holds fewer keys than the block has threads (a pass
//     costs several block-wide steps; more bins cost only a wider histogram);
//   * after one digit pass the keys of the threshold's bin are gathered in any order (the
//     threshold does not need it), each warp reserving its slots with one atomic, so this
//     costs one pass and no block scan; if they are at most one per thread each finds its
//     exact rank among them directly; larger bins take further radix passes over the
//     gathered keys only;
//   * a pass over whole 16-byte groups carries no per-key bound test; the partial last
//     group goes to one thread (a bound test on every key made a count loop ~6x slower);
//   * histograms take plain shared-memory atomics into a bank-padded array (warp-wide
//     match instructions cost hundreds of cycles when a warp holds many distinct digits);
//     their throughput (~1.6 keys per clock per SM) is what a pass over many keys costs, so
//     long groups keeping few pages histogram only the keys at or above a bound taken from
//     a sample (cta_threshold), gathered with their pages in page order;
//   * block reductions read the per-warp words one per lane and reduce with warp
//     instructions, rather than every thread reading every warp's word;
//   * the ordered compaction of the whole list gives each warp a contiguous segment of
//     pages, walked 32 at a time with ballots, after one scan of the per-warp counts; the
//     compaction of a short window of positions (one attention CTA's run) gives each thread
//     a contiguous segment of 16-byte groups instead, counted with a rotated start (no
//     bank conflicts) and one block scan, and one warp walks from the segment holding the
//     window's first position, four rows a step, so its cost does not depend on where the
//     window lies; after the sample filter, a window is compacted from the page-ordered
//     candidates alone (cta_compact_list).
#pragma once

#include "kv_internal.cuh"

namespace skv {

struct CtaKeys {
  uint32_t* keys;   // shared, 16-byte aligned, cta_key_words(n) words: keys[i] is page i's
  int n;            // key for i < n
  uint32_t common;  // AND over the keys: every bit on which they agree has its shared value
  uint32_t diff;    // OR ^ AND over the keys: the bits on which they differ
};

// The keys >= some bound L, with their pages, in page order (cta_threshold's prefilter): every
// kept key is among them, so the kept list can be compacted from these alone. n < 0: none.
struct CtaCand {
  const uint32_t* keys;
  const int32_t* pages;
  int n;
};

// Shared words the keys of n pages take (bulk copies move whole 16-byte chunks).
__host__ __device__ constexpr int cta_key_words(int n) { return (n + 3) & ~3; }

// Shared words of the reduction scratch (`red`) that cta_keys_finish needs.
template <int NT>
__host__ __device__ constexpr int cta_red_words() { return 2 * (NT / 32); }

// Whether a row of 4-byte entries can be bulk-copied: the row 16-byte aligned and the row
// stride a multiple of four entries (so the copy's rounding up to 16 bytes stays inside the
// row).
__device__ __forceinline__ bool cta_row_bulk_ok(const void* row, long row_stride) {
  return (reinterpret_cast<uintptr_t>(row) & 15u) == 0 && (row_stride & 3) == 0;
}

// One thread: copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// memory into shared memory, completion counted on bar, whose expected transaction count the
// caller raised by `bytes` (mbar_arrive_expect_tx) in the same phase.
__device__ __forceinline__ void cta_bulk_copy(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  constexpr uint32_t kChunk = 32768;
  for (uint32_t off = 0; off < bytes; off += kChunk) {
    const uint32_t len = bytes - off < kChunk ? bytes - off : kChunk;
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(reinterpret_cast<char*>(dst) + off)),
          "l"(reinterpret_cast<const char*>(src) + off), "r"(len), "r"(smem_addr(bar))
        : "memory");
  }
}

// One thread: start the copy of the raw bits of row[0, cta_key_words(n)) into keys, counted
// on bar (initialised with count 1 and visible to the block). The row must pass
// cta_row_bulk_ok.
__device__ __forceinline__ void cta_fill_bulk_issue(uint32_t* keys, const float* row, int n,
                                                    uint64_t* bar) {
  const uint32_t bytes = 4u * (uint32_t)cta_key_words(n);
  mbar_arrive_expect_tx(bar, bytes);
  if (bytes != 0u) cta_bulk_copy(keys, row, bytes, bar);
}

// Every thread: copy the raw bits of row[0, n) (any alignment) into keys with loads, sixteen in
// flight per thread. Thread t writes the 16-byte groups of keys t, t + NT, ..., the ones
// cta_keys_finish has it read, so no barrier is needed between the two (padding past n is 0).
template <int NT>
__device__ __forceinline__ void cta_fill_loads(uint32_t* keys, const float* row, int n) {
  constexpr int kB4 = 4;
  const int tid = threadIdx.x;
  const int n4 = (n + 3) >> 2;
  uint4* k4 = reinterpret_cast<uint4*>(keys);
  for (int base = 0; base < n4; base += NT * kB4) {
    uint32_t v[kB4][4];
#pragma unroll
    for (int u = 0; u < kB4; ++u) {
      const int j = base + u * NT + tid;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        v[u][e] = 4 * j + e < n ? __float_as_uint(__ldcg(row + 4 * j + e)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kB4; ++u) {
      const int j = base + u * NT + tid;
      if (j < n4) k4[j] = make_uint4(v[u][0], v[u][1], v[u][2], v[u][3]);
    }
  }
}

// Every thread: f(i, key) for its share of keys[0, n) (16-byte aligned, cta_key_words(n)
// words), read four at a time: thread t takes the whole 16-byte groups t, t + NT, ...; the
// loads of a batch are all issued before f runs on any of them (f may store or do atomics).
// The keys of a partial last group (n not a multiple of four) go to that group's thread t
// after its whole groups. The order in which a thread visits its keys is not page order.
template <int NT, typename F>
__device__ __forceinline__ void cta_for_keys4(const uint32_t* keys, int n, F&& f) {
  constexpr int kB4 = 4;
  const int tid = threadIdx.x;
  const int nf = n >> 2;                                   // whole groups
  const uint4* k4 = reinterpret_cast<const uint4*>(keys);
  for (int base = 0; base < nf; base += NT * kB4) {
    uint4 v[kB4];
#pragma unroll
    for (int u = 0; u < kB4; ++u) {
      const int j = base + u * NT + tid;
      v[u] = j < nf ? k4[j] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kB4; ++u) {
      const int j = base + u * NT + tid;
      if (j < nf) {
        f(4 * j, v[u].x);
        f(4 * j + 1, v[u].y);
        f(4 * j + 2, v[u].z);
        f(4 * j + 3, v[u].w);
      }
    }
  }
  if ((n & 3) != 0 && tid == nf % NT)
    for (int i = 4 * nf; i < n; ++i) f(i, keys[i]);
}

// Make keys[0, n) final and find the bits on which they differ. CONVERT: the words hold raw
// score bits and become fix(i, score_order_key(score_i)); otherwise they already are keys.
// red: cta_red_words<NT>() words. Ends with __syncthreads (the keys are then visible to every
// thread).
template <int NT, bool CONVERT, typename Fix>
__device__ __forceinline__ CtaKeys cta_keys_finish(uint32_t* keys, int n, uint32_t* red, Fix fix) {
  constexpr int kB4 = 4, NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t orv = 0u, andv = 0xffffffffu;
  auto one = [&](uint32_t& w, int i) {
    if constexpr (CONVERT) w = fix(i, score_order_key(__uint_as_float(w)));
    orv |= w;
    andv &= w;
  };
  const int nf = n >> 2;                                   // whole groups
  uint4* k4 = reinterpret_cast<uint4*>(keys);
  for (int base = 0; base < nf; base += NT * kB4) {
    uint4 v[kB4];
#pragma unroll
    for (int u = 0; u < kB4; ++u) {
      const int j = base + u * NT + tid;
      v[u] = j < nf ? k4[j] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kB4; ++u) {
      const int j = base + u * NT + tid;
      if (j < nf) {
        one(v[u].x, 4 * j);
        one(v[u].y, 4 * j + 1);
        one(v[u].z, 4 * j + 2);
        one(v[u].w, 4 * j + 3);
        if constexpr (CONVERT) k4[j] = v[u];
      }
    }
  }
  if ((n & 3) != 0 && tid == nf % NT) {                    // the partial last group
    for (int i = 4 * nf; i < n; ++i) {
      uint32_t w = keys[i];
      one(w, i);
      if constexpr (CONVERT) keys[i] = w;
    }
  }
  orv = __reduce_or_sync(0xffffffffu, orv);
  andv = __reduce_and_sync(0xffffffffu, andv);
  if (lane == 0) {
    red[warp] = orv;
    red[NW + warp] = andv;
  }
  __syncthreads();
  const uint32_t o = __reduce_or_sync(0xffffffffu, lane < NW ? red[lane] : 0u);
  const uint32_t a = __reduce_and_sync(0xffffffffu, lane < NW ? red[NW + lane] : 0xffffffffu);
  CtaKeys K;
  K.keys = keys;
  K.n = n;
  K.common = a;
  K.diff = o ^ a;
  return K;
}

// The raw score bits in keys become their order keys.
template <int NT>
__device__ __forceinline__ CtaKeys cta_keys_finish(uint32_t* keys, int n, uint32_t* red) {
  return cta_keys_finish<NT, true>(keys, n, red, [](int, uint32_t key) { return key; });
}

// Radix digits of kDigitBits bits; histogram words: one pad word after every 32 bins.
constexpr int kDigitBits = 11;
constexpr int kBins = 1 << kDigitBits;
constexpr int kHistWords = kBins + kBins / 32;

namespace topk_detail {

constexpr int kB = 16;   // keys per thread per register batch

__device__ __forceinline__ int hslot(uint32_t bin) { return (int)(bin + (bin >> 5)); }

// Exclusive block scan of one count per thread; wsum: NT/32 words. Every thread gets the
// total. Ends with the block synchronised once (wsum is not reused before the next sync).
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  const uint32_t wv = lane < NW ? wsum[lane] : 0u;
  total = __reduce_add_sync(0xffffffffu, wv);
  return __reduce_add_sync(0xffffffffu, lane < warp ? wv : 0u) + incl - v;
}

// Every thread: from the top bin down, the bin holding the remaining-th largest key. Thread t
// owns kBins / NT consecutive bins, the highest for t = 0, so one exclusive block scan of the
// per-thread sums gives the keys above each thread's bins. misc[0] = bin, misc[1] = rank still
// needed inside it, misc[2] = the bin's count; misc + 8: NT/32 words of scan scratch.
template <int NT>
__device__ __forceinline__ void pick_bin(const uint32_t* hist, uint32_t remaining,
                                         uint32_t* misc) {
  constexpr int B = kBins / NT;
  static_assert(B >= 1 && B * NT == kBins, "bins per thread");
  const int hi = kBins - 1 - (int)threadIdx.x * B;     // this thread's highest bin
  uint32_t c[B], sum = 0u;
#pragma unroll
  for (int j = 0; j < B; ++j) {
    c[j] = hist[hslot((uint32_t)(hi - j))];
    sum += c[j];
  }
  uint32_t total;
  uint32_t above = block_excl_scan<NT>(sum, misc + 8, total);
  if (above < remaining && remaining <= above + sum) {
#pragma unroll
    for (int j = 0; j < B; ++j) {
      if (above + c[j] >= remaining) {
        misc[0] = (uint32_t)(hi - j);
        misc[1] = remaining - above;
        misc[2] = c[j];
        break;
      }
      above += c[j];
    }
  }
}

}  // namespace topk_detail

namespace topk_detail {

// Every thread: append each key v of keys[0, n) with (v & mask) == prefix to cand, in any
// order, through the shared counter *ctr (zero on entry). Per batch of sixteen keys a thread
// counts its matches, its warp scans the counts and one lane reserves the warp's slots with
// one atomic, so the matches of a bin do not queue on the counter one by one.
template <int NT>
__device__ __forceinline__ void gather_prefix(const uint32_t* keys, int n, uint32_t mask,
                                              uint32_t prefix, uint32_t* cand, uint32_t* ctr) {
  constexpr int kB4 = 4;
  const int tid = threadIdx.x, lane = tid & 31;
  const int n4 = (n + 3) >> 2;
  const uint4* k4 = reinterpret_cast<const uint4*>(keys);
  for (int base = 0; base < n4; base += NT * kB4) {      // block-uniform
    uint32_t w[4 * kB4], hit = 0u;                        // hit: bit e for a matching w[e]
#pragma unroll
    for (int u = 0; u < kB4; ++u) {
      const int j = base + u * NT + tid;
      const uint4 v = j < n4 ? k4[j] : make_uint4(0u, 0u, 0u, 0u);
      w[4 * u] = v.x;
      w[4 * u + 1] = v.y;
      w[4 * u + 2] = v.z;
      w[4 * u + 3] = v.w;
    }
#pragma unroll
    for (int e = 0; e < 4 * kB4; ++e) {
      const int i = 4 * (base + (e >> 2) * NT + tid) + (e & 3);
      hit |= (uint32_t)(i < n && (w[e] & mask) == prefix) << e;
    }
    const uint32_t c = __popc(hit);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t at = 0u;
    if (lane == 31 && incl != 0u) at = atomicAdd(ctr, incl);
    at = __shfl_sync(0xffffffffu, at, 31) + incl - c;
#pragma unroll
    for (int e = 0; e < 4 * kB4; ++e)
      if ((hit >> e) & 1u) cand[at++] = w[e];
  }
}

// The k-th largest of keys[0, n) (0 < k <= n) by radix passes, every key known to share the
// bits `mask` with `prefix` and the highest bit of the remaining search being `top`. Returns
// (block-uniform) T and take_eq as cta_threshold does; after max_passes digits without an
// answer, the lower edge of the bin holding it instead (a lower bound of the k-th largest,
// with take_eq = all). gather: after the first pass the bin's
// keys may be gathered into cand (keys must then not be cand) and ranked directly when they
// are at most one per thread; otherwise every pass runs over keys.
template <int NT>
__device__ __forceinline__ void radix_kth(const uint32_t* keys, int n, int k, int top, uint32_t mask,
                          uint32_t prefix, bool gather, uint32_t* hist, uint32_t* misc,
                          uint32_t* cand, int cand_cap, uint32_t& T, uint32_t& take_eq,
                          int max_passes = 64) {
  const int tid = threadIdx.x;
  uint32_t remaining = (uint32_t)k;
  int ncand = -1;                            // -1: histogram keys, else cand[0, ncand)
  for (int pass = 1;; ++pass) {
    const int lo = top >= kDigitBits - 1 ? top - (kDigitBits - 1) : 0;
    const uint32_t dmask = (2u << (top - lo)) - 1u;      // digit bits [lo, top]
    if ((reinterpret_cast<uintptr_t>(hist) & 15u) == 0u)
      for (int i = tid; i < kHistWords / 4; i += NT)
        reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    else
      for (int i = tid; i < kHistWords; i += NT) hist[i] = 0u;
    if (tid == 0) misc[4] = 0u;              // the gather's counter
    __syncthreads();
    const uint32_t* src = ncand < 0 ? keys : cand;
    const int m = ncand < 0 ? n : ncand;
    cta_for_keys4<NT>(src, m, [&](int, uint32_t v) {
      if ((v & mask) == prefix) atomicAdd(&hist[hslot((v >> lo) & dmask)], 1u);
    });
    __syncthreads();
    pick_bin<NT>(hist, remaining, misc);
    __syncthreads();
    const uint32_t bin = misc[0];
    remaining = misc[1];
    const uint32_t bin_count = misc[2];
    // misc[0..2] are next written by the following pass's pick_bin, two barriers later
    prefix |= bin << lo;
    mask |= dmask << lo;
    if (remaining == bin_count || lo == 0) { // the whole bin is kept, or the key is complete
      T = prefix;
      take_eq = remaining == bin_count ? 0xffffffffu : remaining;
      return;
    }
    if (pass == max_passes) {                // bound only: the bin's lower edge
      T = prefix;
      take_eq = 0xffffffffu;
      return;
    }
    top = lo - 1;
    if (gather && ncand < 0 && (int)bin_count <= (cand_cap & ~3)) {
      gather_prefix<NT>(keys, n, mask, prefix, cand, &misc[4]);   // the bin's keys
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

// The search window (highest bit, mask, prefix) of keys known to lie in [lo_key, hi_key].
__device__ __forceinline__ int window_of(uint32_t lo_key, uint32_t hi_key, uint32_t& mask,
                                         uint32_t& prefix) {
  const int top = 31 - __clz(lo_key ^ hi_key);
  mask = top == 31 ? 0u : ~((2u << top) - 1u);
  prefix = lo_key & mask;
  return top;
}

// Thread t's segment of the 16-byte groups of keys[0, n): groups [g0, g0 + len), len =
// ceil(ceil(n/4) / NT) but for the last threads, visited from the rotated start r = t mod len
// so that the eight threads of a quarter warp read different banks. f(j, v, lim) per group in
// visit order: j its index in the segment, v its keys, lim = n - 4 (g0 + j) (keys e < lim are
// real). Batches of four groups are loaded before f runs on any of them.
template <int NT, typename F>
__device__ __forceinline__ void for_segment4(const uint32_t* keys, int n, int& g0, int& len,
                                             int& r, F&& f) {
  const int n4 = (n + 3) >> 2;
  const int q = (n4 + NT - 1) / NT;
  g0 = min(n4, (int)threadIdx.x * q);
  len = min(n4, g0 + q) - g0;
  r = len > 0 ? (int)threadIdx.x % len : 0;
  const uint4* k4 = reinterpret_cast<const uint4*>(keys) + g0;
  constexpr int kU = 4;
  int j = r, c = 0;
  for (; c + kU <= len; c += kU) {
    uint4 v[kU];
    int jj[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      jj[u] = j;
      v[u] = k4[j];
      j = j + 1 == len ? 0 : j + 1;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) f(jj[u], v[u], n - 4 * (g0 + jj[u]));
  }
  for (; c < len; ++c) {
    f(j, k4[j], n - 4 * (g0 + j));
    j = j + 1 == len ? 0 : j + 1;
  }
}

// Keys of a group v that are >= L, as bits 0-3 (lim: keys e < lim are real).
__device__ __forceinline__ uint32_t ge_bits(const uint4& v, uint32_t L, int lim) {
  return (uint32_t)(v.x >= L) | (uint32_t)(v.y >= L && lim > 1) << 1 |
         (uint32_t)(v.z >= L && lim > 2) << 2 | (uint32_t)(v.w >= L && lim > 3) << 3;
}

constexpr int kSample = 512;            // prefilter sample size
constexpr int kPrefilterMinPages = 4096;

}  // namespace topk_detail

// Threshold of the top k keys (0 < k < n). On return (block-uniform) the kept keys are those
// > T and the first take_eq keys == T in page order. hist: kHistWords words; misc: 8 +
// NT/32 words; cand: cand_cap words of 16-byte aligned scratch for the gathered keys; list
// (if given) receives the prefilter's ordered candidates, or n = -1 when the search ran over
// every key. NT divides kBins.

//
// Histogram passes cost what the shared-memory atomics cost (~1.6 keys per clock per SM), so
// a long group keeping few pages (n >= 4096, k <= n/16) is first filtered. From a strided
// sample of 512 keys the same radix search takes a lower bound L of the ks-th largest sample
// key (the lower edge of its bin after two digits), ks lying about four standard deviations
// of the sample rank above the rank the k-th largest key is expected to have there, so that
// at least k keys are >= L but not many more. One compare pass over each thread's contiguous
// segment of groups counts the keys >= L; if they are at least k and fit in cand (with their
// pages, half each), one block scan of the counts places them, a second visit of only the
// groups that hold some gathers them in page order, and they are searched alone (every key
// > T or == T is among them, since T >= L). Otherwise the search runs over every key, so the
// sample decides the speed, never the result.
// PREFILTER = false compiles the filter out: merely present, it measured ~4 us slower on
// 2048-page groups in the attention kernel, where it never runs.
template <int NT, bool PREFILTER = true>
__device__ void cta_threshold(const CtaKeys& K, int k, uint32_t* hist, uint32_t* misc,
                              uint32_t* cand, int cand_cap, uint32_t& T, uint32_t& take_eq,
                              CtaCand* list = nullptr) {
  using namespace topk_detail;
  const int tid = threadIdx.x;
  const uint32_t* keys = K.keys;
  const int n = K.n;
  if (list != nullptr) list->n = -1;
  if (K.diff == 0u) {                        // every key equal: the first k pages
    T = K.common;
    take_eq = (uint32_t)k;
    return;
  }
  const uint32_t key_or = K.common | K.diff;  // >= every key
  uint32_t mask, prefix;
  const int top = window_of(K.common, key_or, mask, prefix);
  if (PREFILTER && n >= kPrefilterMinPages && 16 * k <= n && cand_cap >= kSample) {
    const float mu = (float)k * kSample / (float)n;
    const int ks = (int)ceilf(mu + 4.f * sqrtf(mu * (1.f - (float)k / (float)n)) + 4.f);
    if (ks < kSample) {
      const int st = (n / kSample) | 1;      // j * st < 2n: one subtraction wraps it
      for (int j = tid; j < kSample; j += NT) {
        int x = j * st;
        if (x >= n) x -= n;
        cand[j] = keys[x];
      }
      __syncthreads();
      uint32_t L, te;
      radix_kth<NT>(cand, kSample, ks, top, mask, prefix, false, hist, misc, cand, 0, L, te, 2);
      // count the keys >= L of this thread's segment, noting which of its (first 64) groups
      // hold any, so that the gather visits only those
      int g0, len, r;
      uint32_t mine = 0u, total = 0u;
      uint64_t held = 0ull;
      for_segment4<NT>(keys, n, g0, len, r, [&](int j, const uint4& v, int lim) {
        const uint32_t m = __popc(ge_bits(v, L, lim));
        mine += m;
        if (m != 0u && j < 64) held |= 1ull << j;
      });
      const uint32_t at = block_excl_scan<NT>(mine, misc + 8, total);
      const int half = (cand_cap / 2) & ~3;
      if (total >= (uint32_t)k && total <= (uint32_t)half) {
        uint32_t* ck = cand;
        int32_t* cp = reinterpret_cast<int32_t*>(cand + half);
        const uint4* k4 = reinterpret_cast<const uint4*>(keys);
        uint32_t w = at;
        auto put = [&](int j) {              // group g0 + j's keys >= L, in page order
          const uint4 v = k4[g0 + j];
          const uint32_t b = ge_bits(v, L, n - 4 * (g0 + j));
          const int i = 4 * (g0 + j);
          if (b & 1u) { ck[w] = v.x; cp[w] = i; ++w; }
          if (b & 2u) { ck[w] = v.y; cp[w] = i + 1; ++w; }
          if (b & 4u) { ck[w] = v.z; cp[w] = i + 2; ++w; }
          if (b & 8u) { ck[w] = v.w; cp[w] = i + 3; ++w; }
        };
        for (uint64_t h = held; h != 0ull; h &= h - 1ull) put(__ffsll((long long)h) - 1);
        for (int j = 64; j < len; ++j) put(j);
        __syncthreads();
        if (list != nullptr) {
          list->keys = ck;
          list->pages = cp;
          list->n = (int)total;
        }
        if (L == key_or) {                   // every candidate equals L: the first k pages
          T = L;
          take_eq = (uint32_t)k;
          return;
        }
        uint32_t cmask, cprefix;
        const int ctop = window_of(L, key_or, cmask, cprefix);
        radix_kth<NT>(ck, (int)total, k, ctop, cmask, cprefix, false, hist, misc, ck, 0, T,
                      take_eq);
        return;
      }
      __syncthreads();                       // misc + 8 is reused below
    }
  }
  radix_kth<NT>(keys, n, k, top, mask, prefix, true, hist, misc, cand, cand_cap, T, take_eq);
}

// Ordered compaction: calls emit(page, pos) for every kept page whose position pos in the
// ascending kept list lies in [w0, w1) (a CTA that needs one run of the list asks for that
// window; 0 and k give the whole list). Warp w walks the pages [w * seg, (w + 1) * seg) 32 at
// a time (seg a multiple of 32), so ballots order the pages inside each step; a warp whose
// positions miss the window does nothing after the count, a batch of rounds whose kept pages
// all precede the window only advances the counts, and a warp stops once past the window. The
// ballots of a batch of rounds are taken before any emit branches. wtot: NT/32 doublewords.
template <int NT, typename F>
__device__ void cta_compact(const CtaKeys& K, uint32_t T, uint32_t take_eq, uint64_t* wtot,
                            int w0, int w1, F&& emit) {
  using topk_detail::kB;
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t* keys = K.keys;
  const int seg = ((K.n + NW - 1) / NW + 31) & ~31;
  const int s0 = min(K.n, warp * seg), s1 = min(K.n, s0 + seg);
  uint32_t gt = 0u, eq = 0u;
  for (int base = s0; base < s1; base += 32 * kB) {
    uint32_t v[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = base + u * 32 + lane;
      v[u] = i < s1 ? keys[i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const bool in = base + u * 32 + lane < s1;
      gt += in && v[u] > T;
      eq += in && v[u] == T;
    }
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) wtot[warp] = ((uint64_t)gt << 32) | eq;
  __syncthreads();
  const uint64_t wv = lane < NW ? wtot[lane] : 0ull;
  uint32_t gt_before = __reduce_add_sync(0xffffffffu, lane < warp ? (uint32_t)(wv >> 32) : 0u);
  uint32_t eq_before = __reduce_add_sync(0xffffffffu, lane < warp ? (uint32_t)wv : 0u);
  const uint32_t first = gt_before + min(eq_before, take_eq);
  const uint32_t last = gt_before + gt + min(eq_before + eq, take_eq);   // exclusive
  if (last <= (uint32_t)w0 || first >= (uint32_t)w1) return;           // warp-uniform
  const uint32_t below = (1u << lane) - 1u;
  for (int base = s0; base < s1; base += 32 * kB) {
    uint32_t v[kB], bg[kB], be[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = base + u * 32 + lane;
      v[u] = i < s1 ? keys[i] : 0u;
    }
    uint32_t batch_gt = 0u, batch_eq = 0u;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const bool in = base + u * 32 + lane < s1;
      bg[u] = __ballot_sync(0xffffffffu, in && v[u] > T);
      be[u] = __ballot_sync(0xffffffffu, in && v[u] == T);
      batch_gt += __popc(bg[u]);
      batch_eq += __popc(be[u]);
    }
    // a batch whose kept pages all come before the window only advances the counts
    if (gt_before + batch_gt + min(eq_before + batch_eq, take_eq) <= (uint32_t)w0) {
      gt_before += batch_gt;
      eq_before += batch_eq;
      continue;
    }
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = base + u * 32 + lane;
      const uint32_t g_me = gt_before + __popc(bg[u] & below);
      const uint32_t e_me = eq_before + __popc(be[u] & below);
      int pos = -1;
      if ((bg[u] >> lane) & 1u) pos = (int)(g_me + min(e_me, take_eq));
      else if (((be[u] >> lane) & 1u) && e_me < take_eq) pos = (int)(g_me + e_me);
      if (pos >= w0 && pos < w1) emit(i, pos);
      gt_before += __popc(bg[u]);
      eq_before += __popc(be[u]);
    }
    if (gt_before + min(eq_before, take_eq) >= (uint32_t)w1) break;    // past the window
  }
}

// Ordered compaction of a window: calls emit(page, pos) for every kept page whose position
// pos in the ascending kept list lies in [w0, w1), like cta_compact, for windows much shorter
// than the list (one attention CTA's run), at a cost that does not depend on where the window
// lies. Thread t counts the kept pages of its segment of 16-byte groups (for_segment4: rotated
// starts, no bank conflicts); one block scan of the (> T, == T) counts gives each segment its
// first position; the thread whose segment holds position w0 publishes where that segment
// starts and the counts before it, and warp 0 walks the pages from there, four rows of 32 per
// step (their loads and ballots before any emit), until it passes w1. wtot: NT/32
// doublewords; misc2: 4 words. Ends with the emits done by warp 0 only: the caller
// synchronises before reading what emit wrote.
template <int NT, typename F>
__device__ void cta_compact_window(const CtaKeys& K, uint32_t T, uint32_t take_eq,
                                   uint64_t* wtot, uint32_t* misc2, int w0, int w1, F&& emit) {
  constexpr int NW = NT / 32, kR = 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (w0 >= w1) return;                                         // block-uniform
  const uint32_t* keys = K.keys;
  const int n = K.n;
  uint32_t gt = 0u, eq = 0u;
  int g0, len, r;
  topk_detail::for_segment4<NT>(keys, n, g0, len, r, [&](int, const uint4& v, int lim) {
    gt += (v.x > T) + (v.y > T && lim > 1) + (v.z > T && lim > 2) + (v.w > T && lim > 3);
    eq += (v.x == T) + (v.y == T && lim > 1) + (v.z == T && lim > 2) + (v.w == T && lim > 3);
  });
  // exclusive scan of the packed counts over the block
  const uint64_t mine = ((uint64_t)gt << 32) | eq;
  uint64_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wtot[warp] = incl;
  if (tid == 0) misc2[0] = 0xffffffffu;                          // no segment holds w0 yet
  __syncthreads();
  const uint64_t wv = lane < NW ? wtot[lane] : 0ull;
  const uint64_t before = incl - mine;
  const uint32_t gt_before =
      (uint32_t)(before >> 32) +
      __reduce_add_sync(0xffffffffu, lane < warp ? (uint32_t)(wv >> 32) : 0u);
  const uint32_t eq_before =
      (uint32_t)before + __reduce_add_sync(0xffffffffu, lane < warp ? (uint32_t)wv : 0u);
  const uint32_t first = gt_before + min(eq_before, take_eq);
  const uint32_t last = gt_before + gt + min(eq_before + eq, take_eq);   // exclusive
  if (len > 0 && first <= (uint32_t)w0 && (uint32_t)w0 < last) {        // exactly one thread
    misc2[0] = (uint32_t)(4 * g0);
    misc2[1] = gt_before;
    misc2[2] = eq_before;
  }
  __syncthreads();
  if (warp != 0 || misc2[0] == 0xffffffffu) return;            // the window is past the list
  uint32_t g_run = misc2[1], e_run = misc2[2];
  const uint32_t below = (1u << lane) - 1u;
  for (int base = (int)misc2[0]; base < n; base += 32 * kR) {
    uint32_t bg[kR], be[kR];
    uint32_t v[kR];
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      const int i = base + 32 * u + lane;
      v[u] = i < n ? keys[i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      const bool in = base + 32 * u + lane < n;
      bg[u] = __ballot_sync(0xffffffffu, in && v[u] > T);
      be[u] = __ballot_sync(0xffffffffu, in && v[u] == T);
    }
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      const uint32_t g_me = g_run + __popc(bg[u] & below);
      const uint32_t e_me = e_run + __popc(be[u] & below);
      int pos = -1;
      if ((bg[u] >> lane) & 1u) pos = (int)(g_me + min(e_me, take_eq));
      else if (((be[u] >> lane) & 1u) && e_me < take_eq) pos = (int)(g_me + e_me);
      if (pos >= w0 && pos < w1) emit(base + 32 * u + lane, pos);
      g_run += __popc(bg[u]);
      e_run += __popc(be[u]);
    }
    if (g_run + min(e_run, take_eq) >= (uint32_t)w1) break;       // past the window
  }
}

// Ordered compaction from the prefilter's candidates (cta_threshold's list: every kept key
// with its page, in page order): emit(page, pos) for every kept page whose position lies in
// [w0, w1). Thread t takes a contiguous run of the list, counts its (> T, == T) keys, one
// block scan gives the run's first position, and the threads whose runs meet the window emit
// theirs. wtot: NT/32 doublewords. Ends with emits from any thread: the caller synchronises
// before reading what emit wrote.
template <int NT, typename F>
__device__ void cta_compact_list(const CtaCand& C, uint32_t T, uint32_t take_eq,
                                 uint64_t* wtot, int w0, int w1, F&& emit) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = C.n;
  const int q = (m + NT - 1) / NT;
  const int a0 = min(m, tid * q), a1 = min(m, a0 + q);
  uint32_t gt = 0u, eq = 0u;
  for (int i = a0; i < a1; ++i) {
    const uint32_t v = C.keys[i];
    gt += v > T;
    eq += v == T;
  }
  const uint64_t mine = ((uint64_t)gt << 32) | eq;
  uint64_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  const uint64_t wv = lane < NW ? wtot[lane] : 0ull;
  const uint64_t before = incl - mine;
  uint32_t g = (uint32_t)(before >> 32) +
               __reduce_add_sync(0xffffffffu, lane < warp ? (uint32_t)(wv >> 32) : 0u);
  uint32_t e = (uint32_t)before + __reduce_add_sync(0xffffffffu, lane < warp ? (uint32_t)wv : 0u);
  const uint32_t first = g + min(e, take_eq);
  const uint32_t last = g + gt + min(e + eq, take_eq);          // exclusive
  if (last <= (uint32_t)w0 || first >= (uint32_t)w1) return;
  for (int i = a0; i < a1; ++i) {
    const uint32_t v = C.keys[i];
    int pos = -1;
    if (v > T) {
      pos = (int)(g + min(e, take_eq));
      ++g;
    } else if (v == T) {
      if (e < take_eq) pos = (int)(g + e);
      ++e;
    }
    if (pos >= w0 && pos < w1) emit(C.pages[i], pos);
  }
}

}  // namespace skv
