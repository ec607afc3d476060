// Entmax decoding over selected pages: the next-step row "entmax sparse attention +
// Gaussian-aware threshold selector", after "EntmaxKV: Support-Aware Decoding for Entmax
// Attention" (abstract). alpha-entmax gives exact zeros, so attention over the selected
// pages equals full attention as soon as the selection holds the support; a selector that
// estimates the entmax threshold from page statistics adapts the kept budget to the scores.
//
// Readings (the page is an abstract): alpha = 1.5, so with z_t = scale * q.k_t / 2 the
// weights are p_t = max(z_t - tau, 0)^2 with sum_t p_t = 1; sparse entmax normalises over
// the selected tokens; the selector models the group's z as Gaussian with moments taken from
// each page's [min, max] box (centre logit, uniform-in-box variance) and keeps the pages whose
// upper bound exceeds the estimated threshold for some head, plus each head's top page.
//
// Kernels:
//   entmax_moments_kernel  per (page, KV head) row of statistics, for each query head of the
//                          group: upper bound zb, centre logit c and within-box variance v of
//                          z. Eight lanes own a row and hold the same columns of its min and
//                          max halves, so (max - min)^2 is formed element-wise.
//   entmax_select_kernel   one block of 1024 threads per (sequence, KV head): one pass
//                          loading every head's moments of a batch of pages at once into
//                          token-weighted double sums, one block reduction, a warp per head
//                          solving tau_hat on the closed-form Gaussian tail (32 points per
//                          round, then Newton), then the kept pages in ascending order by one
//                          ballot-and-scan pass per 1024 pages.
//   entmax_logits_kernel   split over the selected list; each warp takes a page, each lane a
//                          token (or half of one), and computes the G heads' logits from the
//                          page's keys: K is read once per group.
//   entmax_out_kernel      one block per (sequence, query head): the largest z, the
//                          candidates within 1 of it (tau >= max z - 1), tau bracketed by
//                          bisection and then solved exactly from the support's sums, and the
//                          output sum over the support, reading V rows of support tokens only.
#include "kv_internal.cuh"

namespace skv {
namespace {

constexpr int kMomWarps = 4;                 // moments: 4 warps x 4 rows = 16 pages per block
constexpr int kESelThreads = 512;
constexpr int kLogitWarps = 4;
constexpr int kOutThreads = 512;
constexpr int kCandCap = 16384;              // candidate logits held in shared memory

// ------------------------------------------------------------------------------ moments

template <typename T, int D, int G>
__global__ void __launch_bounds__(kMomWarps * 32)
entmax_moments_kernel(kv_cache_desc d, const T* __restrict__ q, const T* __restrict__ stats,
                      float half_scale, float* __restrict__ zb, float* __restrict__ cz,
                      float* __restrict__ vz, int stride, DevCtx ctx) {
  constexpr int EPC = 16 / ElemTraits<T>::bytes;   // elements per 16-byte chunk
  constexpr int CH = D / EPC;                      // chunks per half row
  constexpr int NU = CH / 8;                       // chunks per lane per half row
  __shared__ float s_q[G][D], s_pos[G][D], s_neg[G][D];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.z, g = blockIdx.y, tid = threadIdx.x;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G;
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, d.page_size);
  const int p_block = blockIdx.x * kMomWarps * 4;
  if (p_block >= n_pages) return;
  const int warp = tid >> 5, lane = tid & 31, j = lane & 7;
  const int p = p_block + warp * 4 + (lane >> 3);
  uint4 rmn[NU], rmx[NU];
  bool ok = false;
  if (p < n_pages) {
    const int P = d.page_table[(long)b * d.page_table_stride + p];
    if (P >= 0 && P < d.num_phys_pages) {
      ok = true;
      const uint4* row = reinterpret_cast<const uint4*>(stats + ((long)P * Hkv + g) * 2 * D);
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        rmn[u] = __ldg(row + j + 8 * u);
        rmx[u] = __ldg(row + CH + j + 8 * u);
      }
    } else if (j == 0) {
      flag(ctx, KV_DEVERR_BAD_PAGE);
    }
  }
  for (int i = tid; i < G * D; i += kMomWarps * 32) {
    const int h = i / D, t = i - h * D;
    const float x = load_elem<T>(q, ((long)b * Hq + g * G + h) * D + t);
    s_q[h][t] = x;
    s_pos[h][t] = fmaxf(x, 0.f);
    s_neg[h][t] = fminf(x, 0.f);
  }
  __syncthreads();
  float bnd[G], cen[G], var[G];
#pragma unroll
  for (int h = 0; h < G; ++h) bnd[h] = cen[h] = var[h] = 0.f;
  if (ok) {
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      float lo[EPC], hi[EPC];
      chunk_to_f32<T>(rmn[u], lo);
      chunk_to_f32<T>(rmx[u], hi);
      const int d0 = (j + 8 * u) * EPC;
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const float w = hi[e] - lo[e], s = lo[e] + hi[e];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float qd = s_q[h][d0 + e];
          bnd[h] = fmaf(s_pos[h][d0 + e], hi[e], fmaf(s_neg[h][d0 + e], lo[e], bnd[h]));
          cen[h] = fmaf(qd, s, cen[h]);
          var[h] = fmaf(qd * qd, w * w, var[h]);
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      bnd[h] += __shfl_xor_sync(0xffffffffu, bnd[h], o);
      cen[h] += __shfl_xor_sync(0xffffffffu, cen[h], o);
      var[h] += __shfl_xor_sync(0xffffffffu, var[h], o);
    }
  }
  if (j == 0 && ok) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const long i = ((long)b * Hq + g * G + h) * stride + p;
      zb[i] = half_scale * bnd[h];
      cz[i] = half_scale * 0.5f * cen[h];
      vz[i] = half_scale * half_scale * var[h] / 12.f;
    }
  }
}

// ------------------------------------------------------------------------------ selector
//
// Everything here is float: FP64 is scarce on this part (a double erfc costs microseconds),
// and the threshold is an estimate, so float accuracy (a relative 1e-6 or so) is ample.

// E[max(Z - tau, 0)^2] for Z ~ N(mu, sigma^2) and its derivative in tau,
// -2 E[max(Z - tau, 0)] = -2 sigma (u Phi(u) + phi(u)), u = (mu - tau) / sigma.
__device__ __forceinline__ void gaussian_tail(float mu, float sigma, float tau, float& f2,
                                              float& f1) {
  if (!(sigma > 0.f)) {
    const float x = fmaxf(mu - tau, 0.f);
    f2 = x * x;
    f1 = x;
    return;
  }
  const float u = (mu - tau) / sigma;
  const float Phi = 0.5f * erfcf(-u * 0.70710678f);      // 1/sqrt(2)
  const float phi = expf(-0.5f * u * u) * 0.39894228f;    // 1/sqrt(2 pi)
  f2 = sigma * sigma * ((u * u + 1.f) * Phi + u * phi);
  f1 = sigma * (u * Phi + phi);
}

// tau_hat with count * E[max(Z - tau_hat, 0)^2] = 1: f(t) = count * E[...] - 1 is convex and
// decreasing in t. Called by a whole warp with the same arguments: each round the 32 lanes
// evaluate f at 32 interior points of the bracket and keep the sub-interval where f changes
// sign (four rounds shrink it about a million-fold), then Newton steps from its f >= 0 end
// converge to float precision. Every lane returns the same value.
__device__ float gaussian_threshold_warp(float mu, float var, float count) {
  const int lane = threadIdx.x & 31;
  const float sigma = sqrtf(fmaxf(var, 0.f));
  float lo = mu - 1.f - 40.f * sigma, hi = mu + 40.f * sigma + 1.f;
  float f2, f1;
  gaussian_tail(mu, sigma, lo, f2, f1);
  if (count * f2 < 1.f) return lo;
  for (int round = 0; round < 4; ++round) {
    const float t = lo + (hi - lo) * (float)(lane + 1) / 33.f;
    gaussian_tail(mu, sigma, t, f2, f1);
    const uint32_t pos = __ballot_sync(0xffffffffu, count * f2 >= 1.f);   // a prefix of lanes
    const int j = __popc(pos) - 1;                   // last point with f >= 0 (-1: none)
    const float tj = __shfl_sync(0xffffffffu, t, j < 0 ? 0 : j);
    const float tn = __shfl_sync(0xffffffffu, t, j + 1 > 31 ? 31 : j + 1);
    const float nlo = j < 0 ? lo : tj;
    const float nhi = j >= 31 ? hi : tn;
    if (!(nlo < nhi)) break;
    lo = nlo;
    hi = nhi;
  }
  float t = lo;
  for (int i = 0; i < 6; ++i) {
    gaussian_tail(mu, sigma, t, f2, f1);
    const float step = (count * f2 - 1.f) / (2.f * count * f1);
    if (!(step > 0.f) || !(f1 > 0.f)) break;
    const float tn = t + step;
    if (!(tn > t) || !(tn < hi)) break;
    t = tn;
  }
  return t;
}

// One block of 512 threads per (sequence, KV head). Thread t takes pages t, t + 512, ...;
// one pass loads every head's (c, v, zb) of a batch of its pages at once and accumulates, per
// head, the token-weighted sums of (c - c0), (c - c0)^2 and v in float, c0 being the head's
// first-page centre (so the variance of c is sum (c - c0)^2 / N - (sum (c - c0) / N)^2 with
// little cancellation: the centres spread over a few standard deviations), and the first
// maximum of zb; one block reduction; a warp per head solves tau_hat; then the kept pages,
// ascending, by one ballot-and-scan pass per 512 pages. G: the group's query heads (1 to 8).
// (FP64 is scarce on this part: double sums here cost more than the rest of the kernel.)
template <int G>
__global__ void __launch_bounds__(kESelThreads)
entmax_select_kernel(const int32_t* __restrict__ seq_lens, int PS, int Hq, int Hkv,
                     int table_stride, const float* __restrict__ zb,
                     const float* __restrict__ cz, const float* __restrict__ vz, int stride,
                     int k_max, int32_t* __restrict__ sel_idx, int32_t* __restrict__ sel_cnt,
                     float* __restrict__ tau_hat, DevCtx ctx) {
  constexpr int NW = kESelThreads / 32;
  constexpr int U = G <= 4 ? 2 : 1;              // pages per thread per batch
  static_assert(G >= 1 && G <= 8 && G <= NW, "group size");
  __shared__ float s_sum[3][G][NW];
  __shared__ float s_bv[G][NW];
  __shared__ int s_bi[G][NW];
  __shared__ float s_tau[G];
  __shared__ int s_arg[G];
  __shared__ uint32_t s_wsum[NW];
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  const int warp = tid >> 5;
  int len = seq_lens[b];
  if (len < 0 || len > table_stride * PS) {
    if (tid == 0) flag(ctx, KV_DEVERR_BAD_LEN);
    len = len < 0 ? 0 : table_stride * PS;
  }
  const int n = ceil_div(len, PS);
  const long grp = (long)b * Hkv + g;
  const long row0 = ((long)b * Hq + g * G) * stride;     // head h of the group: row0 + h*stride
  if (n == 0) {
    if (tid == 0) sel_cnt[grp] = 0;
    if (tid < G && tau_hat != nullptr)
      tau_hat[(long)b * Hq + g * G + tid] = __int_as_float(0x7fc00000);
    return;
  }
  // one pass: every head's sums and first maximum
  float s1[G], s2[G], sv[G], c0[G];
  float best[G];
  int besti[G];
#pragma unroll
  for (int h = 0; h < G; ++h) c0[h] = __ldg(cz + row0 + (long)h * stride);   // page 0
#pragma unroll
  for (int h = 0; h < G; ++h) {
    s1[h] = s2[h] = sv[h] = 0.f;
    best[h] = -INFINITY;
    besti[h] = 0x7fffffff;
  }
  for (int base = 0; base < n; base += kESelThreads * U) {
    float cv[G][U], vv[G][U], zv[G][U];
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int p = base + u * kESelThreads + tid;
        const bool in = p < n;
        const long i = row0 + (long)h * stride + p;
        cv[h][u] = in ? cz[i] : 0.f;
        vv[h][u] = in ? vz[i] : 0.f;
        zv[h][u] = in ? zb[i] : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int p = base + u * kESelThreads + tid;
      if (p < n) {
        const float wt = (float)min(PS, len - p * PS);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float dc = cv[h][u] - c0[h];
          s1[h] = fmaf(wt, dc, s1[h]);
          s2[h] = fmaf(wt * dc, dc, s2[h]);
          sv[h] = fmaf(wt, vv[h][u], sv[h]);
          if (zv[h][u] > best[h]) { best[h] = zv[h][u]; besti[h] = p; }   // pages increase
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s1[h] += __shfl_xor_sync(0xffffffffu, s1[h], o);
        s2[h] += __shfl_xor_sync(0xffffffffu, s2[h], o);
        sv[h] += __shfl_xor_sync(0xffffffffu, sv[h], o);
        const float ov = __shfl_xor_sync(0xffffffffu, best[h], o);
        const int oi = __shfl_xor_sync(0xffffffffu, besti[h], o);
        if (ov > best[h] || (ov == best[h] && oi < besti[h])) { best[h] = ov; besti[h] = oi; }
      }
      if (lane == 0) {
        s_sum[0][h][warp] = s1[h];
        s_sum[1][h][warp] = s2[h];
        s_sum[2][h][warp] = sv[h];
        s_bv[h][warp] = best[h];
        s_bi[h][warp] = besti[h];
      }
    }
  }
  __syncthreads();
  if (warp < G) {                                // warp h: head h's moments and tau_hat
    const int h = warp;
    const bool lv = lane < NW;
    float a1 = lv ? s_sum[0][h][lane] : 0.f, a2 = lv ? s_sum[1][h][lane] : 0.f;
    float av = lv ? s_sum[2][h][lane] : 0.f;
    float bv = lv ? s_bv[h][lane] : -INFINITY;
    int bi = lv ? s_bi[h][lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a1 += __shfl_xor_sync(0xffffffffu, a1, o);
      a2 += __shfl_xor_sync(0xffffffffu, a2, o);
      av += __shfl_xor_sync(0xffffffffu, av, o);
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    const float N = (float)len;
    const float m1 = a1 / N;                     // mean of c - c0
    const float var = fmaxf(a2 / N - m1 * m1, 0.f) + av / N;
    const float t = gaussian_threshold_warp(__ldg(cz + row0 + (long)h * stride) + m1, var, N);
    if (lane == 0) {
      s_tau[h] = t;
      s_arg[h] = bi;
      if (tau_hat != nullptr) tau_hat[(long)b * Hq + g * G + h] = t;
    }
  }
  __syncthreads();
  // kept pages, ascending: one ballot-and-scan pass per 1024 pages
  uint32_t carry = 0;
  int32_t* out = sel_idx + grp * k_max;
  for (int base = 0; base < n; base += kESelThreads) {
    const int p = base + tid;
    bool keep = false;
    if (p < n) {
      float zvv[G];
#pragma unroll
      for (int h = 0; h < G; ++h)                // the group's heads' loads together
        zvv[h] = zb[row0 + (long)h * stride + p];
#pragma unroll
      for (int h = 0; h < G; ++h) keep |= zvv[h] > s_tau[h] || p == s_arg[h];
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_wsum[warp] = __popc(bal);
    __syncthreads();
    const uint32_t wv = lane < NW ? s_wsum[lane] : 0u;
    const uint32_t before = carry + __reduce_add_sync(0xffffffffu, lane < warp ? wv : 0u) +
                            __popc(bal & ((1u << lane) - 1u));
    const uint32_t all = __reduce_add_sync(0xffffffffu, wv);
    if (keep && (int)before < k_max) out[before] = p;
    carry += all;
    __syncthreads();
  }
  if (tid == 0) {
    if ((int)carry > k_max) flag(ctx, KV_DEVERR_KEEP);
    sel_cnt[grp] = min((int)carry, k_max);
  }
}

// ------------------------------------------------------------------------------ logits

constexpr int kLogitRun = 1024;              // run entries resolved per pass
constexpr int kMaxEntSplits = 1024;          // splits of the logits pass (their maxima kept)

template <typename T, int D, int G>
__global__ void __launch_bounds__(kLogitWarps * 32)
entmax_logits_kernel(kv_cache_desc d, const T* __restrict__ q, float scale,
                     const int32_t* __restrict__ sel_idx, const int32_t* __restrict__ sel_cnt,
                     int sel_stride, float* __restrict__ logits, int cap_slots,
                     float* __restrict__ split_max, DevCtx ctx) {
  constexpr int EPC = 16 / ElemTraits<T>::bytes;
  constexpr int MAXC = D / EPC;                // chunks per lane at most (one lane per token)
  __shared__ float s_q[G][D];
  __shared__ float s_wmax[kLogitWarps][G];
  __shared__ int s_P[kLogitRun];
  __shared__ int s_valid[kLogitRun];
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, S = gridDim.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, PS = d.page_size;
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, PS);
  const long grp = (long)b * Hkv + g;
  int cnt = n_pages;
  if (sel_idx != nullptr) {
    cnt = sel_cnt[grp];
    if (cnt < 0 || cnt > sel_stride) {
      if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      cnt = cnt < 0 ? 0 : sel_stride;
    }
  }
  const int c = ceil_div(cnt, S);
  const int pos0 = min(cnt, s * c), pos1 = min(cnt, pos0 + c);
  float* smax = split_max + ((long)b * Hq + g * G) * S + s;     // head h: smax[h * S]
  if (pos0 >= pos1) {
    if (tid < G) smax[(long)tid * S] = -INFINITY;
    return;
  }
  for (int i = tid; i < G * D; i += kLogitWarps * 32) {
    const int h = i / D, t = i - h * D;
    s_q[h][t] = load_elem<T>(q, ((long)b * Hq + g * G + h) * D + t);
  }
  float lmax[G];                               // this lane's largest logit per head
#pragma unroll
  for (int h = 0; h < G; ++h) lmax[h] = -INFINITY;
  const int TPW = PS < 32 ? PS : 32;           // tokens per item
  const int SPT = 32 / TPW;                    // lanes per token (1 or 2)
  const int DS = D / SPT;                      // columns per lane
  const int NCH = DS / EPC;                    // 16-byte chunks per lane
  const int IPP = PS / TPW;                    // items per page
  const int sl = lane / TPW, tl = lane % TPW;
  const T* __restrict__ kp = static_cast<const T*>(d.k_pool);
  for (int r0 = pos0; r0 < pos1; r0 += kLogitRun) {
    const int rn = min(kLogitRun, pos1 - r0);
    __syncthreads();                           // the previous pass is done with s_P
    for (int i = tid; i < rn; i += kLogitWarps * 32) {
      const int pos = r0 + i;
      const int page = sel_idx != nullptr ? sel_idx[grp * sel_stride + pos] : pos;
      int P = -1, valid = 0;
      if (page < 0 || page >= n_pages) {
        flag(ctx, KV_DEVERR_BAD_SEL);
      } else {
        P = d.page_table[(long)b * d.page_table_stride + page];
        if (P < 0 || P >= d.num_phys_pages) {
          flag(ctx, KV_DEVERR_BAD_PAGE);
          P = -1;
        } else {
          valid = min(PS, len - page * PS);
        }
      }
      s_P[i] = P;
      s_valid[i] = valid;
    }
    __syncthreads();
    // items (page, token group) of this warp: two buffers alternate, so the next item's keys
    // are in flight while the current one is computed (no register copy waits for them)
    uint4 bufA[MAXC], bufB[MAXC];
    auto load = [&](int item, uint4* buf) {
      const int i = item / IPP, t = (item - i * IPP) * TPW + tl;
      const int P = s_P[i];
      const bool live = P >= 0 && t < s_valid[i];
      const uint4* row = reinterpret_cast<const uint4*>(
          kp + (((long)(live ? P : 0) * Hkv + g) * PS + (live ? t : 0)) * D + sl * DS);
#pragma unroll
      for (int u = 0; u < MAXC; ++u)
        buf[u] = (live && u < NCH) ? __ldg(row + u) : make_uint4(0, 0, 0, 0);
    };
    const int items = rn * IPP;
    auto compute = [&](int item, const uint4* cur) {
      const int i = item / IPP, t = (item - i * IPP) * TPW + tl;
      const bool live = s_P[i] >= 0 && t < s_valid[i];
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
      for (int u = 0; u < MAXC; ++u) {
        if (u >= NCH) break;
        float f[EPC];
        chunk_to_f32<T>(cur[u], f);
        const int dd = sl * DS + u * EPC;
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h] = fmaf(s_q[h][dd + e], f[e], acc[h]);
        }
      }
      if (SPT == 2) {
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 16);
      }
      if (sl == 0) {
        const long slot = (long)(r0 + i) * PS + t;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float x = live ? scale * acc[h] : -INFINITY;
          logits[((long)b * Hq + g * G + h) * cap_slots + slot] = x;
          lmax[h] = fmaxf(lmax[h], x);
        }
      }
    };
    int item = warp;
    if (item < items) load(item, bufA);
    for (; item < items; item += 2 * kLogitWarps) {
      const int i2 = item + kLogitWarps;
      if (i2 < items) load(i2, bufB);
      compute(item, bufA);
      if (i2 >= items) break;
      if (i2 + kLogitWarps < items) load(i2 + kLogitWarps, bufA);
      compute(i2, bufB);
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax[h] = fmaxf(lmax[h], __shfl_xor_sync(0xffffffffu, lmax[h], o));
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) s_wmax[warp][h] = lmax[h];
  }
  __syncthreads();
  if (tid < G) {
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kLogitWarps; ++w) m = fmaxf(m, s_wmax[w][tid]);
    smax[(long)tid * S] = m;
  }
}

// ------------------------------------------------------------------------------ output

// Warp-level: from the splits' maxima z_s = sm[s]/2 (one token each), a floor below tau. The
// entmax threshold of a subset of the tokens is at most the full one (adding tokens only
// raises it); Newton on f(t) = sum max(z_s - t, 0)^2 - 1 (convex, decreasing) from
// t = max z - 1, where f >= 0, stays at f >= 0 and rises to the subset's threshold. Every
// lane returns the same value (the gather and the output kernels call this on the same data).
// sm: the S maxima in shared memory (the Newton passes re-read them).
__device__ float entmax_floor(const float* sm, int S, int lane) {
  float zmax = -INFINITY;
  for (int s = lane; s < S; s += 32) zmax = fmaxf(zmax, 0.5f * sm[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, off));
  if (zmax == -INFINITY) return zmax;
  float t = zmax - 1.f;
  for (int it = 0; it < 32; ++it) {
    float s1 = 0.f, s2 = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float e = 0.5f * sm[s] - t;
      if (e > 0.f) { s1 += e; s2 = fmaf(e, e, s2); }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
      s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    }
    const float step = (s2 - 1.f) / (2.f * s1);
    if (!(step > 1e-6f * (fabsf(t) + 1.f))) break;
    t += 0.999f * step;                        // stay on the f >= 0 side despite rounding
  }
  return t - 1e-5f * (fabsf(t) + 1.f);         // margin: the floor must not pass tau
}

// Group (b, g)'s attended page count.
__device__ __forceinline__ int entmax_count(const kv_cache_desc& d, int b, long grp, int n_pages,
                                            const int32_t* sel_idx, const int32_t* sel_cnt,
                                            int sel_stride) {
  int cnt = n_pages;
  if (sel_idx != nullptr) {
    cnt = sel_cnt[grp];
    cnt = cnt < 0 ? 0 : (cnt > sel_stride ? sel_stride : cnt);   // flagged by the logits pass
  }
  return cnt;
}

// One CTA per (split, query head): the split's candidates (z > floor), in slot order, to
// cand_z / cand_slot at the split's first slot; their count to split_cnt.
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads)
entmax_gather_kernel(kv_cache_desc d, int G, const int32_t* __restrict__ sel_idx,
                     const int32_t* __restrict__ sel_cnt, int sel_stride,
                     const float* __restrict__ logits, int cap_slots,
                     const float* __restrict__ split_max, float* __restrict__ cand_z,
                     int* __restrict__ cand_slot, int* __restrict__ split_cnt, DevCtx ctx) {
  constexpr int NW = kGatherThreads / 32;
  constexpr int U = 4;
  __shared__ float s_floor;
  __shared__ int s_cnt[U][NW];
  __shared__ float s_sm[kMaxEntSplits];
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, S = gridDim.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, g = h / G, PS = d.page_size;
  const int len = checked_len(ctx, d, b);
  const long grp = (long)b * Hkv + g;
  const int cnt = entmax_count(d, b, grp, ceil_div(len, PS), sel_idx, sel_cnt, sel_stride);
  const int cps = ceil_div(cnt, S);
  const int a0 = min(cnt, s * cps) * PS, a1 = min(cnt, (s + 1) * cps) * PS;
  const long row = (long)b * Hq + h;
  for (int i = tid; i < S; i += kGatherThreads) s_sm[i] = __ldcg(split_max + row * S + i);
  __syncthreads();
  if (warp == 0) {
    const float f = entmax_floor(s_sm, S, lane);
    if (lane == 0) s_floor = f;
  }
  __syncthreads();
  const float zfloor = s_floor;
  int carry = 0;
  if (a0 < a1 && 0.5f * s_sm[s] > zfloor) {
    const float* x = logits + row * cap_slots;
    float* cz = cand_z + row * cap_slots;
    int* cs = cand_slot + row * cap_slots;
    for (int base = a0; base < a1; base += kGatherThreads * U) {
      float z[U];
      uint32_t bal[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * kGatherThreads + tid;
        z[u] = i < a1 ? 0.5f * __ldcg(x + i) : -INFINITY;
        bal[u] = __ballot_sync(0xffffffffu, z[u] > zfloor);
      }
      __syncthreads();
      if (lane == 0) {
#pragma unroll
        for (int u = 0; u < U; ++u) s_cnt[u][warp] = __popc(bal[u]);
      }
      __syncthreads();
      int pre = carry;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        int in_chunk_before = 0, chunk_total = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          in_chunk_before += w < warp ? s_cnt[u][w] : 0;
          chunk_total += s_cnt[u][w];
        }
        if (z[u] > zfloor) {
          const int at = a0 + pre + in_chunk_before + __popc(bal[u] & ((1u << lane) - 1u));
          cz[at] = z[u];
          cs[at] = base + u * kGatherThreads + tid;
        }
        pre += chunk_total;
      }
      carry = pre;
    }
  }
  if (tid == 0) split_cnt[row * S + s] = carry;
}

template <typename T, int D>
__global__ void __launch_bounds__(kOutThreads)
entmax_out_kernel(kv_cache_desc d, int G, const int32_t* __restrict__ sel_idx,
                  const int32_t* __restrict__ sel_cnt, int sel_stride,
                  const float* __restrict__ logits, int cap_slots,
                  const float* __restrict__ split_max, const float* __restrict__ cand_z,
                  const int* __restrict__ cand_slot, const int* __restrict__ split_cnt, int S,
                  float* __restrict__ out, float* __restrict__ tau_out, DevCtx ctx) {
  constexpr int NW = kOutThreads / 32;
  constexpr int EPL = D / 32;
  extern __shared__ __align__(16) unsigned char dyn[];
  float* s_z = reinterpret_cast<float*>(dyn);                     // [kCandCap]
  int* s_slot = reinterpret_cast<int*>(s_z + kCandCap);           // [kCandCap]
  __shared__ double s_redd[5 * NW];
  __shared__ int s_redi[NW];
  __shared__ float s_acc[NW][D];
  __shared__ int s_off[kMaxEntSplits + 1];
  __shared__ float s_sm[kMaxEntSplits];
  __shared__ float s_floor;
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, g = h / G, PS = d.page_size;
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, PS);
  const long grp = (long)b * Hkv + g;
  const int cnt = entmax_count(d, b, grp, n_pages, sel_idx, sel_cnt, sel_stride);
  const int n_slots = cnt * PS;
  const long row = (long)b * Hq + h;
  const float* x = logits + row * cap_slots;
  float* o = out + row * D;
  if (n_slots == 0) {
    for (int i = tid; i < D; i += kOutThreads) o[i] = 0.f;
    if (tid == 0 && tau_out != nullptr) tau_out[row] = __int_as_float(0x7fc00000);
    return;
  }
  const int cps = ceil_div(cnt, S);
  for (int i = tid; i < S; i += kOutThreads) s_sm[i] = __ldcg(split_max + row * S + i);
  __syncthreads();
  // warp 0: the floor (as the gather kernel found it) and the splits' candidate offsets
  if (warp == 0) {
    const float f = entmax_floor(s_sm, S, lane);
    int run = 0;
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int sp = s0 + lane;
      const int c_ = sp < S ? split_cnt[row * S + sp] : 0;
      int incl = c_;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (sp < S) s_off[sp] = run + incl - c_;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) { s_off[S] = run; s_floor = f; }
  }
  __syncthreads();
  const float zfloor = s_floor;
  const int total = s_off[S];
  const bool in_smem = total <= kCandCap;
  if (in_smem) {
    // the candidates in order: candidate i belongs to the last split with s_off <= i (binary
    // search), so every load is independent of the others
    for (int i = tid; i < total; i += kOutThreads) {
      int lo = 0, hi = S;                      // s_off[lo] <= i < s_off[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= i) lo = mid;
        else hi = mid;
      }
      const long src = row * cap_slots + (long)min(cnt, lo * cps) * PS + (i - s_off[lo]);
      s_z[i] = __ldcg(cand_z + src);
      s_slot[i] = __ldcg(cand_slot + src);
    }
  }
  __syncthreads();
  const int nc = in_smem ? total : n_slots;
  auto cand_z_at = [&](int i) -> float { return in_smem ? s_z[i] : 0.5f * __ldcg(x + i); };
  // tau: from zfloor (f >= 0), each pass sums over S = {z > tau}; the exact root of
  // sum_S (z - t)^2 = 1, t* = (Z1 - sqrt(Z1^2 - k (Z2 - 1))) / k, is tau when every z of S
  // lies above it (S is then the support); otherwise a Newton step (f = A2 - 1, f' = -2 A1),
  // which from the f >= 0 side stays there and rises to the root, and another pass. Small
  // candidate sets are solved by warp 0 alone (no block barrier per pass).
  double tau = (double)zfloor;
  const bool one_warp = in_smem && nc <= 1024;
  if (!one_warp || warp == 0) {
    for (int it = 0; it < 64; ++it) {
      double a1 = 0.0, a2 = 0.0, z1 = 0.0, z2 = 0.0, zmin = INFINITY;
      int k = 0;
      const int step_i = one_warp ? 32 : kOutThreads;
      for (int i = one_warp ? lane : tid; i < nc; i += step_i) {
        const double z = (double)cand_z_at(i);
        if (z > tau) {
          const double e = z - tau;
          a1 += e; a2 += e * e; z1 += z; z2 += z * z; ++k;
          zmin = z < zmin ? z : zmin;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        a1 += __shfl_xor_sync(0xffffffffu, a1, off);
        a2 += __shfl_xor_sync(0xffffffffu, a2, off);
        z1 += __shfl_xor_sync(0xffffffffu, z1, off);
        z2 += __shfl_xor_sync(0xffffffffu, z2, off);
        zmin = fmin(zmin, __shfl_xor_sync(0xffffffffu, zmin, off));
        k += __shfl_xor_sync(0xffffffffu, k, off);
      }
      double A1 = a1, A2 = a2, Z1 = z1, Z2 = z2, ZMIN = zmin;
      int K = k;
      if (!one_warp) {
        __syncthreads();
        if (lane == 0) {
          s_redd[warp] = a1; s_redd[NW + warp] = a2; s_redd[2 * NW + warp] = z1;
          s_redd[3 * NW + warp] = z2; s_redd[4 * NW + warp] = zmin; s_redi[warp] = k;
        }
        __syncthreads();
        A1 = A2 = Z1 = Z2 = 0.0;
        ZMIN = INFINITY;
        K = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          A1 += s_redd[w]; A2 += s_redd[NW + w]; Z1 += s_redd[2 * NW + w];
          Z2 += s_redd[3 * NW + w]; ZMIN = fmin(ZMIN, s_redd[4 * NW + w]); K += s_redi[w];
        }
      }
      if (K == 0) break;
      const double disc = Z1 * Z1 - (double)K * (Z2 - 1.0);
      const double t_star = (Z1 - sqrt(disc > 0.0 ? disc : 0.0)) / (double)K;
      if (disc >= 0.0 && ZMIN > t_star) {
        tau = t_star;
        break;
      }
      const double t_new = tau + (A2 - 1.0) / (2.0 * A1);
      if (!(t_new > tau)) break;
      tau = t_new;
    }
  }
  if (one_warp) {
    if (tid == 0) s_redd[0] = tau;
    __syncthreads();
    tau = s_redd[0];
  }
  // out = sum over the support of (z - tau)^2 v. The support (in candidate order) is
  // compacted into the candidate buffer's front as (weight, slot) when the candidates are in
  // shared memory; warps then take four support tokens at a time, loads in flight together.
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  const T* __restrict__ vp = static_cast<const T*>(d.v_pool);
  auto v_row = [&](int slot) -> const T* {
    const int pos = slot / PS, t = slot - pos * PS;
    const int page = sel_idx != nullptr ? sel_idx[grp * sel_stride + pos] : pos;
    if (page < 0 || page >= n_pages) return nullptr;
    const int P = d.page_table[(long)b * d.page_table_stride + page];
    if (P < 0 || P >= d.num_phys_pages) return nullptr;
    return vp + (((long)P * Hkv + g) * PS + t) * D + lane * EPL;
  };
  if (in_smem) {
    // in place, round by round: every thread reads its candidate before any write of the
    // round, and a support token lands at an index no larger than its own
    int ns = 0;
    for (int base = 0; base < nc; base += kOutThreads) {
      const int i = base + tid;
      float zi = 0.f;
      int si = 0;
      bool keep = false;
      if (i < nc) {
        zi = s_z[i];
        si = s_slot[i];
        keep = (double)zi > tau;
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      __syncthreads();                         // the round's reads are done; s_redi is free
      if (lane == 0) s_redi[warp] = __popc(bal);
      __syncthreads();
      int before = ns, round_total = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        before += w < warp ? s_redi[w] : 0;
        round_total += s_redi[w];
      }
      if (keep) {
        const int at = before + __popc(bal & ((1u << lane) - 1u));
        const double dz = (double)zi - tau;
        s_z[at] = (float)(dz * dz);
        s_slot[at] = si;
      }
      ns += round_total;
    }
    __syncthreads();
    for (int i0 = warp * 4; i0 < ns; i0 += NW * 4) {
      const T* rows[4];
      float pw[4], vals[4][EPL];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        rows[u] = i0 + u < ns ? v_row(s_slot[i0 + u]) : nullptr;
        pw[u] = i0 + u < ns ? s_z[i0 + u] : 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) vals[u][e] = rows[u] ? load_elem<T>(rows[u], e) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pw[u], vals[u][e], acc[e]);
      }
    }
  } else {
    for (int i = warp; i < nc; i += NW) {
      const double z = (double)cand_z_at(i);
      if (!(z > tau)) continue;
      const T* row = v_row(i);
      if (row == nullptr) continue;
      const float pw = (float)((z - tau) * (z - tau));
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pw, load_elem<T>(row, e), acc[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) s_acc[warp][lane * EPL + e] = acc[e];
  __syncthreads();
  for (int i = tid; i < D; i += kOutThreads) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += s_acc[w][i];
    o[i] = s;
  }
  if (tid == 0 && tau_out != nullptr) tau_out[(long)b * Hq + h] = (float)tau;
}

// ------------------------------------------------------------------------------ launchers

template <typename T, int D, int G>
cudaError_t moments_t(const kv_cache_desc& d, const void* q, const void* stats, float scale,
                      float* zb, float* cz, float* vz, int stride, DevCtx ctx, cudaStream_t s) {
  dim3 grid(ceil_div(d.page_table_stride, kMomWarps * 4), d.num_kv_heads, d.batch);
  return launch_pdl(entmax_moments_kernel<T, D, G>, grid, dim3(kMomWarps * 32), 0, s, d,
                    static_cast<const T*>(q), static_cast<const T*>(stats), 0.5f * scale, zb,
                    cz, vz, stride, ctx);
}

template <typename T, int D, int G>
cudaError_t logits_t(const kv_cache_desc& d, const void* q, float scale, const int32_t* sel,
                     const int32_t* cnt, int sel_stride, int S, float* logits, int cap_slots,
                     float* split_max, DevCtx ctx, cudaStream_t s) {
  dim3 grid(S, d.num_kv_heads, d.batch);
  return launch_pdl(entmax_logits_kernel<T, D, G>, grid, dim3(kLogitWarps * 32), 0, s, d,
                    static_cast<const T*>(q), scale, sel, cnt, sel_stride, logits, cap_slots,
                    split_max, ctx);
}

template <typename T, int D>
cudaError_t out_t(const kv_cache_desc& d, int G, const int32_t* sel, const int32_t* cnt,
                  int sel_stride, const float* logits, int cap_slots, const float* split_max,
                  float* cand_z, int* cand_slot, int* split_cnt, int S, float* out, float* tau,
                  DevCtx ctx, cudaStream_t s) {
  cudaError_t e0 = launch_pdl(entmax_gather_kernel, dim3(S, d.num_kv_heads * G, d.batch),
                              dim3(kGatherThreads), 0, s, d, G, sel, cnt, sel_stride, logits,
                              cap_slots, split_max, cand_z, cand_slot, split_cnt, ctx);
  if (e0 != cudaSuccess) return e0;
  const size_t smem = (size_t)kCandCap * (sizeof(float) + sizeof(int));
  auto kern = entmax_out_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(d.num_kv_heads * G, d.batch);
  return launch_pdl(kern, grid, dim3(kOutThreads), smem, s, d, G, sel, cnt, sel_stride, logits,
                    cap_slots, split_max, cand_z, cand_slot, split_cnt, S, out, tau, ctx);
}

#define SKV_G_SWITCH(CALL_T_D)                                                   \
  switch (G) {                                                                   \
    case 1: return CALL_T_D(1);                                                  \
    case 2: return CALL_T_D(2);                                                  \
    case 4: return CALL_T_D(4);                                                  \
    case 8: return CALL_T_D(8);                                                  \
    default: return cudaErrorInvalidValue;                                      \
  }

template <typename T, int D>
cudaError_t moments_d(const kv_cache_desc& d, int G, const void* q, const void* stats,
                      float scale, float* zb, float* cz, float* vz, int stride, DevCtx ctx,
                      cudaStream_t s) {
#define SKV_CALL(GG) moments_t<T, D, GG>(d, q, stats, scale, zb, cz, vz, stride, ctx, s)
  SKV_G_SWITCH(SKV_CALL)
#undef SKV_CALL
}

template <typename T, int D>
cudaError_t logits_d(const kv_cache_desc& d, int G, const void* q, float scale,
                     const int32_t* sel, const int32_t* cnt, int sel_stride, int S,
                     float* logits, int cap_slots, float* split_max, DevCtx ctx,
                     cudaStream_t s) {
#define SKV_CALL(GG) \
  logits_t<T, D, GG>(d, q, scale, sel, cnt, sel_stride, S, logits, cap_slots, split_max, ctx, s)
  SKV_G_SWITCH(SKV_CALL)
#undef SKV_CALL
}

}  // namespace

cudaError_t launch_entmax_moments(const kv_cache_desc& d, int G, const void* q,
                                  const void* stats, float scale, float* zb, float* cz,
                                  float* vz, int stride, DevCtx ctx, cudaStream_t s) {
  const bool bf = d.dtype == KV_BF16;
  if (d.head_dim == 128)
    return bf ? moments_d<bf16_t, 128>(d, G, q, stats, scale, zb, cz, vz, stride, ctx, s)
              : moments_d<float, 128>(d, G, q, stats, scale, zb, cz, vz, stride, ctx, s);
  return bf ? moments_d<bf16_t, 64>(d, G, q, stats, scale, zb, cz, vz, stride, ctx, s)
            : moments_d<float, 64>(d, G, q, stats, scale, zb, cz, vz, stride, ctx, s);
}

cudaError_t launch_entmax_select(const int32_t* seq_lens, int page_size, int batch, int Hq,
                                 int Hkv, int table_stride, const float* zb, const float* cz,
                                 const float* vz, int stride, int k_max, int32_t* sel_idx,
                                 int32_t* sel_cnt, float* tau_hat, DevCtx ctx, cudaStream_t s) {
  dim3 grid(Hkv, batch);
#define SKV_ESEL(GG)                                                                          \
  return launch_pdl(entmax_select_kernel<GG>, grid, dim3(kESelThreads), 0, s, seq_lens,        \
                    page_size, Hq, Hkv, table_stride, zb, cz, vz, stride, k_max, sel_idx,       \
                    sel_cnt, tau_hat, ctx)
  switch (Hq / Hkv) {
    case 1: SKV_ESEL(1);
    case 2: SKV_ESEL(2);
    case 3: SKV_ESEL(3);
    case 4: SKV_ESEL(4);
    case 5: SKV_ESEL(5);
    case 6: SKV_ESEL(6);
    case 7: SKV_ESEL(7);
    case 8: SKV_ESEL(8);
    default: return cudaErrorInvalidValue;
  }
#undef SKV_ESEL
}

int entmax_max_splits() { return kMaxEntSplits; }

cudaError_t launch_entmax_attn(const kv_cache_desc& d, int G, const void* q, float scale,
                               const int32_t* sel, const int32_t* cnt, int sel_stride, int S,
                               const EntmaxScratch& w, int cap_slots, float* out, float* tau,
                               DevCtx ctx, cudaStream_t s) {
  if (S < 1 || S > kMaxEntSplits) return cudaErrorInvalidValue;
  const bool bf = d.dtype == KV_BF16;
  cudaError_t e;
  if (d.head_dim == 128)
    e = bf ? logits_d<bf16_t, 128>(d, G, q, scale, sel, cnt, sel_stride, S, w.logits, cap_slots,
                                   w.split_max, ctx, s)
           : logits_d<float, 128>(d, G, q, scale, sel, cnt, sel_stride, S, w.logits, cap_slots,
                                  w.split_max, ctx, s);
  else
    e = bf ? logits_d<bf16_t, 64>(d, G, q, scale, sel, cnt, sel_stride, S, w.logits, cap_slots,
                                  w.split_max, ctx, s)
           : logits_d<float, 64>(d, G, q, scale, sel, cnt, sel_stride, S, w.logits, cap_slots,
                                 w.split_max, ctx, s);
  if (e != cudaSuccess) return e;
#define SKV_OUT(TT, DD)                                                                    \
  return out_t<TT, DD>(d, G, sel, cnt, sel_stride, w.logits, cap_slots, w.split_max,       \
                       w.cand_z, w.cand_slot, w.split_cnt, S, out, tau, ctx, s)
  if (d.head_dim == 128) {
    if (bf) SKV_OUT(bf16_t, 128);
    SKV_OUT(float, 128);
  }
  if (bf) SKV_OUT(bf16_t, 64);
  SKV_OUT(float, 64);
#undef SKV_OUT
}

}  // namespace skv
