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
//                          max halves (and of the query, in registers), so the box's width and
//                          centre are formed element-wise.
//   entmax_select_kernel   one block of 512 threads per (sequence, KV head): one pass loading
//                          every head's moments of a batch of pages at once into float sums
//                          shifted by the head's first-page centre, one block reduction, a warp
//                          per head solving tau_hat on the closed-form Gaussian tail (Newton on
//                          its logarithm), then the kept pages in ascending order:
//                          each warp ballots its own run, one block scan, then writes it.
//   entmax_logits_*kernel  split over the attended list, K read once per group for its G
//                          heads (bf16: on the tensor cores); z of a chunk kept in shared
//                          memory, and only the tokens above the chunk's own threshold written
//                          out, as candidates.
//   entmax_out_kernel      one block per (sequence, query head): the splits' candidates, tau
//                          solved exactly over them (Newton from a floor, closed-form finish),
//                          and the output sum over the support, reading V rows of support
//                          tokens only.
#include <algorithm>
#include <cooperative_groups.h>
#include <type_traits>

#include "kv_internal.cuh"

namespace skv {
namespace {

namespace cg = cooperative_groups;

constexpr int kMomWarps = 4;                 // moments: 4 warps x rounds x 4 rows per block
constexpr int kSelThreads = 256;             // selector: threads per CTA
constexpr int kSelCluster = 8;               // selector: CTAs per group (one portable cluster)
constexpr int kSelSteps = 32;               // selector: 32-page ballot words per warp per pass
constexpr int kLogitWarps = 4;
constexpr int kOutThreads = 512;
constexpr int kCandCap = 16384;              // candidate logits held in shared memory

// ------------------------------------------------------------------------------ moments

// One statistics row's three sums for every head (this lane's columns): with s = mn + mx and
// w = mx - mn per column, max(q mn, q mx) = (q s + |q| w) / 2, and q^2 w^2 = (q w)^2. Then summed over the row's 8
// lanes (xor 1, 2, 4), so every lane of the row holds the row's totals.
template <typename T, int G, int NU, int EPC>
__device__ __forceinline__ void mom_row(const uint4 (&rmn)[NU], const uint4 (&rmx)[NU],
                                        const float (&qv)[G][NU][EPC], bool ok, float (&bnd)[G],
                                        float (&cen)[G], float (&var)[G]) {
#pragma unroll
  for (int h = 0; h < G; ++h) bnd[h] = cen[h] = var[h] = 0.f;
  if (ok) {
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      float lo[EPC], hi[EPC];
      chunk_to_f32<T>(rmn[u], lo);
      chunk_to_f32<T>(rmx[u], hi);
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const float w = hi[e] - lo[e], sm = lo[e] + hi[e];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float qd = qv[h][u][e], qw = qd * w;
          cen[h] = fmaf(qd, sm, cen[h]);
          bnd[h] = fmaf(fabsf(qd), w, bnd[h]);
          var[h] = fmaf(qw, qw, var[h]);
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
}

// This lane's query columns (j + 8u) * EPC .. + EPC of every head of group (b, g).
template <typename T, int D, int G, int NU, int EPC>
__device__ __forceinline__ void mom_query(const T* q, long row0, int j, float (&qv)[G][NU][EPC]) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4* qr = reinterpret_cast<const uint4*>(q + (row0 + h) * D);
#pragma unroll
    for (int u = 0; u < NU; ++u) chunk_to_f32<T>(__ldg(qr + j + 8 * u), qv[h][u]);
  }
}

// A warp takes rpw rounds of 4 statistics rows (the next round's loads in flight while a round
// is summed), 8 lanes a row; lane j of a row holds columns (j + 8u) * EPC .. + EPC of both
// halves, and the query's same columns for every head in registers (no shared memory, no
// barrier). rpw is chosen so that the grid is about one wave.
// blocks per SM the moments kernel is sized for (the query's columns of all G heads live in
// registers: 64 floats a lane for 4 bf16 heads)
template <typename T, int G>
constexpr int mom_blocks() { return (ElemTraits<T>::bytes == 4 || G >= 8) ? 2 : 4; }

template <typename T, int D, int G>
__global__ void __launch_bounds__(kMomWarps * 32, mom_blocks<T, G>())
entmax_moments_kernel(kv_cache_desc d, const T* __restrict__ q, const T* __restrict__ stats,
                      float half_scale, float* __restrict__ zb, float* __restrict__ cz,
                      float* __restrict__ vz, int stride, int rpw, DevCtx ctx) {
  constexpr int EPC = 16 / ElemTraits<T>::bytes;   // elements per 16-byte chunk
  constexpr int CH = D / EPC;                      // chunks per half row
  constexpr int NU = CH / 8;                       // chunks per lane per half row
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.z, g = blockIdx.y, tid = threadIdx.x;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G;
  const int warp = tid >> 5, lane = tid & 31, j = lane & 7;
  const int p_block = blockIdx.x * kMomWarps * rpw * 4;
  const int p0 = p_block + warp * rpw * 4 + (lane >> 3);
  const int32_t* trow = d.page_table + (long)b * d.page_table_stride;
  // the first round's page-table entry before the length (it lies in the table's row either
  // way and is used only below the length), so the two loads are in flight together
  const int P0 = p0 < d.page_table_stride ? __ldg(trow + p0) : -1;
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, d.page_size);
  if (p_block >= n_pages) return;
  auto load = [&](int r, uint4 (&rmn)[NU], uint4 (&rmx)[NU]) -> bool {
    const int p = p0 + 4 * r;
    if (r >= rpw || p >= n_pages) return false;
    const int P = r == 0 ? P0 : trow[p];
    if (P < 0 || P >= d.num_phys_pages) {
      if (j == 0) flag(ctx, KV_DEVERR_BAD_PAGE);
      return false;
    }
    const uint4* row = reinterpret_cast<const uint4*>(stats + ((long)P * Hkv + g) * 2 * D);
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      rmn[u] = __ldg(row + j + 8 * u);
      rmx[u] = __ldg(row + CH + j + 8 * u);
    }
    return true;
  };
  uint4 amn[NU], amx[NU], bmn[NU], bmx[NU];
  bool aok = load(0, amn, amx);
  float qv[G][NU][EPC];
  mom_query<T, D, G, NU, EPC>(q, (long)b * Hq + g * G, j, qv);
  for (int r = 0; r < rpw && p0 + 4 * r < n_pages; ++r) {
    const bool bok = load(r + 1, bmn, bmx);
    float bnd[G], cen[G], var[G];
    mom_row<T, G, NU, EPC>(amn, amx, qv, aok, bnd, cen, var);
    if (j == 0 && aok) {
      const int p = p0 + 4 * r;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const long i = ((long)b * Hq + g * G + h) * stride + p;
        zb[i] = half_scale * 0.5f * (cen[h] + bnd[h]);
        cz[i] = half_scale * 0.5f * cen[h];
        vz[i] = half_scale * half_scale * var[h] / 12.f;
      }
    }
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      amn[u] = bmn[u];
      amx[u] = bmx[u];
    }
    aok = bok;
  }
}

// ------------------------------------------------------------------------------ selector
//
// Everything here is float: FP64 is scarce on this part (a double erfc costs microseconds),
// and the threshold is an estimate, so float accuracy (a relative 1e-6 or so) is ample.

// psi(u) = E[max(X + u, 0)^2] for X ~ N(0, 1), = (u^2 + 1) Phi(u) + u phi(u), and its
// derivative psi'(u) = 2 (u Phi(u) + phi(u)).
__device__ __forceinline__ void gaussian_psi(float u, float& p, float& dp) {
  const float Phi = 0.5f * erfcf(-u * 0.70710678f);      // 1/sqrt(2)
  const float phi = __expf(-0.5f * u * u) * 0.39894228f;  // 1/sqrt(2 pi)
  p = (u * u + 1.f) * Phi + u * phi;
  dp = 2.f * (u * Phi + phi);
}

// tau_hat with count * E[max(Z - tau_hat, 0)^2] = 1 for Z ~ N(mu, var). With sigma > 0 and
// u = (mu - tau_hat) / sigma this reads psi(u) = c, c = 1 / (count var). psi is positive,
// increasing and log-concave, so Newton on ln psi(u) - ln c converges from any start: a step
// from the right of the root lands on its left, and from there the iterates rise to it. The
// start: u = sqrt(c - 1) when c >= 1 (psi(u) ~ u^2 + 1 above zero), 0 down to c = 0.05, else
// the tail asymptote psi(u) ~ 2 phi(u) / |u|^3. sigma = 0 gives tau_hat = mu - 1/sqrt(count).
__device__ float gaussian_threshold(float mu, float var, float count) {
  const float sigma = sqrtf(fmaxf(var, 0.f));
  if (!(sigma > 0.f)) return mu - rsqrtf(count);
  const float c = 1.f / (count * sigma * sigma), lnc = logf(c);
  float u;
  if (c >= 1.f) {
    u = sqrtf(c - 1.f);
  } else if (c >= 0.05f) {
    u = 0.f;
  } else {
    const float L2 = 2.f * logf(0.79788456f / c);        // 2 ln(2 / (sqrt(2 pi) c))
    u = -sqrtf(fmaxf(L2 - 3.f * logf(L2), 0.25f));
  }
  for (int it = 0; it < 16; ++it) {
    float p, dp;
    gaussian_psi(u, p, dp);
    if (!(p > 0.f) || !(dp > 0.f)) {                     // underflow far left: move right
      u += 1.f;
      continue;
    }
    const float du = __fdividef((lnc - __logf(p)) * p, dp);
    u += du;
    if (!(fabsf(du) > 2e-6f * (1.f + fabsf(u)))) break;
  }
  return mu - sigma * u;
}

// A cluster of kSelCluster CTAs per (sequence, KV head) group, each over its own range of the
// group's pages. Each CTA loads every head's (c, v, zb) of its pages (a batch of pages per
// thread at once) and accumulates, per head, the token-weighted sums of (c - c0), (c - c0)^2
// and v in float, c0 being the head's first-page centre (so the variance of c is
// sum (c - c0)^2 / N - (sum (c - c0) / N)^2 with little cancellation: the centres spread over
// a few standard deviations), and the first maximum of zb. The CTAs' sums are added in rank
// order through distributed shared memory, so every CTA holds the same totals and a warp per
// head solves the same tau_hat in each. Each CTA then counts its kept pages; the counts of the
// lower ranks (again through distributed shared memory) give its offset, and it writes its
// kept pages, ascending, by warp ballots over contiguous runs. G: the group's query heads (1
// to 8). (FP64 is scarce on this part: double sums here cost more than the rest.)
template <int G>
__global__ void __launch_bounds__(kSelThreads)
entmax_select_kernel(const int32_t* __restrict__ seq_lens, int PS, int Hq, int Hkv,
                     int table_stride, const float* __restrict__ zb,
                     const float* __restrict__ cz, const float* __restrict__ vz, int stride,
                     int k_max, int32_t* __restrict__ sel_idx, int32_t* __restrict__ sel_cnt,
                     float* __restrict__ tau_hat, DevCtx ctx) {
  constexpr int NW = kSelThreads / 32;
  constexpr int U = G <= 4 ? 4 : 2;              // pages per thread per batch
  static_assert(G >= 1 && G <= 8 && G <= NW, "group size");
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  __shared__ float s_wsum[3][G][NW];
  __shared__ float s_wbest[G][NW];
  __shared__ int s_wbi[G][NW];
  __shared__ float s_part[3 * G];                // this CTA's sums (read by the cluster)
  __shared__ float s_best[G];
  __shared__ int s_bidx[G];
  __shared__ float s_tau[G];
  __shared__ int s_arg[G];
  __shared__ float s_c0[G];
  __shared__ uint32_t s_bal[NW][kSelSteps];
  __shared__ int s_wcnt[NW];
  __shared__ int s_cnt;                          // this CTA's kept pages (read by the cluster)
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.y, b = blockIdx.z, tid = threadIdx.x, lane = tid & 31;
  const int warp = tid >> 5;
  int len = seq_lens[b];
  if (len < 0 || len > table_stride * PS) {
    if (tid == 0 && rank == 0) flag(ctx, KV_DEVERR_BAD_LEN);
    len = len < 0 ? 0 : table_stride * PS;
  }
  const int n = ceil_div(len, PS);
  const long grp = (long)b * Hkv + g;
  const long row0 = ((long)b * Hq + g * G) * stride;     // head h of the group: row0 + h*stride
  if (n == 0) {                                  // every CTA of the cluster returns here
    if (rank == 0) {
      if (tid == 0) sel_cnt[grp] = 0;
      if (tid < G && tau_hat != nullptr)
        tau_hat[(long)b * Hq + g * G + tid] = __int_as_float(0x7fc00000);
    }
    return;
  }
  const int PC = ceil_div(n, CL);
  const int p_begin = min(n, rank * PC), p_end = min(n, p_begin + PC);
  if (tid < G) s_c0[tid] = __ldg(cz + row0 + (long)tid * stride);   // page 0
  __syncthreads();
  float c0[G];
#pragma unroll
  for (int h = 0; h < G; ++h) c0[h] = s_c0[h];
  // one pass over this CTA's pages: every head's sums and first maximum
  float s1[G], s2[G], sv[G], best[G];
  int besti[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    s1[h] = s2[h] = sv[h] = 0.f;
    best[h] = -INFINITY;
    besti[h] = 0x7fffffff;
  }
  for (int base = p_begin; base < p_end; base += kSelThreads * U) {
    float cv[G][U], vv[G][U], zv[G][U];
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int p = base + u * kSelThreads + tid;
        const bool in = p < p_end;
        const long i = row0 + (long)h * stride + p;
        cv[h][u] = in ? cz[i] : 0.f;
        vv[h][u] = in ? vz[i] : 0.f;
        zv[h][u] = in ? zb[i] : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int p = base + u * kSelThreads + tid;
      if (p < p_end) {
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
      s_wsum[0][h][warp] = s1[h];
      s_wsum[1][h][warp] = s2[h];
      s_wsum[2][h][warp] = sv[h];
      s_wbest[h][warp] = best[h];
      s_wbi[h][warp] = besti[h];
    }
  }
  __syncthreads();
  if (warp < G) {                                // warp h: this CTA's sums for head h
    const int h = warp;
    const bool lv = lane < NW;
    float a1 = lv ? s_wsum[0][h][lane] : 0.f, a2 = lv ? s_wsum[1][h][lane] : 0.f;
    float av = lv ? s_wsum[2][h][lane] : 0.f;
    float bv = lv ? s_wbest[h][lane] : -INFINITY;
    int bi = lv ? s_wbi[h][lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a1 += __shfl_xor_sync(0xffffffffu, a1, o);
      a2 += __shfl_xor_sync(0xffffffffu, a2, o);
      av += __shfl_xor_sync(0xffffffffu, av, o);
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) {
      s_part[3 * h] = a1;
      s_part[3 * h + 1] = a2;
      s_part[3 * h + 2] = av;
      s_best[h] = bv;
      s_bidx[h] = bi;
    }
  }
  cluster.sync();                                // every CTA's sums are final
  if (warp < G) {                                // warp h: the group's totals, rank order
    const int h = warp;
    float a1 = 0.f, a2 = 0.f, av = 0.f, bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int rk = 0; rk < CL; ++rk) {
      const float* part = cluster.map_shared_rank(s_part, rk);
      a1 += part[3 * h];
      a2 += part[3 * h + 1];
      av += part[3 * h + 2];
      const float ob = cluster.map_shared_rank(s_best, rk)[h];
      const int oi = cluster.map_shared_rank(s_bidx, rk)[h];
      if (ob > bv || (ob == bv && oi < bi)) { bv = ob; bi = oi; }
    }
    const float N = (float)len;
    const float m1 = a1 / N;                     // mean of c - c0
    const float var = fmaxf(a2 / N - m1 * m1, 0.f) + av / N;
    const float t = gaussian_threshold(c0[h] + m1, var, N);
    if (lane == 0) {
      s_tau[h] = t;
      s_arg[h] = bi;
      if (tau_hat != nullptr && rank == 0) tau_hat[(long)b * Hq + g * G + h] = t;
    }
  }
  __syncthreads();
  auto kept_page = [&](int p) -> bool {
    bool keep = false;
#pragma unroll
    for (int h = 0; h < G; ++h) keep |= zb[row0 + (long)h * stride + p] > s_tau[h] || p == s_arg[h];
    return keep;
  };
  int mine = 0;
  for (int p = p_begin + tid; p < p_end; p += kSelThreads) mine += kept_page(p) ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) s_wcnt[warp] = mine;
  __syncthreads();
  if (tid == 0) {
    int c = 0;
    for (int w = 0; w < NW; ++w) c += s_wcnt[w];
    s_cnt = c;
  }
  cluster.sync();                                // every CTA's count is final
  int carry = 0, total_all = 0;
  for (int rk = 0; rk < CL; ++rk) {
    const int c = *cluster.map_shared_rank(&s_cnt, rk);
    carry += rk < rank ? c : 0;
    total_all += c;
  }
  // this CTA's kept pages from its offset: warp-contiguous runs, 32 pages a ballot
  int32_t* out = sel_idx + grp * k_max;
  for (int c0p = p_begin; c0p < p_end; c0p += NW * 32 * kSelSteps) {
    const int c1p = min(p_end, c0p + NW * 32 * kSelSteps);
    const int pw = ceil_div(c1p - c0p, NW * 32) * 32;     // pages per warp
    const int w0 = c0p + warp * pw, w1 = min(c1p, w0 + pw);
    const int st_n = pw / 32;
    int wcount = 0;
    for (int st = 0; st < st_n; ++st) {
      const int p = w0 + st * 32 + lane;
      const uint32_t bal = __ballot_sync(0xffffffffu, p < w1 && kept_page(p));
      if (lane == 0) s_bal[warp][st] = bal;
      wcount += __popc(bal);
    }
    __syncthreads();                             // earlier readers of s_wcnt are done
    if (lane == 0) s_wcnt[warp] = wcount;
    __syncthreads();
    int at = carry, total = 0;
    for (int w = 0; w < NW; ++w) {
      at += w < warp ? s_wcnt[w] : 0;
      total += s_wcnt[w];
    }
    for (int st = 0; st < st_n; ++st) {
      const uint32_t bal = s_bal[warp][st];
      if ((bal >> lane) & 1u) {
        const int pos = at + __popc(bal & ((1u << lane) - 1u));
        if (pos < k_max) out[pos] = w0 + st * 32 + lane;
      }
      at += __popc(bal);
    }
    carry += total;
  }
  if (rank == 0 && tid == 0) {
    if (total_all > k_max) flag(ctx, KV_DEVERR_KEEP);
    sel_cnt[grp] = min(total_all, k_max);
  }
  cluster.sync();                                // no CTA leaves while another reads its memory
}

// ------------------------------------------------------------------------------ threshold
//
// The entmax threshold of a set of z values solves f(t) = sum max(z - t, 0)^2 = 1. f is
// convex and decreasing, so Newton from a point where f >= 0 (any t <= max z - 1) rises to the
// root; once every member of {z > t} lies above the closed-form root of that set (and the root
// is not below t, where the non-members lie), the root is the threshold. The closed form is
// taken about a pivot p: with y = z - p over the K members, tau = p + mean(y) - sqrt((1 - Q)
// / K), Q = sum (y - mean)^2 = sum y^2 - K mean^2. That difference keeps its digits only while
// the pivot lies within about a standard deviation of the members' mean, so a root is taken
// only then; otherwise the pass is repeated about the mean. Float throughout: FP64 is scarce
// on this part, and the logits themselves carry float rounding.

struct TauSums {
  float k, y1, y2, e1, e2, zmin;               // count, sums of y, y^2, e = z - t, e^2; min z
};

__device__ __forceinline__ TauSums tau_zero() { return {0.f, 0.f, 0.f, 0.f, 0.f, INFINITY}; }

__device__ __forceinline__ void tau_add(TauSums& s, float z, float t, float pivot) {
  if (z > t) {
    const float y = z - pivot, e = z - t;
    s.k += 1.f;
    s.y1 += y;
    s.y2 = fmaf(y, y, s.y2);
    s.e1 += e;
    s.e2 = fmaf(e, e, s.e2);
    s.zmin = fminf(s.zmin, z);
  }
}

// Butterfly: every lane ends with bitwise the same sums.
__device__ __forceinline__ void tau_warp_reduce(TauSums& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s.k += __shfl_xor_sync(0xffffffffu, s.k, o);
    s.y1 += __shfl_xor_sync(0xffffffffu, s.y1, o);
    s.y2 += __shfl_xor_sync(0xffffffffu, s.y2, o);
    s.e1 += __shfl_xor_sync(0xffffffffu, s.e1, o);
    s.e2 += __shfl_xor_sync(0xffffffffu, s.e2, o);
    s.zmin = fminf(s.zmin, __shfl_xor_sync(0xffffffffu, s.zmin, o));
  }
}

// The closed form over the members {z > t} from their sums about pivot.
struct TauClosed {
  float root, mean_z;
  bool valid;                                  // members at or above root, root >= t
  bool pivot_ok;                               // pivot within a standard deviation of mean_z
};

__device__ __forceinline__ TauClosed tau_closed(const TauSums& s, float pivot, float t) {
  TauClosed c{-INFINITY, pivot, false, true};
  if (s.k == 0.f) return c;
  const float m = s.y1 / s.k;
  const float q = fmaxf(s.y2 - s.y1 * m, 0.f);
  c.mean_z = pivot + m;
  c.pivot_ok = m * m <= q / s.k + 1e-6f;
  const float r = 1.f - q;
  if (r >= 0.f) {
    c.root = c.mean_z - sqrtf(r / s.k);
    c.valid = s.zmin >= c.root && c.root >= t;
  }
  return c;
}

// One step from the sums over {z > t}: true when t is final (the closed form holds about a
// good pivot, or Newton cannot advance any further); else t has taken a Newton step, or the
// pivot has moved to the members' mean for another pass at the same t.
__device__ __forceinline__ bool tau_step(const TauSums& s, float& pivot, float& t) {
  if (s.k == 0.f) return true;
  const TauClosed c = tau_closed(s, pivot, t);
  if (c.valid) {
    if (c.pivot_ok) {
      t = c.root;
      return true;
    }
    pivot = c.mean_z;
    return false;
  }
  const float step = (s.e2 - 1.f) / (2.f * s.e1);
  if (!(step > 0.f)) return true;
  t += step;
  pivot = c.mean_z;
  return false;
}

// The threshold of zat(0 .. n-1) by one warp, from t (f(t) >= 0); all lanes return it.
template <class ZAt>
__device__ float warp_entmax_tau(ZAt zat, int n, float t, float pivot, int lane) {
  for (int it = 0; it < 64; ++it) {
    TauSums s = tau_zero();
    for (int i = lane; i < n; i += 32) tau_add(s, zat(i), t, pivot);
    tau_warp_reduce(s);
    if (tau_step(s, pivot, t)) break;
  }
  return t;
}

// The same by a block of NT threads (two barriers a step; warp 0 takes the step).
template <int NT, class ZAt>
__device__ float block_entmax_tau(ZAt zat, int n, float t, float pivot, TauSums* s_red,
                                  float* s_bc) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int it = 0; it < 64; ++it) {
    TauSums s = tau_zero();
    for (int i = tid; i < n; i += NT) tau_add(s, zat(i), t, pivot);
    tau_warp_reduce(s);
    if (lane == 0) s_red[warp] = s;
    __syncthreads();
    if (warp == 0) {
      TauSums w = lane < NW ? s_red[lane] : tau_zero();
      tau_warp_reduce(w);
      float tn = t, pn = pivot;
      const bool done = tau_step(w, pn, tn);
      if (lane == 0) {
        s_bc[0] = tn;
        s_bc[1] = done ? 1.f : 0.f;
        s_bc[2] = pn;
      }
    }
    __syncthreads();
    t = s_bc[0];
    pivot = s_bc[2];
    if (s_bc[1] != 0.f) break;
  }
  return t;
}

// A block's first pass: warp w takes the point lo + (hi - lo) w / NW of a bracket [lo, hi]
// with f(lo) >= 0 and sums over all n values there (no barrier inside the pass). A point
// whose closed form holds about a good pivot gives tau; otherwise the Newton passes start
// from the highest point with f >= 0, within 1/NW of the bracket from the root.
template <int NT, class ZAt>
__device__ float block_entmax_tau_bracket(ZAt zat, int n, float lo, float hi, float pivot,
                                          TauSums* s_red, float* s_pts, float* s_bc) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float tw = lo + (hi - lo) * (float)warp / (float)NW;
  TauSums s = tau_zero();
  for (int i = lane; i < n; i += 32) tau_add(s, zat(i), tw, pivot);
  tau_warp_reduce(s);
  if (lane == 0) {
    const TauClosed c = tau_closed(s, pivot, tw);
    s_pts[warp] = s.e2 - 1.f;                    // f(tw)
    s_pts[NW + warp] = c.valid && c.pivot_ok ? c.root : -INFINITY;
  }
  __syncthreads();
  float start = lo;
  for (int w = 0; w < NW; ++w) {
    if (s_pts[NW + w] != -INFINITY) return s_pts[NW + w];
    if (s_pts[w] >= 0.f) start = lo + (hi - lo) * (float)w / (float)NW;
  }
  return block_entmax_tau<NT>(zat, n, start, pivot, s_red, s_bc);
}

// The exact threshold of the 32 values v held one per lane (-inf: no value), by the sorting
// form: with the values descending, the support is the longest prefix whose k-th value lies
// above the closed-form root of the first k. A lower bound on the threshold of any set that
// holds these values; .x the threshold, .y the mean of that support (-inf, -inf when every
// value is -inf). Every lane returns the same.
__device__ float2 warp32_tau(float v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {          // bitonic sort, descending across the lanes
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, j);
      v = (((lane & k) == 0) == ((lane & j) == 0)) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  const float v0 = __shfl_sync(0xffffffffu, v, 0);
  if (v0 == -INFINITY) return make_float2(v0, v0);
  const float y = v - v0;
  float s1 = y, s2 = y * y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float a = __shfl_up_sync(0xffffffffu, s1, o), b = __shfl_up_sync(0xffffffffu, s2, o);
    if (lane >= o) {
      s1 += a;
      s2 += b;
    }
  }
  const float k = (float)(lane + 1), mean = s1 / k;
  const float r = 1.f - fmaxf(s2 - s1 * mean, 0.f);
  const float root = v0 + mean - sqrtf(r / k);
  const uint32_t ok = __ballot_sync(0xffffffffu, r >= 0.f && v > root);   // a prefix of lanes
  const int K = 31 - __clz(ok | 1u);
  return make_float2(__shfl_sync(0xffffffffu, root, K), v0 + __shfl_sync(0xffffffffu, mean, K));
}

// A start for the Newton passes from the lanes' largest values: .x the threshold of those
// values less a rounding margin (f >= 0 there), never below max - 1; .y a pivot, the mean of
// their support.
__device__ __forceinline__ float2 tau_start(float lane_max, float zmax, int lane) {
  const float2 w = warp32_tau(lane_max, lane);
  return make_float2(fmaxf(zmax - 1.f, w.x - 1e-6f * (fabsf(w.x) + 1.f)), w.y);
}

// ------------------------------------------------------------------------------ logits
//
// One CTA per (split, KV head, sequence) over its run of the attended pages, in chunks of
// kChunkFloats / G tokens whose z values (all G heads) stay in shared memory. After each
// chunk, a warp per head bounds the chunk's entmax threshold from below by the exact threshold
// of its lanes' largest values: the threshold of any subset of a head's tokens is at most the
// full one (adding tokens only raises it), so a token at or below it has weight zero. The tokens above it (less a rounding margin) are appended in list
// order to the head's candidate list of this split, as (z, row of the token in the V pool);
// the split's floor (its chunks' largest bound, a lower bound on tau) and candidate count
// are written at the end. No logit goes to memory.

constexpr int kMaxEntSplits = 1024;          // splits of the logits pass
constexpr int kChunkFloats = 8192;           // z values of one chunk (all heads): 32 KB

template <int G, int NW>
struct ChunkLists {                          // a warp's heads: warp, warp + NW, ...
  static constexpr int HPW = (G + NW - 1) / NW;
  int count[HPW];
  float floor[HPW];
  __device__ void init() {
#pragma unroll
    for (int j = 0; j < HPW; ++j) {
      count[j] = 0;
      floor[j] = -INFINITY;
    }
  }
};

// The chunk's candidates (tokens above the bound). s_z + h * zs: head h's n values (-inf for
// tokens past the sequence);
// token i of the chunk sits in physical page s_P[i / PS] (PS = 1 << ps_log2), KV head g;
// cz/cs: the split's candidate region of head 0 of the group (head h at + h * cap_slots).
template <int G, int NW>
__device__ void chunk_candidates(const float* s_z, int zs, int n, const int* s_P, int ps_log2,
                                 int Hkv, int g, int warp, int lane, float* cz, uint32_t* cs,
                                 long cap_slots, ChunkLists<G, NW>& L) {
#pragma unroll
  for (int j = 0; j < ChunkLists<G, NW>::HPW; ++j) {
    const int h = warp + j * NW;
    if (h >= G) break;
    const float* z = s_z + h * zs;
    float lm = -INFINITY;
    for (int i = lane; i < n; i += 32) lm = fmaxf(lm, z[i]);
    float m = lm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (m == -INFINITY) continue;
    // the threshold of the lanes' largest values bounds the chunk's own from below (a subset
    // of its tokens), and measured closer to it than the Newton passes are worth here
    const float thr = tau_start(lm, m, lane).x;
    L.floor[j] = fmaxf(L.floor[j], thr);
    float* oz = cz + (long)h * cap_slots;
    uint32_t* os = cs + (long)h * cap_slots;
    int c = L.count[j];
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      const float v = i < n ? z[i] : -INFINITY;
      const bool keep = v > thr;
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const int at = c + __popc(bal & ((1u << lane) - 1u));
        const int pg = i >> ps_log2;
        oz[at] = v;
        os[at] = ((uint32_t)s_P[pg] * (uint32_t)Hkv + (uint32_t)g) * (1u << ps_log2) +
                 (uint32_t)(i - (pg << ps_log2));
      }
      c += __popc(bal);
    }
    L.count[j] = c;
  }
}

// Resolves the chunk's pages (list positions r0 .. r0 + rn) to physical pages and valid
// token counts; flags bad entries (their tokens count as past the sequence).
__device__ __forceinline__ void resolve_chunk(const kv_cache_desc& d, int b, long grp,
                                              const int32_t* sel_idx, int sel_stride, int r0,
                                              int rn, int n_pages, int len, int* s_P,
                                              int* s_valid, DevCtx ctx) {
  for (int i = threadIdx.x; i < rn; i += blockDim.x) {
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
        valid = min(d.page_size, len - page * d.page_size);
      }
    }
    s_P[i] = P;
    s_valid[i] = valid;
  }
}

// The group's attended page count (clamped and flagged when out of range) and this split's
// run [pos0, pos1) of it.
__device__ __forceinline__ int split_run(const int32_t* sel_idx, const int32_t* sel_cnt,
                                         int sel_stride, long grp, int n_pages, int s, int S,
                                         int& pos0, int& pos1, DevCtx ctx) {
  int cnt = n_pages;
  if (sel_idx != nullptr) {
    cnt = sel_cnt[grp];
    if (cnt < 0 || cnt > sel_stride) {
      if (threadIdx.x == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      cnt = cnt < 0 ? 0 : sel_stride;
    }
  }
  const int cps = ceil_div(cnt, S);
  pos0 = min(cnt, s * cps);
  pos1 = min(cnt, pos0 + cps);
  return cnt;
}

template <int G, int NW>
__device__ __forceinline__ void write_split(const ChunkLists<G, NW>& L, int warp, int lane,
                                            float* split_floor, int* split_cnt, long row0,
                                            int S, int s) {
#pragma unroll
  for (int j = 0; j < ChunkLists<G, NW>::HPW; ++j) {
    const int h = warp + j * NW;
    if (h < G && lane == 0) {
      split_floor[(row0 + h) * S + s] = L.floor[j];
      split_cnt[(row0 + h) * S + s] = L.count[j];
    }
  }
}

// CUDA-core form (float caches): a warp takes a page, a lane a token (or half of one).
template <typename T, int D, int G>
__global__ void __launch_bounds__(kLogitWarps * 32)
entmax_logits_kernel(kv_cache_desc d, const T* __restrict__ q, float scale,
                     const int32_t* __restrict__ sel_idx, const int32_t* __restrict__ sel_cnt,
                     int sel_stride, int cap_slots, float* __restrict__ split_floor,
                     float* __restrict__ cand_z, uint32_t* __restrict__ cand_row,
                     int* __restrict__ split_cnt, DevCtx ctx) {
  constexpr int EPC = 16 / ElemTraits<T>::bytes;
  constexpr int MAXC = D / EPC;                // chunks per lane at most (one lane per token)
  constexpr int CT = kChunkFloats / G;         // tokens per chunk
  constexpr int ZS = CT + 4;
  __shared__ float s_q[G][D];
  __shared__ __align__(16) float s_z[G * ZS];
  __shared__ int s_P[CT / 16];
  __shared__ int s_valid[CT / 16];
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, S = gridDim.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, PS = d.page_size;
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, PS);
  const long grp = (long)b * Hkv + g, row0 = (long)b * Hq + g * G;
  int pos0, pos1;
  split_run(sel_idx, sel_cnt, sel_stride, grp, n_pages, s, S, pos0, pos1, ctx);
  ChunkLists<G, kLogitWarps> L;
  L.init();
  if (pos0 >= pos1) {
    write_split(L, warp, lane, split_floor, split_cnt, row0, S, s);
    return;
  }
  for (int i = tid; i < G * D; i += kLogitWarps * 32) {
    const int h = i / D, t = i - h * D;
    s_q[h][t] = load_elem<T>(q, (row0 + h) * D + t);
  }
  const int TPW = PS < 32 ? PS : 32;           // tokens per item
  const int SPT = 32 / TPW;                    // lanes per token (1 or 2)
  const int DS = D / SPT;                      // columns per lane
  const int NCH = DS / EPC;                    // 16-byte chunks per lane
  const int IPP = PS / TPW;                    // items per page
  const int sl = lane / TPW, tl = lane % TPW;
  const int CP = CT / PS;                      // pages per chunk
  const int ps_log2 = __ffs(PS) - 1;
  const T* __restrict__ kp = static_cast<const T*>(d.k_pool);
  float* cz = cand_z + row0 * cap_slots + (long)pos0 * PS;
  uint32_t* cs = cand_row + row0 * cap_slots + (long)pos0 * PS;
  for (int r0 = pos0; r0 < pos1; r0 += CP) {
    const int rn = min(CP, pos1 - r0);
    __syncthreads();                           // the previous chunk is done with s_z, s_P
    resolve_chunk(d, b, grp, sel_idx, sel_stride, r0, rn, n_pages, len, s_P, s_valid, ctx);
    __syncthreads();
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
#pragma unroll
        for (int h = 0; h < G; ++h) s_z[h * ZS + i * PS + t] = live ? 0.5f * scale * acc[h] : -INFINITY;
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
    __syncthreads();
    chunk_candidates(s_z, ZS, rn * PS, s_P, ps_log2, Hkv, g, warp, lane, cz, cs, cap_slots,
                     L);
  }
  write_split(L, warp, lane, split_floor, split_cnt, row0, S, s);
}

// Tensor-core form (bf16 caches). A warp takes 16-token tiles of the chunk's pages: one
// mma.sync m16n8k16 per 16 key columns, the tile's tokens as the m rows and the group's G
// query heads as the n columns (zero-padded to 8). A dot product does not depend on the order
// of the head dimension, so each lane loads whole 16-byte pieces of its two rows straight into
// A fragments and takes the query's words at the same positions for its B fragment: lane
// (r = lane / 4, c = lane % 4) holds words 16u + 4c + e (e < 4) of rows r and r + 8, and
// k-step k uses words e = 2 (k % 2) and e + 1 of piece u = k / 2. Four lanes read 64
// contiguous bytes of a row per load; the next tile's loads are in flight while the current
// one is multiplied. bf16 products are exact in f32, as in the CUDA-core form.
constexpr int kLogitMmaWarps = 4;

template <int D, int G>
__global__ void __launch_bounds__(kLogitMmaWarps * 32, 4)
entmax_logits_mma_kernel(kv_cache_desc d, const bf16_t* __restrict__ q, float scale,
                         const int32_t* __restrict__ sel_idx, const int32_t* __restrict__ sel_cnt,
                         int sel_stride, int cap_slots, float* __restrict__ split_floor,
                         float* __restrict__ cand_z, uint32_t* __restrict__ cand_row,
                         int* __restrict__ split_cnt, DevCtx ctx) {
  static_assert(G >= 1 && G <= 8, "at most 8 query heads per KV head");
  constexpr int U = D / 32;                    // 16-byte pieces per lane per row
  constexpr int ROW4 = D / 8;                  // 16-byte pieces per row
  constexpr int CT = kChunkFloats / G;         // tokens per chunk
  constexpr int ZS = CT + 4;                   // head stride: the 4 lanes of a row hit 4 banks
  __shared__ __align__(16) float s_z[G * ZS];
  __shared__ int s_P[CT / 16];
  __shared__ int s_valid[CT / 16];
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, S = gridDim.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, PS = d.page_size, TPP = PS / 16;
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, PS);
  const long grp = (long)b * Hkv + g, row0 = (long)b * Hq + g * G;
  int pos0, pos1;
  split_run(sel_idx, sel_cnt, sel_stride, grp, n_pages, s, S, pos0, pos1, ctx);
  ChunkLists<G, kLogitMmaWarps> L;
  L.init();
  if (pos0 >= pos1) {
    write_split(L, warp, lane, split_floor, split_cnt, row0, S, s);
    return;
  }
  // B fragment: head r of the group (zero for r >= G), the words this lane's A pieces cover
  uint32_t bq[U][4];
  {
    const uint16_t* qh = reinterpret_cast<const uint16_t*>(q) + (row0 + r) * D;
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int w = 16 * u + 4 * c + e;
        bq[u][e] = r < G ? (uint32_t)qh[2 * w] | ((uint32_t)qh[2 * w + 1] << 16) : 0u;
      }
    }
  }
  const float zscale = 0.5f * scale;
  const uint4* __restrict__ kp = static_cast<const uint4*>(d.k_pool);
  const int CP = CT / PS;                      // pages per chunk
  const int ps_log2 = __ffs(PS) - 1;
  float* cz = cand_z + row0 * cap_slots + (long)pos0 * PS;
  uint32_t* cs = cand_row + row0 * cap_slots + (long)pos0 * PS;
  for (int r0 = pos0; r0 < pos1; r0 += CP) {
    const int rn = min(CP, pos1 - r0);
    __syncthreads();                           // the previous chunk is done with s_z, s_P
    resolve_chunk(d, b, grp, sel_idx, sel_stride, r0, rn, n_pages, len, s_P, s_valid, ctx);
    __syncthreads();
    const int tiles = rn * TPP;
    auto load = [&](int it, uint4 (&a)[2][U]) {
      const int i = it / TPP, t0 = (it - i * TPP) * 16;
      const int P = s_P[i], valid = s_valid[i];
      const bool la = P >= 0 && t0 + r < valid, lb = P >= 0 && t0 + r + 8 < valid;
      const uint4* rowa = kp + (((long)(P >= 0 ? P : 0) * Hkv + g) * PS + t0 + r) * ROW4 + c;
      const uint4* rowb = rowa + 8 * ROW4;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        a[0][u] = la ? __ldg(rowa + 4 * u) : make_uint4(0, 0, 0, 0);
        a[1][u] = lb ? __ldg(rowb + 4 * u) : make_uint4(0, 0, 0, 0);
      }
    };
    auto compute = [&](int it, const uint4 (&a)[2][U]) {
      const int i = it / TPP, t0 = (it - i * TPP) * 16;
      const int P = s_P[i], valid = s_valid[i];
      const bool la = P >= 0 && t0 + r < valid, lb = P >= 0 && t0 + r + 8 < valid;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < U; ++u) {
        mma_bf16(acc, a[0][u].x, a[1][u].x, a[0][u].y, a[1][u].y, bq[u][0], bq[u][1]);
        mma_bf16(acc, a[0][u].z, a[1][u].z, a[0][u].w, a[1][u].w, bq[u][2], bq[u][3]);
      }
      const int tok = it * 16 + r;             // = i * PS + t0 + r
      if (2 * c < G) {
        s_z[(2 * c) * ZS + tok] = la ? zscale * acc[0] : -INFINITY;
        s_z[(2 * c) * ZS + tok + 8] = lb ? zscale * acc[2] : -INFINITY;
      }
      if (2 * c + 1 < G) {
        s_z[(2 * c + 1) * ZS + tok] = la ? zscale * acc[1] : -INFINITY;
        s_z[(2 * c + 1) * ZS + tok + 8] = lb ? zscale * acc[3] : -INFINITY;
      }
    };
    uint4 bufA[2][U], bufB[2][U];
    int it = warp;
    if (it < tiles) load(it, bufA);
    for (; it < tiles; it += 2 * kLogitMmaWarps) {
      const int i2 = it + kLogitMmaWarps;
      if (i2 < tiles) load(i2, bufB);
      compute(it, bufA);
      if (i2 >= tiles) break;
      if (i2 + kLogitMmaWarps < tiles) load(i2 + kLogitMmaWarps, bufA);
      compute(i2, bufB);
    }
    __syncthreads();
    chunk_candidates(s_z, ZS, rn * PS, s_P, ps_log2, Hkv, g, warp, lane, cz, cs, cap_slots,
                     L);
  }
  write_split(L, warp, lane, split_floor, split_cnt, row0, S, s);
}

// ------------------------------------------------------------------------------ output

// Group (b, g)'s attended page count (out-of-range counts were flagged by the logits pass).
__device__ __forceinline__ int entmax_count(bool selected, const int32_t* sel_cnt, int sel_stride,
                                            long grp, int n_pages) {
  if (!selected) return n_pages;
  const int cnt = sel_cnt[grp];
  return cnt < 0 ? 0 : (cnt > sel_stride ? sel_stride : cnt);
}

// One block per (sequence, query head): the splits' candidate lists joined in split order (in
// shared memory when they fit), tau solved over them from the largest split floor, then the
// output sum over the support, reading V rows of support tokens only.
template <typename T, int D>
__global__ void __launch_bounds__(kOutThreads)
entmax_out_kernel(kv_cache_desc d, int G, const int32_t* __restrict__ sel_cnt, int sel_stride,
                  bool selected, int cap_slots, const float* __restrict__ split_floor,
                  const float* __restrict__ cand_z, const uint32_t* __restrict__ cand_row,
                  const int* __restrict__ split_cnt, int S, float* __restrict__ out,
                  float* __restrict__ tau_out, DevCtx ctx) {
  constexpr int NW = kOutThreads / 32;
  constexpr int EPL = D / 32;
  extern __shared__ __align__(16) unsigned char dyn[];
  float* s_z = reinterpret_cast<float*>(dyn);                     // [kCandCap]
  uint32_t* s_row = reinterpret_cast<uint32_t*>(s_z + kCandCap);  // [kCandCap]
  __shared__ TauSums s_red[NW];
  __shared__ int s_redi[NW];
  __shared__ float s_acc[NW][D];
  __shared__ int s_off[kMaxEntSplits + 1];
  __shared__ float s_fl[kMaxEntSplits];
  __shared__ float s_bc[4];
  __shared__ float s_wt[3 * NW];
  __shared__ float s_pts[2 * NW];
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, g = h / G, PS = d.page_size;
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, PS);
  const long grp = (long)b * Hkv + g;
  const int cnt = entmax_count(selected, sel_cnt, sel_stride, grp, n_pages);
  const long row = (long)b * Hq + h;
  float* o = out + row * D;
  if (cnt * PS == 0) {
    for (int i = tid; i < D; i += kOutThreads) o[i] = 0.f;
    if (tid == 0 && tau_out != nullptr) tau_out[row] = __int_as_float(0x7fc00000);
    return;
  }
  const int cps = ceil_div(cnt, S);
  for (int i = tid; i < S; i += kOutThreads) {
    s_fl[i] = __ldcg(split_floor + row * S + i);
    s_off[i] = __ldcg(split_cnt + row * S + i);
  }
  __syncthreads();
  // warp 0: the largest floor and the splits' candidate offsets (exclusive scan in place)
  if (warp == 0) {
    float f = -INFINITY;
    int run = 0;
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int sp = s0 + lane;
      const int c_ = sp < S ? s_off[sp] : 0;
      if (sp < S) f = fmaxf(f, s_fl[sp]);
      int incl = c_;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (sp < S) s_off[sp] = run + incl - c_;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, off));
    if (lane == 0) {
      s_off[S] = run;
      s_bc[2] = f;
    }
  }
  __syncthreads();
  const float floor_t = s_bc[2];
  const int nc = s_off[S];
  const bool in_smem = nc <= kCandCap;
  // candidate i -> its place in memory: it belongs to the last split with s_off <= i
  auto cand_src = [&](int i) -> long {
    int lo = 0, hi = S;                        // s_off[lo] <= i < s_off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= i) lo = mid;
      else hi = mid;
    }
    return row * cap_slots + (long)min(cnt, lo * cps) * PS + (i - s_off[lo]);
  };
  // in shared memory: only the candidates above the largest floor (every other one has weight
  // zero), compacted in candidate order; four per thread per round, loads in flight together
  int nk = nc;                                  // candidates held (block-uniform)
  if (in_smem) {
    nk = 0;
    for (int base = 0; base < nc; base += 4 * kOutThreads) {
      float zv[4];
      uint32_t rv[4];
      int mine = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + 4 * tid + u;
        const long src = i < nc ? cand_src(i) : 0;
        zv[u] = i < nc ? __ldcg(cand_z + src) : -INFINITY;
        rv[u] = i < nc ? __ldcg(cand_row + src) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) mine += zv[u] > floor_t ? 1 : 0;
      int incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_redi[warp] = incl;
      __syncthreads();
      int at = nk + incl - mine, round_total = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        at += w < warp ? s_redi[w] : 0;
        round_total += s_redi[w];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (zv[u] > floor_t) {
          s_z[at] = zv[u];
          s_row[at] = rv[u];
          ++at;
        }
      }
      nk += round_total;
      __syncthreads();                           // s_redi is reused
    }
  }
  // tau from the larger of the floor and the threshold of the lanes' largest candidates (both
  // lower bounds, f >= 0 there), about the mean of that threshold's support
  float tau;
  if (in_smem && nk <= 1024) {
    if (warp == 0) {
      float lm = -INFINITY;
      for (int i = lane; i < nk; i += 32) lm = fmaxf(lm, s_z[i]);
      const float2 w32 = warp32_tau(lm, lane);
      const float t0 = fmaxf(floor_t, w32.x - 1e-6f * (fabsf(w32.x) + 1.f));
      const float t = warp_entmax_tau([&](int i) { return s_z[i]; }, nk, t0, w32.y, lane);
      if (lane == 0) s_bc[0] = t;
    }
    __syncthreads();
    tau = s_bc[0];
  } else {
    // lower end: the larger of the floor and the threshold of a warp's lanes' largest
    // candidates; upper end: max z - 1/sqrt(nc) (the support, at most nc tokens, carries
    // weights summing to 1, each at most (max z - tau)^2)
    float lm = -INFINITY;
    for (int i = tid; i < nk; i += kOutThreads)
      lm = fmaxf(lm, in_smem ? s_z[i] : __ldcg(cand_z + cand_src(i)));
    const float2 w32 = warp32_tau(lm, lane);
    float wm = lm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
    if (lane == 0) {
      s_wt[warp] = w32.x;
      s_wt[NW + warp] = wm;
      s_wt[2 * NW + warp] = w32.y;
    }
    __syncthreads();
    float t0 = -INFINITY, zm = -INFINITY, pivot = floor_t;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if (s_wt[w] > t0) {                        // the pivot: the highest warp's support mean
        t0 = s_wt[w];
        pivot = s_wt[2 * NW + w];
      }
      zm = fmaxf(zm, s_wt[NW + w]);
    }
    t0 = fmaxf(floor_t, t0 - 1e-6f * (fabsf(t0) + 1.f));
    const float hi = fmaxf(t0, zm - rsqrtf((float)nk));
    if (in_smem)
      tau = block_entmax_tau_bracket<kOutThreads>([&](int i) { return s_z[i]; }, nk, t0, hi,
                                                  pivot, s_red, s_pts, s_bc);
    else
      tau = block_entmax_tau_bracket<kOutThreads>(
          [&](int i) { return __ldcg(cand_z + cand_src(i)); }, nc, t0, hi, pivot, s_red, s_pts,
          s_bc);
  }
  // out = sum over the support of (z - tau)^2 v. In shared memory the support (in candidate
  // order) is first compacted to the buffer's front as (weight, row); warps then take four
  // support tokens at a time, loads in flight together.
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  const T* __restrict__ vp = static_cast<const T*>(d.v_pool) + lane * EPL;
  if (in_smem) {
    // in place, round by round: every thread reads its candidate before any write of the
    // round, and a support token lands at an index no larger than its own
    int ns = 0;
    for (int base = 0; base < nk; base += kOutThreads) {
      const int i = base + tid;
      float zi = 0.f;
      uint32_t ri = 0;
      bool keep = false;
      if (i < nk) {
        zi = s_z[i];
        ri = s_row[i];
        keep = zi > tau;
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
        const float dz = zi - tau;
        s_z[at] = dz * dz;
        s_row[at] = ri;
      }
      ns += round_total;
    }
    __syncthreads();
    for (int i0 = warp * 4; i0 < ns; i0 += NW * 4) {
      float pw[4], vals[4][EPL];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool live = i0 + u < ns;
        pw[u] = live ? s_z[i0 + u] : 0.f;
        const T* rw = vp + (long)(live ? s_row[i0 + u] : 0u) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) vals[u][e] = live ? load_elem<T>(rw, e) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pw[u], vals[u][e], acc[e]);
      }
    }
  } else {
    for (int i = warp; i < nc; i += NW) {
      const long src = cand_src(i);
      const float z = __ldcg(cand_z + src);
      if (!(z > tau)) continue;
      const T* rw = vp + (long)__ldcg(cand_row + src) * D;
      const float pw = (z - tau) * (z - tau);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pw, load_elem<T>(rw, e), acc[e]);
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
  if (tid == 0 && tau_out != nullptr) tau_out[row] = tau;
}

// ------------------------------------------------------------------------------ launchers

template <typename T, int D, int G>
cudaError_t moments_t(const kv_cache_desc& d, const void* q, const void* stats, float scale,
                      float* zb, float* cz, float* vz, int stride, int sms, DevCtx ctx,
                      cudaStream_t s) {
  // rounds per warp: at least 2, and enough that the grid is about one wave
  const long rows = (long)d.page_table_stride * d.num_kv_heads * d.batch;
  const long slots = (long)mom_blocks<T, G>() * (sms > 0 ? sms : 1) * kMomWarps * 4;
  const int rpw = (int)std::max(2L, (rows + slots - 1) / slots);
  dim3 grid(ceil_div(d.page_table_stride, kMomWarps * rpw * 4), d.num_kv_heads, d.batch);
  return launch_pdl(entmax_moments_kernel<T, D, G>, grid, dim3(kMomWarps * 32), 0, s, d,
                    static_cast<const T*>(q), static_cast<const T*>(stats), 0.5f * scale, zb,
                    cz, vz, stride, rpw, ctx);
}

template <typename T, int D, int G>
cudaError_t logits_t(const kv_cache_desc& d, const void* q, float scale, const int32_t* sel,
                     const int32_t* cnt, int sel_stride, int S, const EntmaxScratch& w,
                     int cap_slots, DevCtx ctx, cudaStream_t s) {
  dim3 grid(S, d.num_kv_heads, d.batch);
  if constexpr (std::is_same<T, bf16_t>::value)
    return launch_pdl(entmax_logits_mma_kernel<D, G>, grid, dim3(kLogitMmaWarps * 32), 0, s, d,
                      static_cast<const T*>(q), scale, sel, cnt, sel_stride, cap_slots,
                      w.split_floor, w.cand_z, w.cand_row, w.split_cnt, ctx);
  else
    return launch_pdl(entmax_logits_kernel<T, D, G>, grid, dim3(kLogitWarps * 32), 0, s, d,
                      static_cast<const T*>(q), scale, sel, cnt, sel_stride, cap_slots,
                      w.split_floor, w.cand_z, w.cand_row, w.split_cnt, ctx);
}

template <typename T, int D>
cudaError_t out_t(const kv_cache_desc& d, int G, const int32_t* sel, const int32_t* cnt,
                  int sel_stride, const EntmaxScratch& w, int cap_slots, int S, float* out,
                  float* tau, DevCtx ctx, cudaStream_t s) {
  const size_t smem = (size_t)kCandCap * (sizeof(float) + sizeof(uint32_t));
  auto kern = entmax_out_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(d.num_kv_heads * G, d.batch);
  return launch_pdl(kern, grid, dim3(kOutThreads), smem, s, d, G, cnt, sel_stride,
                    sel != nullptr, cap_slots, w.split_floor, w.cand_z, w.cand_row, w.split_cnt,
                    S, out, tau, ctx);
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
                      float scale, float* zb, float* cz, float* vz, int stride, int sms,
                      DevCtx ctx, cudaStream_t s) {
#define SKV_CALL(GG) moments_t<T, D, GG>(d, q, stats, scale, zb, cz, vz, stride, sms, ctx, s)
  SKV_G_SWITCH(SKV_CALL)
#undef SKV_CALL
}

template <typename T, int D>
cudaError_t logits_d(const kv_cache_desc& d, int G, const void* q, float scale,
                     const int32_t* sel, const int32_t* cnt, int sel_stride, int S,
                     const EntmaxScratch& w, int cap_slots, DevCtx ctx, cudaStream_t s) {
#define SKV_CALL(GG) \
  logits_t<T, D, GG>(d, q, scale, sel, cnt, sel_stride, S, w, cap_slots, ctx, s)
  SKV_G_SWITCH(SKV_CALL)
#undef SKV_CALL
}

template <typename T, int D>
cudaError_t attn_d(const kv_cache_desc& d, int G, const void* q, float scale, const int32_t* sel,
                   const int32_t* cnt, int sel_stride, int S, const EntmaxScratch& w,
                   int cap_slots, float* out, float* tau, DevCtx ctx, cudaStream_t s) {
  const cudaError_t e = logits_d<T, D>(d, G, q, scale, sel, cnt, sel_stride, S, w, cap_slots,
                                       ctx, s);
  if (e != cudaSuccess) return e;
  return out_t<T, D>(d, G, sel, cnt, sel_stride, w, cap_slots, S, out, tau, ctx, s);
}

}  // namespace

cudaError_t launch_entmax_moments(const kv_cache_desc& d, int G, const void* q,
                                  const void* stats, float scale, float* zb, float* cz,
                                  float* vz, int stride, int sms, DevCtx ctx, cudaStream_t s) {
  const bool bf = d.dtype == KV_BF16;
  if (d.head_dim == 128)
    return bf ? moments_d<bf16_t, 128>(d, G, q, stats, scale, zb, cz, vz, stride, sms, ctx, s)
              : moments_d<float, 128>(d, G, q, stats, scale, zb, cz, vz, stride, sms, ctx, s);
  return bf ? moments_d<bf16_t, 64>(d, G, q, stats, scale, zb, cz, vz, stride, sms, ctx, s)
            : moments_d<float, 64>(d, G, q, stats, scale, zb, cz, vz, stride, sms, ctx, s);
}

cudaError_t launch_entmax_select(const int32_t* seq_lens, int page_size, int batch, int Hq,
                                 int Hkv, int table_stride, const float* zb, const float* cz,
                                 const float* vz, int stride, int k_max, int32_t* sel_idx,
                                 int32_t* sel_cnt, float* tau_hat, DevCtx ctx, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSelCluster, Hkv, batch);
  cfg.blockDim = dim3(kSelThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSelCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e;
#define SKV_ESEL(GG)                                                                           \
  e = cudaLaunchKernelEx(&cfg, entmax_select_kernel<GG>, seq_lens, page_size, Hq, Hkv,         \
                         table_stride, zb, cz, vz, stride, k_max, sel_idx, sel_cnt, tau_hat,    \
                         ctx);                                                                 \
  break
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
  return e != cudaSuccess ? e : cudaGetLastError();
}

int entmax_max_splits() { return kMaxEntSplits; }

cudaError_t launch_entmax_attn(const kv_cache_desc& d, int G, const void* q, float scale,
                               const int32_t* sel, const int32_t* cnt, int sel_stride, int S,
                               const EntmaxScratch& w, int cap_slots, float* out, float* tau,
                               DevCtx ctx, cudaStream_t s) {
  if (S < 1 || S > kMaxEntSplits) return cudaErrorInvalidValue;
  const bool bf = d.dtype == KV_BF16;
  if (d.head_dim == 128)
    return bf ? attn_d<bf16_t, 128>(d, G, q, scale, sel, cnt, sel_stride, S, w, cap_slots, out,
                                    tau, ctx, s)
              : attn_d<float, 128>(d, G, q, scale, sel, cnt, sel_stride, S, w, cap_slots, out,
                                   tau, ctx, s);
  return bf ? attn_d<bf16_t, 64>(d, G, q, scale, sel, cnt, sel_stride, S, w, cap_slots, out, tau,
                                 ctx, s)
            : attn_d<float, 64>(d, G, q, scale, sel, cnt, sel_stride, S, w, cap_slots, out, tau,
                                ctx, s);
}

}  // namespace skv
