// One sparse decode step in a single launch, for bf16 caches: page scores, top-k selection,
// split-K attention over the selected pages and the log-sum-exp merge.
//
// Sources: "EntmaxKV: Support-Aware Decoding for Entmax Attention", abstract (query-aware
// page scores from per-page statistics); "SparDA: Sparse Decoupled Attention for Efficient
// Long-Context LLM Inference", section 3.1 and appendix A (group-summed scores, top-k);
// "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding", abstract and
// Table 11 (dense and sparse decoding through the same split-K attention; dense is this
// kernel with every page kept).
//
// Why one launch: at 32K tokens the step moves ~49 MB, ~7 us at HBM speed, while four
// dependent launches each pay a ramp-up (first loads, launch latency) of several us. Here a
// thread-block cluster of CL CTAs (one per SM) owns one (sequence, KV head) group:
//   1. scores   CTA r scores pages [r*cp, (r+1)*cp): statistics rows come in by bulk
//               copies through the kernel's mbarrier ring; keys stay in shared memory.
//   2. select   radix select of the k-th key: every pass each CTA counts its own keys into
//               a shared histogram and the CL histograms are summed over distributed shared
//               memory (one cluster barrier per pass, double-buffered histograms).
//   3. compact  each CTA learns the (greater, equal) counts of the CTAs before it over
//               DSMEM, scans its keys in page order, and writes each kept page (physical id,
//               valid tokens) straight into the shared memory of the CTA whose split holds
//               that list position (split r takes [r*c, (r+1)*c), c = ceil(k / CL), the
//               split rule of kv_sparse_decode_attn with CL splits).
//   4. attend   the tensor-core attention of attn_mma.cuh over the CTA's run (same device
//               code as kv_sparse_decode_attn's kernel).
//   5. merge    CTA r merges a slice of the G*D outputs from all CL partials over DSMEM.
// Every CTA of a cluster takes the same branches (they depend only on the group's length,
// keep count and the summed histograms), so every cluster barrier is reached by all of them;
// bounded copy waits that run out mark the CTA's share empty, never skip a barrier.
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include "attn_mma.cuh"
#include "kv_internal.cuh"

namespace cg = cooperative_groups;

namespace skv {

constexpr int kFusedThreads = 128;
constexpr int kFusedNST = 4;
constexpr int kFusedMaxRange = 4096;   // pages one CTA scores
constexpr int kFusedMaxRun = 4096;     // selected pages one CTA attends

template <int D, int G>
struct FusedCfg {
  using M = MmaCfg<D, G>;
  static constexpr int NST = kFusedNST;
  static constexpr int ROW = 2 * D * 2;                       // bf16 stats row bytes
  static constexpr int CH = M::STAGE_BYTES / ROW;             // stats rows per ring stage
  static constexpr size_t OFF_RING = 0;
  static constexpr size_t OFF_KEYS = OFF_RING + (size_t)NST * M::STAGE_BYTES;
  static constexpr size_t OFF_RPHYS = OFF_KEYS + 4 * kFusedMaxRange;
  static constexpr size_t OFF_RUNP = OFF_RPHYS + 4 * kFusedMaxRange;
  static constexpr size_t OFF_RUNV = OFF_RUNP + 4 * kFusedMaxRun;
  static constexpr size_t OFF_W = OFF_RUNV + 2 * kFusedMaxRun;
  static constexpr size_t OFF_HIST = OFF_W + 4 * 2 * D;       // uint32 [2][256]
  static constexpr size_t OFF_GH = OFF_HIST + 4 * 2 * 256;    // uint32 [256]
  static constexpr size_t OFF_MISC = OFF_GH + 4 * 256;        // uint32 [16] + uint64 [8]
  static constexpr size_t OFF_BAR = OFF_MISC + 128;
  static constexpr size_t SMEM = OFF_BAR + 8 * NST + 1024;    // + alignment slack
  static_assert(M::MERGE_BYTES + 4 * M::PARTIAL_FLOATS <= (size_t)NST * M::STAGE_BYTES,
                "merge buffers must fit in the ring");
};

namespace {

__device__ __forceinline__ uint32_t fused_key(float s) {
  const uint32_t u = __float_as_uint(s + 0.0f);               // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int fused_keep(int n, double ratio, int budget) {
  if (n <= 0) return 0;
  if (budget > 0) return budget < n ? budget : n;
  if (ratio >= 1.0) return n;
  int k = (int)ceil(ratio * (double)n - 1e-9);
  k = k < 1 ? 1 : k;
  return k < n ? k : n;
}

// Exclusive scan over the 128 threads of (gt << 32 | eq); total written to *total.
__device__ __forceinline__ uint64_t scan128(uint64_t v, uint64_t* wtot, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  for (int w = 0; w < 4; ++w) before += (w < warp) ? wtot[w] : 0ull;
  if (threadIdx.x == 0) *total = wtot[0] + wtot[1] + wtot[2] + wtot[3];
  __syncthreads();
  return before + incl - v;
}

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kFusedThreads)
fused_step_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  kv_cache_desc d, const uint16_t* __restrict__ q,
                  const uint16_t* __restrict__ stats, float qk_scale_log2, double keep_ratio,
                  int budget, int k_max, int dense, int32_t* __restrict__ sel_out,
                  int32_t* __restrict__ cnt_out, float* __restrict__ out,
                  float* __restrict__ lse, DevCtx ctx) {
  using C = FusedCfg<D, G>;
  using M = MmaCfg<D, G>;
  extern __shared__ __align__(128) char smem_raw[];
  char* smem = reinterpret_cast<char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  char* ring = smem + C::OFF_RING;
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(smem + C::OFF_KEYS);
  int32_t* s_rphys = reinterpret_cast<int32_t*>(smem + C::OFF_RPHYS);
  int32_t* s_runp = reinterpret_cast<int32_t*>(smem + C::OFF_RUNP);
  int16_t* s_runv = reinterpret_cast<int16_t*>(smem + C::OFF_RUNV);
  float* s_w = reinterpret_cast<float*>(smem + C::OFF_W);
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(smem + C::OFF_HIST);
  uint32_t* s_gh = reinterpret_cast<uint32_t*>(smem + C::OFF_GH);
  uint32_t* s_misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);   // [0..15]
  uint64_t* s_misc64 = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC + 64);   // [0..7]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int r = (int)cluster.block_rank();
  const int g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, PS = d.page_size;

  pdl_trigger();
  if (tid == 0) {
    for (int i = 0; i < C::NST; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  pdl_wait();
  const int len = checked_len(ctx, d, b);
  const int n = ceil_div(len, PS);
  int k = dense ? n : fused_keep(n, keep_ratio, budget);
  if (!dense && k > k_max) {
    if (tid == 0 && r == 0) flag(ctx, KV_DEVERR_KEEP);
    k = k_max;
  }
  const long grp = (long)b * Hkv + g;
  const int32_t* table = d.page_table + (long)b * d.page_table_stride;
  uint32_t ring_uses = 0;
  int np = 0;

  if (!dense && k > 0 && k < n) {
    // ================= 1. scores of this CTA's page range =================================
    const int cp = ceil_div(n, CL);
    const int p0 = min(n, r * cp);
    int nr = min(n, p0 + cp) - p0;
    if (nr > kFusedMaxRange) {                 // the host keeps ranges within the limit
      if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      nr = kFusedMaxRange;
    }
    for (int i = tid; i < nr; i += kFusedThreads) {
      int P = table[p0 + i];
      if (P < 0 || P >= d.num_phys_pages) {
        flag(ctx, KV_DEVERR_BAD_PAGE);
        P = -1;
      }
      s_rphys[i] = P;
    }
    for (int t = tid; t < D; t += kFusedThreads) {
      float pos = 0.f, neg = 0.f;
      for (int h = g * G; h < (g + 1) * G; ++h) {
        const float x = __uint_as_float((uint32_t)q[((long)b * Hq + h) * D + t] << 16);
        pos += fmaxf(x, 0.f);
        neg += fminf(x, 0.f);
      }
      s_w[t] = neg;
      s_w[D + t] = pos;
    }
    __syncthreads();
    const int nch = ceil_div(nr, C::CH);
    auto issue_stats = [&](int c) {
      const uint32_t u = ring_uses + (uint32_t)c;
      const int st = (int)(u % C::NST);
      char* dst = ring + (size_t)st * M::STAGE_BYTES;
      const int i0 = c * C::CH, i1 = min(nr, i0 + C::CH);
      uint32_t bytes = 0;
      for (int i = i0; i < i1; ++i) bytes += s_rphys[i] >= 0 ? (uint32_t)C::ROW : 0u;
      mbar_arrive_expect_tx(&bars[st], bytes);
      const uint64_t pol = l2_evict_first_policy();
      for (int i = i0; i < i1; ++i) {
        const int P = s_rphys[i];
        if (P < 0) continue;
        bulk_g2s(dst + (size_t)(i - i0) * C::ROW,
                 reinterpret_cast<const char*>(stats) + ((size_t)P * Hkv + g) * C::ROW,
                 (uint32_t)C::ROW, &bars[st], pol);
      }
    };
    if (tid == 0) {
      for (int c = 0; c < C::NST && c < nch; ++c) issue_stats(c);
    }
    bool ok1 = true;
    int c = 0;
    for (; c < nch; ++c) {
      const uint32_t u = ring_uses + (uint32_t)c;
      const int st = (int)(u % C::NST);
      const bool ok = mbar_wait_bounded(&bars[st], (u / C::NST) & 1u, ctx.wait_ns);
      if (__syncthreads_or(!ok)) { ok1 = false; break; }
      const char* rows = ring + (size_t)st * M::STAGE_BYTES;
      const int i0 = c * C::CH, cnt = min(C::CH, nr - i0);
      const int j8 = tid & 7;
      constexpr int EPC = 8, CPL = (C::ROW / 16) / 8;
      for (int jj = tid >> 3; jj < ((cnt + 15) & ~15); jj += kFusedThreads / 8) {
        float acc = 0.f;
        const bool live = jj < cnt && s_rphys[i0 + jj] >= 0;
        if (live) {
          const uint4* row = reinterpret_cast<const uint4*>(rows + (size_t)jj * C::ROW);
#pragma unroll
          for (int uu = 0; uu < CPL; ++uu) {
            float f[EPC];
            chunk_to_f32<bf16_t>(row[j8 + 8 * uu], f);
            const float* wc = s_w + (j8 + 8 * uu) * EPC;
#pragma unroll
            for (int e = 0; e < EPC; ++e) acc = fmaf(wc[e], f[e], acc);
          }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (j8 == 0 && jj < cnt) s_keys[i0 + jj] = live ? fused_key(acc) : 0u;
      }
      __syncthreads();
      if (tid == 0 && c + C::NST < nch) issue_stats(c + C::NST);
    }
    if (!ok1) {
      if (tid == 0) {
        flag(ctx, KV_DEVERR_TIMEOUT);
        for (int v = c; v < nch && v < c + C::NST; ++v) {
          const uint32_t u = ring_uses + (uint32_t)v;
          mbar_wait_bounded(&bars[u % C::NST], (u / C::NST) & 1u, ctx.wait_ns);
        }
      }
      for (int i = tid; i < nr; i += kFusedThreads) s_keys[i] = 0u;
      __syncthreads();
    }
    ring_uses += (uint32_t)nch;

    // ================= 2. radix select across the cluster =================================
    uint32_t prefix = 0, mask = 0, remaining = (uint32_t)k;
    bool exact = false;
    const int iters = ceil_div(nr, kFusedThreads);
    int pass = 0;
    for (int shift = 24; shift >= 0 && !exact; shift -= 8, ++pass) {
      uint32_t* hist = s_hist + (pass & 1) * 256;
      for (int i = tid; i < 256; i += kFusedThreads) hist[i] = 0u;
      __syncthreads();
      for (int it = 0; it < iters; ++it) {
        const int i = it * kFusedThreads + tid;
        uint32_t digit = 256;
        if (i < nr) {
          const uint32_t key = s_keys[i];
          if ((key & mask) == prefix) digit = (key >> shift) & 255u;
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        if (digit < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
      cluster.sync();                          // every CTA's histogram of this pass is final
      for (int i = tid; i < 256; i += kFusedThreads) {
        uint32_t v = 0;
        for (int rk = 0; rk < CL; ++rk) v += cluster.map_shared_rank(hist, rk)[i];
        s_gh[i] = v;
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t cc[8], lane_sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) { cc[e] = s_gh[lane * 8 + e]; lane_sum += cc[e]; }
        uint32_t incl = lane_sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
          if (lane + o < 32) incl += y;
        }
        uint32_t above = incl - lane_sum;
        if (above < remaining && remaining <= incl) {
#pragma unroll
          for (int e = 7; e >= 0; --e) {
            if (above + cc[e] >= remaining) {
              s_misc[0] = prefix | ((uint32_t)(lane * 8 + e) << shift);
              s_misc[1] = remaining - above;
              s_misc[2] = (above + cc[e] == remaining) ? 1u : 0u;
              break;
            }
            above += cc[e];
          }
        }
      }
      __syncthreads();
      prefix = s_misc[0];
      remaining = s_misc[1];
      exact = s_misc[2] != 0u;
      mask |= 255u << shift;
      __syncthreads();                         // s_misc is rewritten next pass
    }
    const uint32_t T = prefix;
    const uint32_t take_eq = exact ? 0xffffffffu : remaining;

    // ================= 3. ordered compaction into the splits' runs ========================
    const int ipt = ceil_div(nr, kFusedThreads);          // keys per thread (contiguous)
    const int a0 = min(nr, tid * ipt), a1 = min(nr, a0 + ipt);
    uint32_t gt = 0, eq = 0;
    for (int i = a0; i < a1; ++i) {
      const uint32_t key = s_keys[i];
      gt += key > T;
      eq += key == T;
    }
    uint64_t* wtot = s_misc64;                 // [4]
    uint64_t* total = s_misc64 + 4;
    const uint64_t ex = scan128(((uint64_t)gt << 32) | eq, wtot, total);
    uint32_t* pub = s_misc + 4;                // this CTA's (gt, eq) totals for the others
    if (tid == 0) {
      pub[0] = (uint32_t)(*total >> 32);
      pub[1] = (uint32_t)(*total & 0xffffffffu);
    }
    cluster.sync();                            // totals published
    uint32_t gt_b = 0, eq_b = 0;
    for (int rk = 0; rk < r; ++rk) {
      const uint32_t* rp = cluster.map_shared_rank(pub, rk);
      gt_b += rp[0];
      eq_b += rp[1];
    }
    uint32_t gt_before = gt_b + (uint32_t)(ex >> 32);
    uint32_t eq_before = eq_b + (uint32_t)(ex & 0xffffffffu);
    const int c2 = ceil_div(k, CL);
    for (int i = a0; i < a1; ++i) {
      const uint32_t key = s_keys[i];
      int pos = -1;
      if (key > T) {
        pos = (int)(gt_before + min(eq_before, take_eq));
        ++gt_before;
      } else if (key == T) {
        if (eq_before < take_eq) pos = (int)(gt_before + eq_before);
        ++eq_before;
      }
      if (pos >= 0 && pos < k) {
        const int p = p0 + i;
        const int owner = pos / c2, idx = pos - owner * c2;
        const int P = s_rphys[i];
        cluster.map_shared_rank(s_runp, owner)[idx] = P;
        cluster.map_shared_rank(s_runv, owner)[idx] =
            (int16_t)(P >= 0 ? min(PS, len - p * PS) : 0);
        if (sel_out != nullptr) sel_out[grp * k_max + pos] = p;
      }
    }
    if (cnt_out != nullptr && r == 0 && tid == 0) cnt_out[grp] = k;
    cluster.sync();                            // every split's run is complete
    np = min(k, (r + 1) * c2) - min(k, r * c2);
  } else {
    // dense, nothing kept, or everything kept: split r takes its run of pages directly
    const int kk = (!dense && k == 0) ? 0 : (dense ? n : k);
    const int c2 = kk > 0 ? ceil_div(kk, CL) : 0;
    const int pos0 = min(kk, r * c2);
    np = min(kk, pos0 + c2) - pos0;
    if (np > kFusedMaxRun) {
      if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      np = kFusedMaxRun;
    }
    for (int i = tid; i < np; i += kFusedThreads) {
      const int p = pos0 + i;
      int P = table[p], valid = 0;
      if (P < 0 || P >= d.num_phys_pages) {
        flag(ctx, KV_DEVERR_BAD_PAGE);
        P = -1;
      } else {
        valid = min(PS, len - p * PS);
      }
      s_runp[i] = P;
      s_runv[i] = (int16_t)valid;
      if (!dense && sel_out != nullptr) sel_out[grp * k_max + p] = p;
    }
    if (!dense && cnt_out != nullptr && r == 0 && tid == 0) cnt_out[grp] = kk;
    __syncthreads();
  }

  // ================= 4. attention over this CTA's run ====================================
  uint32_t qa0[M::KSTEPS], qa2[M::KSTEPS];
  load_q_frags<D, G>(q, (long)b * Hq + g * G, qa0, qa2);
  WarpAcc<D> acc;
  acc.init();
  const bool ok4 = attend_run<D, G, C::NST>(&tmK, &tmV, ring, bars, ring_uses, s_runp, s_runv,
                                            np, g, Hkv, PS, qa0, qa2, qk_scale_log2, acc,
                                            ctx.wait_ns);
  float* scratch = reinterpret_cast<float*>(ring);
  float* part = scratch + 4 * G * (D + 2);
  cta_partial<D, G>(acc, scratch, part);
  if (!ok4) {
    if (tid == 0) flag(ctx, KV_DEVERR_TIMEOUT);
    for (int i = tid; i < G * D; i += kFusedThreads) part[i] = 0.f;
    if (tid < G) {
      part[G * D + tid] = -INFINITY;
      part[G * D + G + tid] = 0.f;
    }
    __syncthreads();
  }

  // ================= 5. merge the CL partials over DSMEM ===================================
  cluster.sync();                              // every partial is final
  const int E = ceil_div(G * D, CL);
  const int e0 = min(G * D, r * E), e1 = min(G * D, e0 + E);
  for (int e = e0 + tid; e < e1; e += kFusedThreads) {
    const int hl = e / D, dd = e % D;
    float Mx = -INFINITY;
    for (int rk = 0; rk < CL; ++rk)
      Mx = fmaxf(Mx, cluster.map_shared_rank(part, rk)[G * D + hl]);
    float L = 0.f, A = 0.f;
    if (Mx != -INFINITY) {
      for (int rk = 0; rk < CL; ++rk) {
        const float* rp = cluster.map_shared_rank(part, rk);
        const float mw = rp[G * D + hl];
        const float w = mw == -INFINITY ? 0.f : exp2f(mw - Mx);
        L = fmaf(rp[G * D + G + hl], w, L);
        A = fmaf(rp[hl * D + dd], w, A);
      }
    }
    const long oi = (long)b * Hq + g * G + hl;
    out[oi * D + dd] = Mx == -INFINITY ? 0.f : A / L;
    if (dd == 0 && lse != nullptr) lse[oi] = Mx == -INFINITY ? -INFINITY : Mx * kLn2 + logf(L);
  }
  cluster.sync();                              // no CTA leaves while others read its memory
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 fused_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

bool fused_pool_map(CUtensorMap* map, const void* pool, const kv_cache_desc& d) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = fused_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t rows = (cuuint64_t)d.num_phys_pages * d.num_kv_heads * d.page_size;
  const cuuint64_t dims[2] = {(cuuint64_t)d.head_dim, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d.head_dim * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)d.page_size};
  const cuuint32_t elem_strides[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides,
            box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t fused_launch_t(const kv_cache_desc& d, int CL, const void* q, const void* stats,
                           float sm_scale, double keep_ratio, int budget, int k_max, int dense,
                           int32_t* sel_out, int32_t* cnt_out, float* out, float* lse,
                           DevCtx ctx, cudaStream_t s, bool query_only, int* max_clusters) {
  using C = FusedCfg<D, G>;
  auto kern = fused_step_kernel<D, G>;
  static int attr_set_for_device[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set_for_device[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_set_for_device[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, d.num_kv_heads, d.batch);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (query_only) {
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(max_clusters, kern, &cfg);
  }
  CUtensorMap mk, mv;
  if (!fused_pool_map(&mk, d.k_pool, d) || !fused_pool_map(&mv, d.v_pool, d))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mk, mv, d, static_cast<const uint16_t*>(q),
                                     static_cast<const uint16_t*>(stats), sm_scale * kLog2e,
                                     keep_ratio, budget, k_max, dense, sel_out, cnt_out, out,
                                     lse, ctx);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t fused_dispatch(const kv_cache_desc& d, int G, int CL, const void* q,
                           const void* stats, float sm_scale, double keep_ratio, int budget,
                           int k_max, int dense, int32_t* sel_out, int32_t* cnt_out, float* out,
                           float* lse, DevCtx ctx, cudaStream_t s, bool query_only,
                           int* max_clusters) {
#define SKV_FUSED(DD, GG)                                                                   \
  if (d.head_dim == DD && G == GG)                                                          \
    return fused_launch_t<DD, GG>(d, CL, q, stats, sm_scale, keep_ratio, budget, k_max,     \
                                  dense, sel_out, cnt_out, out, lse, ctx, s, query_only,    \
                                  max_clusters);
  SKV_FUSED(128, 1) SKV_FUSED(128, 2) SKV_FUSED(128, 4) SKV_FUSED(128, 8)
  SKV_FUSED(64, 1) SKV_FUSED(64, 2) SKV_FUSED(64, 4) SKV_FUSED(64, 8)
#undef SKV_FUSED
  return cudaErrorInvalidValue;
}

}  // namespace

int fused_cluster_size(const kv_cache_desc& d, int G, int num_sms) {
  if (d.dtype != KV_BF16) return 0;
  if ((long long)d.num_phys_pages * d.num_kv_heads * d.page_size >= (1ll << 31)) return 0;
  const long groups = (long)d.batch * d.num_kv_heads;
  if (groups > num_sms) return 0;                // one CTA per SM: all groups in one wave
  int CL = 16;
  while (CL > 1 && groups * CL > num_sms) CL >>= 1;
  for (; CL >= 1; CL >>= 1) {
    // every CTA's score range and page run must fit its shared-memory arrays
    if (ceil_div(d.page_table_stride, CL) > kFusedMaxRange) return 0;
    int max_clusters = 0;
    if (fused_dispatch(d, G, CL, nullptr, nullptr, 1.f, 1.0, 0, 1, 1, nullptr, nullptr, nullptr,
                       nullptr, DevCtx{nullptr, 0}, 0, true, &max_clusters) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (max_clusters >= 1) return CL;
  }
  return 0;
}

cudaError_t launch_fused_step(const kv_cache_desc& d, int G, int CL, const void* q,
                              const void* stats, float sm_scale, double keep_ratio, int budget,
                              int k_max, int dense, int32_t* sel_out, int32_t* cnt_out,
                              float* out, float* lse, DevCtx ctx, cudaStream_t s) {
  int unused = 0;
  return fused_dispatch(d, G, CL, q, stats, sm_scale, keep_ratio, budget, k_max, dense,
                        sel_out, cnt_out, out, lse, ctx, s, false, &unused);
}

}  // namespace skv
