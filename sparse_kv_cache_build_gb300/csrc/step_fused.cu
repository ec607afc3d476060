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
// thread-block cluster of CL CTAs (one per SM, 8 warps each) owns one (sequence, KV head)
// group, and the cluster size is chosen so that every group's cluster is resident at once:
//   1. scores   CTA r scores pages [r*cp, (r+1)*cp) with all its page-table loads in
//               flight, then all its statistics-row loads (eight lanes per 512-byte row),
//               and writes each page's order key and physical id into the shared memory of
//               every CTA of the cluster (distributed shared memory), so that after one
//               cluster barrier each CTA holds the whole group.
//   2. select   each CTA finds the threshold of the k kept keys locally (cta_topk.cuh:
//               one radix pass from the highest differing bit, then the exact rank of the
//               threshold bin's keys), the same result in every CTA.
//   3. compact  each CTA scans the group's keys in page order and keeps only the list
//               positions of its own split (split r takes [r*c, (r+1)*c), c = ceil(k / CL),
//               the split rule of kv_sparse_decode_attn with CL splits).
//   4. attend   the tensor-core attention of attn_mma.cuh over the CTA's run (same device
//               code as kv_sparse_decode_attn's kernel), run by two independent 4-warp
//               halves of the CTA on the two halves of the run, each with its own two ring
//               stages and named barrier, so one half computes while the other waits on
//               copies (the overlap two CTAs per SM give the split kernel).
//   5. merge    CTA r merges a slice of the G*D outputs from all CL partials over DSMEM.
// Every CTA of a cluster takes the same branches (they depend only on the group's length,
// keep count and the summed histograms), so every cluster barrier is reached by all of them;
// bounded copy waits that run out mark the CTA's share empty, never skip a barrier.
#include <atomic>

#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include "attn_mma.cuh"
#include "cta_topk.cuh"
#include "kv_internal.cuh"

namespace cg = cooperative_groups;

namespace skv {

constexpr int kFusedThreads = 256;
constexpr int kFusedNST = 4;
constexpr int kFusedMaxRange = 4096;   // pages one CTA scores
constexpr int kFusedMaxRun = 4096;     // selected pages one CTA attends

template <int D, int G>
struct FusedCfg {
  using M = MmaCfg<D, G>;
  static constexpr int NST = kFusedNST;
  static constexpr int ROW = 2 * D * 2;                       // bf16 stats row bytes
  static constexpr int RING_WORDS = NST * M::STAGE_BYTES / 4;
  static constexpr size_t OFF_RING = 0;   // keys, physical ids, candidates; then the copies
  static constexpr size_t OFF_RPHYS = OFF_RING + (size_t)NST * M::STAGE_BYTES;
  static constexpr size_t OFF_RUNP = OFF_RPHYS + 4 * kFusedMaxRange;
  static constexpr size_t OFF_RUNV = OFF_RUNP + 4 * kFusedMaxRun;
  static constexpr size_t OFF_W = OFF_RUNV + 2 * kFusedMaxRun;
  static constexpr size_t OFF_HIST = OFF_W + 4 * 2 * D;       // uint32 [kHistWords]
  static constexpr size_t OFF_MISC = OFF_HIST + 4 * kHistWords;   // uint32 [16] + uint64 [16]
  static constexpr size_t OFF_MTAB = OFF_MISC + 192;          // float [16 ranks][2G]
  static constexpr size_t OFF_BAR = OFF_MTAB + 4 * 16 * 2 * G;
  static constexpr size_t SMEM = OFF_BAR + 8 * NST + 1024;    // + alignment slack
  static_assert(4 * (size_t)8 * G * (D + 2) + 4 * M::PARTIAL_FLOATS <=
                    (size_t)NST * M::STAGE_BYTES,
                "merge buffers must fit in the ring");
};


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
  int32_t* s_rphys = reinterpret_cast<int32_t*>(smem + C::OFF_RPHYS);
  int32_t* s_runp = reinterpret_cast<int32_t*>(smem + C::OFF_RUNP);
  int16_t* s_runv = reinterpret_cast<int16_t*>(smem + C::OFF_RUNV);
  float* s_w = reinterpret_cast<float*>(smem + C::OFF_W);
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(smem + C::OFF_HIST);
  uint32_t* s_misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);   // [0..15]
  uint64_t* s_misc64 = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC + 64);   // [0..15]
  float* s_mtab = reinterpret_cast<float*>(smem + C::OFF_MTAB);
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
  int k = dense ? n : keep_rule(n, nullptr, b, keep_ratio, budget);
  if (!dense && k > k_max) {
    if (tid == 0 && r == 0) flag(ctx, KV_DEVERR_KEEP);
    k = k_max;
  }
  const long grp = (long)b * Hkv + g;
  const int32_t* table = d.page_table + (long)b * d.page_table_stride;
  int np = 0;

  if (!dense && k > 0 && k < n) {
    // ================= 1. scores of this CTA's page range, gathered cluster-wide ==========
    const int cp = ceil_div(n, CL);
    const int p0 = min(n, r * cp);
    int nr = min(n, p0 + cp) - p0;
    if (nr > kFusedMaxRange) {                 // the host keeps ranges within the limit
      if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      nr = kFusedMaxRange;
    }
    // every CTA of the cluster must have started before its shared memory is written:
    // arrive now, wait just before the first remote store
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    uint32_t* ring_w = reinterpret_cast<uint32_t*>(ring);
    const int KW = cta_key_words(n);           // keys [KW], then physical ids [KW], by page
    int32_t* s_phys = reinterpret_cast<int32_t*>(ring_w + KW);
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
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    {
      constexpr int EPC = 8, CPL = (C::ROW / 16) / 8;   // 16-byte chunks per lane per row
      constexpr int NG = kFusedThreads / 8;             // 8-lane row groups
      constexpr int RB = 8;                             // rows per group in flight
      const int rg = tid >> 3, j8 = tid & 7;
      for (int base = 0; base < nr; base += NG * RB) {
        uint4 raw[RB][CPL];
        int Pu[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int i = base + u * NG + rg;
          Pu[u] = i < nr ? s_rphys[i] : -1;
          if (Pu[u] >= 0) {
            const uint4* row = reinterpret_cast<const uint4*>(
                reinterpret_cast<const char*>(stats) + ((size_t)Pu[u] * Hkv + g) * C::ROW);
#pragma unroll
            for (int uu = 0; uu < CPL; ++uu) raw[u][uu] = __ldg(row + j8 + 8 * uu);
          }
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int i = base + u * NG + rg;
          float acc = 0.f;
          if (Pu[u] >= 0) {
#pragma unroll
            for (int uu = 0; uu < CPL; ++uu) {
              float f[EPC];
              chunk_to_f32<bf16_t>(raw[u][uu], f);
              const float* wc = s_w + (j8 + 8 * uu) * EPC;
#pragma unroll
              for (int e = 0; e < EPC; ++e) acc = fmaf(wc[e], f[e], acc);
            }
          }
          acc += __shfl_xor_sync(0xffffffffu, acc, 4);
          acc += __shfl_xor_sync(0xffffffffu, acc, 2);
          acc += __shfl_xor_sync(0xffffffffu, acc, 1);
          if (i < nr) {
            const uint32_t key = Pu[u] >= 0 ? score_order_key(acc) : 0u;
            const int sl = p0 + i;
            for (int rk = j8; rk < CL; rk += 8) {      // the 8 lanes share the CL copies
              cluster.map_shared_rank(ring_w, rk)[sl] = key;
              cluster.map_shared_rank(s_phys, rk)[sl] = Pu[u];
            }
          }
        }
      }
    }
    cluster.sync();                            // every CTA holds every key and physical id

    // ================= 2. threshold of the k kept keys (the same in every CTA) ============
    const CtaKeys K = cta_keys_finish<kFusedThreads, false>(
        ring_w, n, reinterpret_cast<uint32_t*>(s_misc64), [](int, uint32_t key) { return key; });
    uint32_t T, take_eq;
    cta_threshold<kFusedThreads, false>(K, k, s_hist, s_misc, ring_w + 2 * KW,
                                        C::RING_WORDS - 2 * KW, T, take_eq);

    // ================= 3. this split's run of the ascending kept list =====================
    const int c2 = ceil_div(k, CL);
    const int pos0 = min(k, r * c2);
    np = min(k, pos0 + c2) - pos0;
    if (np > kFusedMaxRun) {
      if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      np = kFusedMaxRun;
    }
    cta_compact_window<kFusedThreads>(K, T, take_eq, s_misc64, s_misc, pos0, pos0 + np,
                                      [&](int p, int pos) {
      if (pos >= pos0 && pos < pos0 + np) {
        const int P = s_phys[p];
        s_runp[pos - pos0] = P;
        s_runv[pos - pos0] = (int16_t)(P >= 0 ? min(PS, len - p * PS) : 0);
        if (sel_out != nullptr) sel_out[grp * k_max + pos] = p;
      }
    });
    if (cnt_out != nullptr && r == 0 && tid == 0) cnt_out[grp] = k;
    __syncthreads();                           // runs written; the ring is free for copies
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

  // ================= 4. attention over this CTA's run, two halves ============================
  uint32_t qa0[M::KSTEPS], qa2[M::KSTEPS];
  load_q_frags<D, G>(q, (long)b * Hq + g * G, qa0, qa2);
  WarpAcc<D> acc;
  acc.init();
  const int half = warp >> 2;                  // warps 0-3 and 4-7
  const int np0 = (np + 1) / 2;
  const int my_np = half == 0 ? np0 : np - np0;
  const int my_off = half == 0 ? 0 : np0;
  const bool ok4 = attend_run<D, G, 2>(&tmK, &tmV, ring + (size_t)half * 2 * M::STAGE_BYTES,
                                       bars + 2 * half, 0u, s_runp + my_off, s_runv + my_off,
                                       my_np, g, Hkv, PS, qa0, qa2, qk_scale_log2, acc,
                                       ctx.wait_ns, 1 + half, tid & 127);
  const bool ok_all = __syncthreads_and(ok4) != 0;   // both halves done with the ring
  float* scratch = reinterpret_cast<float*>(ring);
  float* part = scratch + 8 * G * (D + 2);
  cta_partial<D, G, 8>(acc, scratch, part);
  if (!ok_all) {
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
  for (int i = tid; i < CL * 2 * G; i += kFusedThreads) {
    const int rk = i / (2 * G), j = i % (2 * G);
    s_mtab[i] = cluster.map_shared_rank(part, rk)[G * D + j];   // m [G] then l [G]
  }
  __syncthreads();
  const int E = ceil_div(G * D, CL);
  const int e0 = min(G * D, r * E), e1 = min(G * D, e0 + E);
  for (int e = e0 + tid; e < e1; e += kFusedThreads) {
    const int hl = e / D, dd = e % D;
    float Mx = -INFINITY;
    for (int rk = 0; rk < CL; ++rk) Mx = fmaxf(Mx, s_mtab[rk * 2 * G + hl]);
    float vals[16];
#pragma unroll
    for (int rk = 0; rk < 16; ++rk)
      vals[rk] = rk < CL ? cluster.map_shared_rank(part, rk)[hl * D + dd] : 0.f;
    float L = 0.f, A = 0.f;
    if (Mx != -INFINITY) {
#pragma unroll
      for (int rk = 0; rk < 16; ++rk) {
        if (rk >= CL) break;
        const float mw = s_mtab[rk * 2 * G + hl];
        const float w = mw == -INFINITY ? 0.f : exp2f(mw - Mx);
        L = fmaf(s_mtab[rk * 2 * G + G + hl], w, L);
        A = fmaf(vals[rk], w, A);
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

template <int D, int G>
cudaError_t fused_launch_t(const kv_cache_desc& d, int CL, const void* q, const void* stats,
                           float sm_scale, double keep_ratio, int budget, int k_max, int dense,
                           int32_t* sel_out, int32_t* cnt_out, float* out, float* lse,
                           DevCtx ctx, cudaStream_t s, bool query_only, int* max_clusters) {
  using C = FusedCfg<D, G>;
  auto kern = fused_step_kernel<D, G>;
  static std::atomic<int> attr_set_for_device[64];   // see launch_mma in attn_bf16.cu
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set_for_device[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_set_for_device[dev].store(1, std::memory_order_release);
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
  if (!pool_tensor_map(&mk, d.k_pool, d) || !pool_tensor_map(&mv, d.v_pool, d))
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
  // the group's keys, physical ids and some candidate room fit the copy ring
  const int ring_w =
      d.head_dim == 128 ? FusedCfg<128, 1>::RING_WORDS : FusedCfg<64, 1>::RING_WORDS;
  if (2 * cta_key_words(d.page_table_stride) + 1024 > ring_w) return 0;
  for (int CL = 16; CL >= 1; --CL) {
    if (groups * CL > num_sms) continue;
    // every CTA's score range and page run must fit its shared-memory arrays
    if (ceil_div(d.page_table_stride, CL) > kFusedMaxRange) return 0;
    int max_clusters = 0;
    if (fused_dispatch(d, G, CL, nullptr, nullptr, 1.f, 1.0, 0, 1, 1, nullptr, nullptr, nullptr,
                       nullptr, DevCtx{nullptr, 0}, 0, true, &max_clusters) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (max_clusters >= groups) return CL;       // every group's cluster resident at once
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
