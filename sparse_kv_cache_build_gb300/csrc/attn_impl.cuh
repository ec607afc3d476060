// Split-K decode attention over the selected pages of a paged KV cache.
//
// Source: "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding",
// abstract and Table 11: dense and sparse decoding read the cache through one split-K
// attention kernel, and the dense baseline is that kernel with every page kept (timing it
// through a masked kernel instead inflates the measured sparse speedup). Here the dense
// call is the same kernel with an implicit identity page list.
//
// Work decomposition: one CTA per (split s, KV head g, sequence b). The CTA handles every
// query head of the group, so each selected K/V page is read from HBM exactly once per
// step. Split s takes positions [s*c, min(cnt, (s+1)*c)), c = ceil(cnt / S), of the
// group's selected-page list.
//
// Data movement: the CTA first resolves its pages (selected index -> page table ->
// physical page, each checked against its bounds) into shared memory. Warp 0 then keeps
// NSTAGE tiles of 64 tokens in flight, one copy per lane: every page of a tile is one contiguous
// PS*D-element chunk of the pool per KV head, moved with one bulk asynchronous copy for K
// and one for V into the stage buffer, counted on the stage's mbarrier (bounded waits).
// K/V are streamed with an L2 evict-first policy.
//
// Compute per tile, warp w = (head half wh, token quarter wt); a warp owns 16 consecutive
// tokens (always inside one page, since PS >= 16) and up to 4 query heads:
//   q.k    eight lanes per token row, each holding D/8 elements of the warp's query heads
//          in registers; the four per-step partial dot products of the 4 rows x HPW heads
//          are reduced across the 8 lanes by a transposing butterfly (each shuffle level
//          halves the values a lane keeps), so a lane ends with whole logits at about one
//          shuffle per logit.
//   softmax online, per warp and head, in base 2 (logits pre-multiplied by
//          sm_scale*log2(e)); tokens past the sequence end or of missing pages are masked.
//   p.v    lane l owns D/32 consecutive output columns of every head of the warp; rows of V
//          are read once per warp with conflict-free 4- to 16-byte shared loads.
// At the end the four token warps of each head half are merged (log-sum-exp) in shared
// memory and the CTA writes its (m, l, acc) partial, m in natural-log units.
#pragma once

#include "kv_internal.cuh"

namespace skv {

template <typename T, int D, int G>
struct AttnCfg {
  static constexpr int EB = ElemTraits<T>::bytes;
  static constexpr int HPW = G < 4 ? G : 4;                // query heads per warp
  static constexpr int NWH = G / HPW;                      // warps across heads (1 or 2)
  static constexpr int NWT = kTileTokens / kWarpTokens;    // warps across tokens (4)
  static constexpr int NWARPS = NWT * NWH;
  static constexpr int THREADS = NWARPS * 32;
  static constexpr int ROW_BYTES = D * EB;
  static constexpr int TILE_BYTES = kTileTokens * ROW_BYTES;   // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int NSTAGE = 3;
  static constexpr int CPL = ROW_BYTES / 16 / 8;           // 16-byte chunks per lane per row
  static constexpr int EPC = 16 / EB;                      // elements per chunk
  static constexpr int EQK = CPL * EPC;                    // q elements per lane per head
  static constexpr int EPV = D / 32;                       // output columns per lane
  static constexpr int V0 = 4 * HPW;                       // partial logits per lane per tile
  static constexpr int FIN = V0 >= 8 ? V0 / 8 : 1;         // whole logits per lane after reduce
  static constexpr int LPH = 32 / HPW;                     // softmax lanes per head
  static constexpr int TPL = LPH >= 16 ? 1 : 16 / LPH;     // softmax tokens per lane

  // dynamic shared memory layout (bytes)
  static constexpr size_t OFF_STAGES = 0;
  static constexpr size_t OFF_PHYS = OFF_STAGES + (size_t)NSTAGE * STAGE_BYTES;
  static constexpr size_t OFF_VALID = OFF_PHYS + 4 * kMaxSplitPages;
  static constexpr size_t OFF_X = OFF_VALID + 2 * kMaxSplitPages;
  static constexpr size_t OFF_BAR = OFF_X + 4 * kTileTokens * G;
  static constexpr size_t SMEM = OFF_BAR + 8 * NSTAGE + 16;
  // end-of-CTA merge buffers alias the stage buffers
  static constexpr size_t MERGE_BYTES = 4 * (size_t)NWARPS * HPW * (D + 2);
  static_assert(MERGE_BYTES <= (size_t)NSTAGE * STAGE_BYTES, "merge buffers must fit");
  static_assert(CPL >= 1 && EPV >= 2, "unsupported shape");
};

template <typename T, int EPV>
__device__ __forceinline__ void load_v_row(const char* p, float* f) {
  if constexpr (sizeof(T) == 2) {
    if constexpr (EPV == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
      f[0] = bf16_lo(v); f[1] = bf16_hi(v);
    }
  } else {
    if constexpr (EPV == 4) {
      const float4 v = *reinterpret_cast<const float4*>(p);
      f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(p);
      f[0] = v.x; f[1] = v.y;
    }
  }
}

template <int HPW>
__device__ __forceinline__ void load_probs(const float* p, float* out) {
  if constexpr (HPW == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  } else if constexpr (HPW == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    out[0] = v.x; out[1] = v.y;
  } else {
    out[0] = p[0];
  }
}

// One level of the transposing butterfly: lanes whose `mask` bit is set keep the upper
// half of their values, the others the lower half; each adds its partner's copy.
template <int H>
__device__ __forceinline__ void butterfly_halve(float* v, int lane, int mask, int& off) {
  const bool up = (lane & mask) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float send = up ? v[i] : v[i + H];
    const float keep = up ? v[i + H] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
  }
  off += up ? H : 0;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(AttnCfg<T, D, G>::THREADS)
split_attn_kernel(kv_cache_desc d, const T* __restrict__ q, float qk_scale_log2,
                  const int32_t* __restrict__ sel_idx, const int32_t* __restrict__ sel_cnt,
                  int sel_stride, int S, float* __restrict__ part_acc,
                  float* __restrict__ part_ml, DevCtx ctx) {
  using C = AttnCfg<T, D, G>;
  extern __shared__ __align__(128) char smem[];
  int32_t* s_phys = reinterpret_cast<int32_t*>(smem + C::OFF_PHYS);
  int16_t* s_valid = reinterpret_cast<int16_t*>(smem + C::OFF_VALID);
  float* s_x = reinterpret_cast<float*>(smem + C::OFF_X);         // [64 tokens][G]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wt = warp % C::NWT, wh = warp / C::NWT;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, PS = d.page_size;
  pdl_trigger();
  pdl_wait();
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, PS);

  // ---- this split's run of the page list ------------------------------------------------
  int cnt = n_pages;
  const long grp = (long)b * Hkv + g;
  if (sel_idx != nullptr) {
    cnt = sel_cnt[grp];
    if (cnt < 0 || cnt > sel_stride) {
      if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      cnt = cnt < 0 ? 0 : sel_stride;
    }
  }
  // split s takes whole 64-token tiles [s T / S, (s + 1) T / S) of the list's T tiles
  const int ppt = kTileTokens / PS;
  const long n_tl = ceil_div(cnt, ppt);
  const int pos0 = min(cnt, (int)((long)s * n_tl / S) * ppt);
  int np = min(cnt, (int)((long)(s + 1) * n_tl / S) * ppt) - pos0;
  if (np > kMaxSplitPages) {                 // the host keeps S large enough; be defensive
    if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
    np = kMaxSplitPages;
  }
  const int32_t* table = d.page_table + (long)b * d.page_table_stride;
  for (int i = tid; i < np; i += C::THREADS) {
    int p = pos0 + i, P = -1, valid = 0;
    if (sel_idx != nullptr) p = sel_idx[grp * sel_stride + pos0 + i];
    if (p < 0 || p >= n_pages) {
      flag(ctx, KV_DEVERR_BAD_SEL);
    } else {
      P = table[p];
      if (P < 0 || P >= d.num_phys_pages) {
        flag(ctx, KV_DEVERR_BAD_PAGE);
        P = -1;
      } else {
        valid = min(PS, len - p * PS);
      }
    }
    s_phys[i] = P;
    s_valid[i] = (int16_t)valid;
  }
  if (tid == 0) {
    for (int i = 0; i < C::NSTAGE; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int PPT = kTileTokens / PS;          // pages per tile
  const int n_tiles = ceil_div(np, PPT);
  const uint32_t page_bytes = (uint32_t)PS * C::ROW_BYTES;
  const char* kbase = static_cast<const char*>(d.k_pool);
  const char* vbase = static_cast<const char*>(d.v_pool);

  // warp 0 issues a stage, lane l copying K (l even) or V (l odd) of page l / 2, so the copies
  // cost the warp one pass between its tiles instead of a loop in one thread
  auto issue = [&](int t) {
    const int st = t % C::NSTAGE;
    char* kdst = smem + C::OFF_STAGES + (size_t)st * C::STAGE_BYTES;
    const int i0 = t * PPT, i1 = min(np, i0 + PPT);
    const int i = i0 + (lane >> 1);
    const bool mine = lane < 2 * PPT && i < i1 && s_valid[i] > 0;
    const uint32_t copies = __popc(__ballot_sync(0xffffffffu, mine));
    if (lane == 0) mbar_arrive_expect_tx(&bars[st], copies * page_bytes);
    __syncwarp();
    if (mine) {
      const size_t src = ((size_t)s_phys[i] * Hkv + g) * page_bytes;
      const uint32_t dst = (uint32_t)(i - i0) * page_bytes + ((lane & 1) ? C::TILE_BYTES : 0u);
      bulk_g2s(kdst + dst, ((lane & 1) ? vbase : kbase) + src, page_bytes, &bars[st],
               l2_evict_first_policy());
    }
  };
  if (warp == 0) {
    for (int t = 0; t < C::NSTAGE && t < n_tiles; ++t) issue(t);
  }

  // ---- query registers (q.k layout: lane j of 8 owns chunks j, j+8, ...) ------------------
  const int grp8 = lane >> 3, j = lane & 7;
  float qr[C::HPW][C::EQK];
#pragma unroll
  for (int hh = 0; hh < C::HPW; ++hh) {
    const int h = g * G + wh * C::HPW + hh;
    const uint4* qrow = reinterpret_cast<const uint4*>(q + ((long)b * Hq + h) * D);
#pragma unroll
    for (int u = 0; u < C::CPL; ++u) chunk_to_f32<T>(qrow[j + 8 * u], &qr[hh][u * C::EPC]);
  }

  // ---- running state --------------------------------------------------------------------
  const int sm_hh = lane / C::LPH;                         // softmax head of this lane
  const int sm_sub = lane % C::LPH;
  const int sm_tok0 = (sm_sub % (16 / C::TPL)) * C::TPL;   // first softmax token
  const bool sm_owner = (C::HPW > 1) || lane < 16;         // lanes 16..31 mirror when HPW == 1
  float m_run = -INFINITY, l_run = 0.f;
  float acc[C::HPW][C::EPV];
#pragma unroll
  for (int hh = 0; hh < C::HPW; ++hh)
#pragma unroll
    for (int e = 0; e < C::EPV; ++e) acc[hh][e] = 0.f;

  bool aborted = false;
  int t = 0;
  for (; t < n_tiles; ++t) {
    const int st = t % C::NSTAGE;
    const bool ok = mbar_wait_bounded(&bars[st], (uint32_t)((t / C::NSTAGE) & 1), ctx.wait_ns);
    if (__syncthreads_or(!ok)) { aborted = true; break; }

    const char* ks = smem + C::OFF_STAGES + (size_t)st * C::STAGE_BYTES;
    const char* vs = ks + C::TILE_BYTES;
    // valid tokens of this warp's 16 (all inside one page)
    const int tok_base = wt * kWarpTokens;
    const int slot = t * PPT + tok_base / PS;
    int vt = 0;
    if (slot < np) vt = max(0, min(kWarpTokens, (int)s_valid[slot] - tok_base % PS));

    if (vt > 0) {
      // q.k: step st4 covers tokens tok_base + 4*st4 + grp8
      float v[C::V0];
#pragma unroll
      for (int st4 = 0; st4 < 4; ++st4) {
        const uint4* row = reinterpret_cast<const uint4*>(
            ks + (size_t)(tok_base + 4 * st4 + grp8) * C::ROW_BYTES);
        float part[C::HPW];
#pragma unroll
        for (int hh = 0; hh < C::HPW; ++hh) part[hh] = 0.f;
#pragma unroll
        for (int u = 0; u < C::CPL; ++u) {
          float f[C::EPC];
          chunk_to_f32<T>(row[j + 8 * u], f);
#pragma unroll
          for (int hh = 0; hh < C::HPW; ++hh)
#pragma unroll
            for (int e = 0; e < C::EPC; ++e) part[hh] = fmaf(qr[hh][u * C::EPC + e], f[e], part[hh]);
        }
#pragma unroll
        for (int hh = 0; hh < C::HPW; ++hh) v[st4 * C::HPW + hh] = part[hh];
      }
      int off = 0;
      butterfly_halve<C::V0 / 2>(v, lane, 4, off);
      butterfly_halve<C::V0 / 4>(v, lane, 2, off);
      if constexpr (C::V0 >= 8) {
        butterfly_halve<C::V0 / 8>(v, lane, 1, off);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
      }
      if (C::HPW > 1 || (lane & 1) == 0) {
#pragma unroll
        for (int i = 0; i < C::FIN; ++i) {
          const int vi = off + i;
          const int tl = (vi / C::HPW) * 4 + grp8;          // token within the warp's 16
          const int hl = wh * C::HPW + vi % C::HPW;
          const float x = tl < vt ? v[i] * qk_scale_log2 : -INFINITY;
          s_x[(tok_base + tl) * G + hl] = x;
        }
      }
      __syncwarp();

      // online softmax for this warp's tokens and heads
      float xs[C::TPL];
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < C::TPL; ++i) {
        xs[i] = s_x[(tok_base + sm_tok0 + i) * G + wh * C::HPW + sm_hh];
        mt = fmaxf(mt, xs[i]);
      }
#pragma unroll
      for (int o = 1; o < C::LPH; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float m_new = fmaxf(m_run, mt);
      float ls = 0.f;
#pragma unroll
      for (int i = 0; i < C::TPL; ++i) {
        const float p = xs[i] == -INFINITY ? 0.f : exp2f(xs[i] - m_new);
        ls += p;
        xs[i] = p;
      }
      __syncwarp();
      if (sm_owner) {
#pragma unroll
        for (int i = 0; i < C::TPL; ++i) s_x[(tok_base + sm_tok0 + i) * G + wh * C::HPW + sm_hh] = xs[i];
      }
      if (!sm_owner) ls = 0.f;
#pragma unroll
      for (int o = 1; o < C::LPH; o <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
      l_run = l_run * alpha + ls;
      m_run = m_new;
      __syncwarp();

      // p.v
      float al[C::HPW];
#pragma unroll
      for (int hh = 0; hh < C::HPW; ++hh) al[hh] = __shfl_sync(0xffffffffu, alpha, hh * C::LPH);
#pragma unroll
      for (int hh = 0; hh < C::HPW; ++hh)
#pragma unroll
        for (int e = 0; e < C::EPV; ++e) acc[hh][e] *= al[hh];
      const char* vrow = vs + (size_t)tok_base * C::ROW_BYTES + lane * C::EPV * C::EB;
      const float* prow = s_x + tok_base * G + wh * C::HPW;
      for (int tl = 0; tl < vt; ++tl) {
        float f[C::EPV], p[C::HPW];
        load_v_row<T, C::EPV>(vrow + (size_t)tl * C::ROW_BYTES, f);
        load_probs<C::HPW>(prow + tl * G, p);
#pragma unroll
        for (int hh = 0; hh < C::HPW; ++hh)
#pragma unroll
          for (int e = 0; e < C::EPV; ++e) acc[hh][e] = fmaf(p[hh], f[e], acc[hh][e]);
      }
    }
    __syncthreads();                                       // stage st is free again
    if (warp == 0 && t + C::NSTAGE < n_tiles) issue(t + C::NSTAGE);
  }

  const long out_row = ((long)b * Hq + g * G) * S + s;     // (b, first head of group, s)
  if (aborted) {
    if (tid == 0) {
      flag(ctx, KV_DEVERR_TIMEOUT);
      // let every copy this CTA issued land before the CTA (and its smem) goes away
      for (int u = t; u < n_tiles && u < t + C::NSTAGE; ++u)
        mbar_wait_bounded(&bars[u % C::NSTAGE], (uint32_t)((u / C::NSTAGE) & 1), ctx.wait_ns);
    }
    for (int i = tid; i < G * D; i += C::THREADS) {
      const int hl = i / D, dd = i % D;
      part_acc[(out_row + (long)hl * S) * D + dd] = 0.f;
      if (dd == 0) {
        part_ml[(out_row + (long)hl * S) * 2 + 0] = -INFINITY;
        part_ml[(out_row + (long)hl * S) * 2 + 1] = 0.f;
      }
    }
    return;
  }

  // ---- merge the token warps of each head half --------------------------------------------
  float* mg_acc = reinterpret_cast<float*>(smem + C::OFF_STAGES);      // [NWARPS][HPW][D]
  float* mg_m = mg_acc + C::NWARPS * C::HPW * D;                       // [NWARPS][HPW]
  float* mg_l = mg_m + C::NWARPS * C::HPW;
  if (sm_owner && sm_sub == 0) {
    mg_m[warp * C::HPW + sm_hh] = m_run;
    mg_l[warp * C::HPW + sm_hh] = l_run;
  }
#pragma unroll
  for (int hh = 0; hh < C::HPW; ++hh)
#pragma unroll
    for (int e = 0; e < C::EPV; ++e)
      mg_acc[(warp * C::HPW + hh) * D + lane * C::EPV + e] = acc[hh][e];
  __syncthreads();
  for (int i = tid; i < G * D; i += C::THREADS) {
    const int hl = i / D, dd = i % D;
    const int hw = hl / C::HPW, hh = hl % C::HPW;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < C::NWT; ++w2) M = fmaxf(M, mg_m[(hw * C::NWT + w2) * C::HPW + hh]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w2 = 0; w2 < C::NWT; ++w2) {
        const int wi = hw * C::NWT + w2;
        const float mw = mg_m[wi * C::HPW + hh];
        const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
        L = fmaf(mg_l[wi * C::HPW + hh], sc, L);
        A = fmaf(mg_acc[(wi * C::HPW + hh) * D + dd], sc, A);
      }
    }
    part_acc[(out_row + (long)hl * S) * D + dd] = A;
    if (dd == 0) {
      part_ml[(out_row + (long)hl * S) * 2 + 0] = M == -INFINITY ? -INFINITY : M * kLn2;
      part_ml[(out_row + (long)hl * S) * 2 + 1] = L;
    }
  }
}

template <typename T, int D, int G>
cudaError_t launch_split_attn_t(const kv_cache_desc& d, const void* q, float sm_scale,
                                const int32_t* sel_idx, const int32_t* sel_cnt, int sel_stride,
                                int S, float* part_acc, float* part_ml, DevCtx ctx,
                                cudaStream_t st) {
  using C = AttnCfg<T, D, G>;
  auto kern = split_attn_kernel<T, D, G>;
  static int attr_set_for_device[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set_for_device[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set_for_device[dev] = 1;
  }
  dim3 grid(S, d.num_kv_heads, d.batch);
  return launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, st, d, static_cast<const T*>(q),
                    sm_scale * kLog2e, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx);
}

template <typename T, int D>
cudaError_t launch_split_attn_d(const kv_cache_desc& d, const void* q, int G, float sm_scale,
                                const int32_t* sel_idx, const int32_t* sel_cnt, int sel_stride,
                                int S, float* part_acc, float* part_ml, DevCtx ctx,
                                cudaStream_t st) {
  switch (G) {
    case 1: return launch_split_attn_t<T, D, 1>(d, q, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx, st);
    case 2: return launch_split_attn_t<T, D, 2>(d, q, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx, st);
    case 4: return launch_split_attn_t<T, D, 4>(d, q, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx, st);
    case 8: return launch_split_attn_t<T, D, 8>(d, q, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
size_t split_attn_smem_t(int head_dim, int G) {
#define SKV_SMEM_CASE(DD, GG) if (head_dim == DD && G == GG) return AttnCfg<T, DD, GG>::SMEM;
  SKV_SMEM_CASE(64, 1) SKV_SMEM_CASE(64, 2) SKV_SMEM_CASE(64, 4) SKV_SMEM_CASE(64, 8)
  SKV_SMEM_CASE(128, 1) SKV_SMEM_CASE(128, 2) SKV_SMEM_CASE(128, 4) SKV_SMEM_CASE(128, 8)
#undef SKV_SMEM_CASE
  return 0;
}

// Per-dtype entry points, defined in attn_bf16.cu and attn_fp32.cu.
cudaError_t launch_split_attn_bf16(const kv_cache_desc& d, const void* q, int G, float sm_scale,
                                   const int32_t* sel_idx, const int32_t* sel_cnt,
                                   int sel_stride, int S, float* part_acc, float* part_ml,
                                   DevCtx ctx, cudaStream_t st);
cudaError_t launch_split_attn_fp32(const kv_cache_desc& d, const void* q, int G, float sm_scale,
                                   const int32_t* sel_idx, const int32_t* sel_cnt,
                                   int sel_stride, int S, float* part_acc, float* part_ml,
                                   DevCtx ctx, cudaStream_t st);
size_t split_attn_smem_bf16(int head_dim, int G);
size_t split_attn_smem_fp32(int head_dim, int G);

// bf16 step mode of the attention kernel (see StepArgs in attn_mma.cuh).
struct StepArgs;
cudaError_t launch_step_attn_bf16(const kv_cache_desc& d, const void* q, int G, float sm_scale,
                                  const int32_t* sel_idx, const int32_t* sel_cnt,
                                  int sel_stride, int S, float* part_acc, float* part_ml,
                                  DevCtx ctx, cudaStream_t st, const StepArgs& sa);
void step_attn_limits_bf16(int head_dim, int G, int* max_select_pages, int* max_splits);

}  // namespace skv
