// Split-K decode attention for bf16 caches on the tensor cores (GQA-packed q-group x page).
//
// Source: "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding",
// abstract and Table 11: dense and sparse decoding read the cache through one split-K
// attention kernel (dense = every page kept). Results are the (m, l, acc) partials of
// kv_sparse_decode_attn, exactly as the CUDA-core kernel of attn_impl.cuh defines them.
//
// Why tensor cores here: per token the work is G dot products of length D for q.k and G
// more for p.v. On CUDA cores that costs ~1200 warp instructions per 16-token tile and the
// kernel measured issue/latency-bound at 30-50% of HBM bandwidth. Packing the group's G
// query heads as the M = 16 rows of an m16n8k16 bf16 MMA cuts it to ~90 instructions:
//   q.k:  S[h][t] = Q[h][:] . K[t][:]   M = heads, N = 8 tokens x 2, K = D (D/16 steps)
//   p.v:  O[h][d] += P[h][t] V[t][d]     M = heads, N = 8 columns x D/8, K = 16 tokens
// The S accumulator fragment of q.k is, register for register, the A fragment of p.v (the
// FlashAttention-2 register reuse), so probabilities never leave registers. P is rounded to
// bf16 as a hi part plus a lo part (two MMAs), which keeps p to ~2^-17 relative: products
// of bf16 inputs are exact and every sum is float32, as on the CUDA-core path.
//
// Data movement: pages arrive by TMA tensor copies (cp.async.bulk.tensor.2d) from a 2-D view
// of the pool, [NP*Hkv*PS rows][D columns], in boxes of 64 columns x PS rows with the
// 128-byte swizzle, so ldmatrix reads eight consecutive rows at one 16-byte column chunk
// without bank conflicts. Each stage holds 64 tokens of K and of V; warp 0 keeps NSTAGE
// stages in flight, one copy per lane, completion counted on one mbarrier per stage (bounded
// waits).
#pragma once

#include <cuda.h>

#include "cta_topk.cuh"
#include "kv_internal.cuh"

namespace skv {

template <int D, int G>
struct MmaCfg {
  static constexpr int HALVES = D / 64;                    // 64-column (128-byte) halves
  static constexpr int HALF_BYTES = kTileTokens * 128;     // 64 rows x 128 B
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;   // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int NSTAGE = 3;
  static constexpr int THREADS = 128;                      // 4 warps x 16 tokens
  static constexpr int KSTEPS = D / 16;
  static constexpr int ONT = D / 8;                        // output n-tiles
  static constexpr size_t OFF_STAGES = 0;                  // from a 1024-aligned base
  static constexpr size_t OFF_PHYS = OFF_STAGES + (size_t)NSTAGE * STAGE_BYTES;
  static constexpr size_t OFF_VALID = OFF_PHYS + 4 * kMaxSplitPages;
  static constexpr size_t OFF_MISC = OFF_VALID + 2 * kMaxSplitPages;   // uint32 [16]
  static constexpr size_t OFF_WTOT = OFF_MISC + 64;                     // uint64 [8]
  static constexpr size_t OFF_BAR = OFF_WTOT + 64;
  static constexpr size_t SMEM = OFF_BAR + 8 * (NSTAGE + 1) + 1024;   // + alignment slack
  // the in-kernel selection keeps the group's keys (and, copied in bulk, its page-table
  // row) in the ring, then the histogram, with at least SELECT_CAND_MIN words left for
  // gathered candidates
  static constexpr int RING_WORDS = (int)((size_t)NSTAGE * STAGE_BYTES / 4);
  static constexpr int SELECT_CAND_MIN = 1024;
  static constexpr int MAX_SELECT_PAGES = RING_WORDS - kHistWords - SELECT_CAND_MIN;
  // a CTA partial: acc [G][D], then m [G] (base 2), then l [G]
  static constexpr size_t PARTIAL_FLOATS = (size_t)G * (D + 2);
  static constexpr size_t MERGE_BYTES = 4 * (size_t)4 * G * (D + 2);
  static_assert(MERGE_BYTES + 4 * PARTIAL_FLOATS <= (size_t)NSTAGE * STAGE_BYTES,
                "merge buffers must fit");
};

// 2-D TMA tile load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// Two floats -> packed bf16x2 (round to nearest even), first in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Byte offset, inside one 1024-byte-aligned half, of 16-byte chunk `c` of row `r` under
// the 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Barrier helpers for a group of `nthreads` threads on named barrier `bar_id`
// (bar_id 0 = the whole CTA through __syncthreads).
__device__ __forceinline__ bool group_or(bool pred, int bar_id, int nthreads) {
  if (bar_id == 0) return __syncthreads_or(pred) != 0;
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"((uint32_t)pred), "r"(bar_id), "r"(nthreads) : "memory");
  return r != 0;
}

__device__ __forceinline__ void group_sync(int bar_id, int nthreads) {
  if (bar_id == 0) __syncthreads();
  else asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
}

// Per-warp running state of the online softmax: O accumulator fragments (rows lane/4 are
// the group's query heads; rows lane/4 + 8 are padding), the row max (base 2) and this
// lane's share of the row sum.
template <int D>
struct WarpAcc {
  float o[D / 8][4];
  float m_run;
  float l_lane;
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    m_run = -INFINITY;
    l_lane = 0.f;
  }
};

// q rows of the group as m16n8k16 A fragments (rows >= G are zero).
template <int D, int G>
__device__ __forceinline__ void load_q_frags(const uint16_t* q, long row0, uint32_t* qa0,
                                             uint32_t* qa2) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  const bool live = gid < G;
  const uint16_t* qrow = q + (row0 + (live ? gid : 0)) * D;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t* p32 = reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tig);
    qa0[ks] = live ? p32[0] : 0u;
    qa2[ks] = live ? p32[4] : 0u;
  }
}

// Stream a run of np pages (physical ids and valid-token counts in shared memory) through a
// ring of NST stages of 64 tokens, accumulating attention of the group's query heads into
// the four warps' WarpAcc. All 128 threads call it; warp 0 issues the TMA copies. Ring use
// number ring_base + t goes to stage (ring_base + t) % NST with phase parity
// ((ring_base + t) / NST) & 1, so one ring can serve several runs or phases of a kernel.
// It consumes ceil(np / (64 / PS)) ring uses. Returns false if a wait ran out (the copies
// this CTA issued have then been drained, bounded).
//
// The group running it is 4 warps (128 threads): by default the whole CTA synchronised with
// __syncthreads; a CTA may run two independent groups, each with its own stages, barriers,
// run and named barrier bar_id (gtid = thread index within the group).
template <int D, int G, int NST, bool WARP_ISSUE = true>
__device__ bool attend_run(const CUtensorMap* tmK, const CUtensorMap* tmV, char* stages,
                          uint64_t* bars, uint32_t ring_base, const int32_t* s_phys,
                          const int16_t* s_valid, int np, int g, int Hkv, int PS,
                          const uint32_t* qa0, const uint32_t* qa2, float qk_scale_log2,
                          WarpAcc<D>& acc, unsigned long long wait_ns, int bar_id = 0,
                          int gtid = -1) {
  using C = MmaCfg<D, G>;
  const int tid = gtid >= 0 ? gtid : (int)threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int tig = lane & 3;
  const int lm = lane >> 3, lr = lane & 7;
  const int PPT = kTileTokens / PS;
  const int n_tiles = ceil_div(np, PPT);
  const uint32_t page_half_bytes = (uint32_t)PS * 128;

  // warp 0 issues a stage. Several pages a stage (PS < 64): lane l copies one 64-column half
  // of K or V of one page (at most 4 pages x 2 halves x 2 tensors = 16 copies), so the issue
  // costs the warp one pass instead of a loop of copies in one thread between its tiles
  // (dense 128K: 115.6 -> 97.6 us a step). With WARP_ISSUE false (the instantiation for long
  // tables, whose larger selection code measured 1.3 us slower at 1M with the warp-wide form
  // compiled in) or one page a stage, lane 0 copies the stage's halves in a loop.
  auto issue = [&](int t) {
    const uint32_t u = ring_base + (uint32_t)t;
    const int st = (int)(u % NST);
    char* kdst = stages + (size_t)st * C::STAGE_BYTES;
    char* vdst = kdst + C::TILE_BYTES;
    const int i0 = t * PPT, i1 = min(np, i0 + PPT);
    const uint64_t pol = l2_evict_first_policy();
    if (!WARP_ISSUE || PPT == 1) {
      if (lane == 0) {
        uint32_t bytes = 0;
        for (int i = i0; i < i1; ++i)
          bytes += s_valid[i] > 0 ? 2u * C::HALVES * page_half_bytes : 0u;
        mbar_arrive_expect_tx(&bars[st], bytes);
        for (int i = i0; i < i1; ++i) {
          if (s_valid[i] <= 0) continue;
          const int y = (s_phys[i] * Hkv + g) * PS;
          const uint32_t off = (uint32_t)(i - i0) * page_half_bytes;
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h) {
            tma_load_2d(kdst + h * C::HALF_BYTES + off, tmK, 64 * h, y, &bars[st], pol);
            tma_load_2d(vdst + h * C::HALF_BYTES + off, tmV, 64 * h, y, &bars[st], pol);
          }
        }
      }
      return;
    }
    constexpr int PER_PAGE = 2 * C::HALVES;
    const int i = i0 + lane / PER_PAGE;
    const bool mine = lane < PPT * PER_PAGE && i < i1 && s_valid[i] > 0;
    const uint32_t copies = __popc(__ballot_sync(0xffffffffu, mine));
    if (lane == 0) mbar_arrive_expect_tx(&bars[st], copies * page_half_bytes);
    __syncwarp();
    if (mine) {
      const int h = (lane >> 1) % C::HALVES;
      const int y = (s_phys[i] * Hkv + g) * PS;
      const uint32_t off = (uint32_t)h * C::HALF_BYTES + (uint32_t)(i - i0) * page_half_bytes;
      if (lane & 1) tma_load_2d(vdst + off, tmV, 64 * h, y, &bars[st], pol);
      else tma_load_2d(kdst + off, tmK, 64 * h, y, &bars[st], pol);
    }
  };
  const bool issuer = WARP_ISSUE ? warp == 0 : tid == 0;
  if (issuer) {
    for (int t = 0; t < NST && t < n_tiles; ++t) issue(t);
  }

  bool aborted = false;
  int t = 0;
  for (; t < n_tiles; ++t) {
    const uint32_t u = ring_base + (uint32_t)t;
    const int st = (int)(u % NST);
    const bool ok = mbar_wait_bounded(&bars[st], (u / NST) & 1u, wait_ns);
    if (group_or(!ok, bar_id, 128)) { aborted = true; break; }

    const int tok_base = warp * kWarpTokens;
    const int slot = t * PPT + tok_base / PS;
    int vt = 0;
    if (slot < np) vt = max(0, min(kWarpTokens, (int)s_valid[slot] - tok_base % PS));

    if (vt > 0) {
      const uint32_t kbase = smem_addr(stages + (size_t)st * C::STAGE_BYTES);
      const uint32_t vbase = kbase + C::TILE_BYTES;
      // ---- S = Q K^T for 16 tokens (two n-tiles of 8) ------------------------------------
      // even and odd k-steps accumulate apart (two dependent chains of KSTEPS/2 MMAs each
      // instead of one of KSTEPS), summed once at the end
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float so[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        const int row = tok_base + (lm >> 1) * 8 + lr;
        const int col = ks * 16 + (lm & 1) * 8;              // element column
        const uint32_t addr = kbase + (col >> 6) * C::HALF_BYTES + swz(row, (col & 63) >> 3);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(addr, b00, b01, b10, b11);
        float (&a)[2][4] = (ks & 1) ? so : sc;
        mma_bf16(a[0], qa0[ks], 0u, qa2[ks], 0u, b00, b01);
        mma_bf16(a[1], qa0[ks], 0u, qa2[ks], 0u, b10, b11);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sc[0][i] += so[0][i];
        sc[1][i] += so[1][i];
      }
      // ---- online softmax (base 2) for row gid; tokens nt*8 + 2*tig + {0,1} ---------------
      float x[4];
      x[0] = (2 * tig < vt) ? sc[0][0] * qk_scale_log2 : -INFINITY;
      x[1] = (2 * tig + 1 < vt) ? sc[0][1] * qk_scale_log2 : -INFINITY;
      x[2] = (8 + 2 * tig < vt) ? sc[1][0] * qk_scale_log2 : -INFINITY;
      x[3] = (8 + 2 * tig + 1 < vt) ? sc[1][1] * qk_scale_log2 : -INFINITY;
      float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      const float m_new = fmaxf(acc.m_run, mt);
      const float alpha = acc.m_run == -INFINITY ? 0.f : exp2f(acc.m_run - m_new);
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = x[i] == -INFINITY ? 0.f : exp2f(x[i] - m_new);
      acc.l_lane = acc.l_lane * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
      acc.m_run = m_new;
      if (!__all_sync(0xffffffffu, alpha == 1.f)) {
#pragma unroll
        for (int nt = 0; nt < C::ONT; ++nt) { acc.o[nt][0] *= alpha; acc.o[nt][1] *= alpha; }
      }
      // P as bf16 hi + lo A fragments (rows gid; rows gid + 8 are zero)
      const uint32_t ph0 = pack_bf16(p[0], p[1]), ph2 = pack_bf16(p[2], p[3]);
      const uint32_t pl0 = pack_bf16(p[0] - bf16_lo_f(ph0), p[1] - bf16_hi_f(ph0));
      const uint32_t pl2 = pack_bf16(p[2] - bf16_lo_f(ph2), p[3] - bf16_hi_f(ph2));
      // masked tokens of a partial page: zero their V elements (may hold any bits)
      uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
      if (vt < kWarpTokens) {
        vm0 = (2 * tig < vt ? 0x0000ffffu : 0u) | (2 * tig + 1 < vt ? 0xffff0000u : 0u);
        vm1 = (8 + 2 * tig < vt ? 0x0000ffffu : 0u) | (8 + 2 * tig + 1 < vt ? 0xffff0000u : 0u);
      }
      // ---- O += P V ------------------------------------------------------------------------
#pragma unroll
      for (int np2 = 0; np2 < C::ONT / 2; ++np2) {
        const int row = tok_base + (lm & 1) * 8 + lr;
        const int col = np2 * 16 + (lm >> 1) * 8;
        const uint32_t addr = vbase + (col >> 6) * C::HALF_BYTES + swz(row, (col & 63) >> 3);
        uint32_t v00, v01, v10, v11;
        ldsm_x4_t(addr, v00, v01, v10, v11);
        v00 &= vm0; v01 &= vm1; v10 &= vm0; v11 &= vm1;
        mma_bf16(acc.o[2 * np2], ph0, 0u, ph2, 0u, v00, v01);
        mma_bf16(acc.o[2 * np2], pl0, 0u, pl2, 0u, v00, v01);
        mma_bf16(acc.o[2 * np2 + 1], ph0, 0u, ph2, 0u, v10, v11);
        mma_bf16(acc.o[2 * np2 + 1], pl0, 0u, pl2, 0u, v10, v11);
      }
    }
    group_sync(bar_id, 128);                               // the stage is free again
    if (issuer && t + NST < n_tiles) issue(t + NST);
  }
  if (aborted && tid == 0) {
    // let every copy this CTA issued land before its shared memory is reused or freed
    for (int v = t; v < n_tiles && v < t + NST; ++v) {
      const uint32_t u = ring_base + (uint32_t)v;
      mbar_wait_bounded(&bars[u % NST], (u / NST) & 1u, wait_ns);
    }
  }
  return !aborted;
}

// Merge the NW warps' states into one CTA partial in shared memory `part`:
// acc [G][D] (relative to m), m [G] in base 2 (-inf when empty), l [G]. `scratch` holds
// NW*G*(D+2) floats and may alias the stage ring once it is idle. Ends with __syncthreads.
template <int D, int G, int NW = 4>
__device__ void cta_partial(WarpAcc<D>& acc, float* scratch, float* part) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  float l_row = acc.l_lane;
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
  float* mg_o = scratch;                                   // [NW][G][D]
  float* mg_m = mg_o + NW * G * D;                         // [NW][G]
  float* mg_l = mg_m + NW * G;
  if (gid < G) {
    if (tig == 0) {
      mg_m[warp * G + gid] = acc.m_run;
      mg_l[warp * G + gid] = l_row;
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      mg_o[(warp * G + gid) * D + nt * 8 + 2 * tig] = acc.o[nt][0];
      mg_o[(warp * G + gid) * D + nt * 8 + 2 * tig + 1] = acc.o[nt][1];
    }
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int hl = i / D, dd = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < NW; ++w2) M = fmaxf(M, mg_m[w2 * G + hl]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) {
        const float mw = mg_m[w2 * G + hl];
        const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
        L = fmaf(mg_l[w2 * G + hl], sc, L);
        A = fmaf(mg_o[(w2 * G + hl) * D + dd], sc, A);
      }
    }
    part[hl * D + dd] = A;
    if (dd == 0) {
      part[G * D + hl] = M;
      part[G * D + G + hl] = L;
    }
  }
  __syncthreads();
}

// Optional parts of a decode step run inside the attention kernel.
//  * scores != nullptr: each CTA selects its own run of the group's kept pages from the
//    score row (keep rule keep_rule(n, ratio, budget) clamped to k_max), instead of reading
//    a selected list; split 0 also writes the whole list to sel_out[grp][k_max] and the
//    count to cnt_out[grp] when those are given.
//  * counters != nullptr: after writing its partial, each CTA counts itself in
//    counters[grp] (which must start at 0); the last CTA of the group merges the S partials
//    into out/lse and resets the counter to 0.
struct StepArgs {
  const float* scores;
  int scores_stride;
  double keep_ratio;
  int budget;
  int k_max;
  int32_t* sel_out;
  int32_t* cnt_out;
  int32_t* counters;
  float* out;
  float* lse;
};

// Two CTAs per SM (shared memory allows no more), so up to 255 registers a thread. LONG: the
// in-kernel selection may filter the keys by a sample first (cta_threshold); launched for
// page tables of at least topk_detail::kPrefilterMinPages pages keeping at most a sixteenth.
template <int D, int G, bool LONG>
__global__ void __launch_bounds__(MmaCfg<D, G>::THREADS, 2)
split_attn_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, kv_cache_desc d,
                      const uint16_t* __restrict__ q, float qk_scale_log2,
                      const int32_t* __restrict__ sel_idx, const int32_t* __restrict__ sel_cnt,
                      int sel_stride, int S, float* __restrict__ part_acc,
                      float* __restrict__ part_ml, DevCtx ctx, StepArgs sa) {
  using C = MmaCfg<D, G>;
  extern __shared__ __align__(128) char smem_raw[];
  char* smem = reinterpret_cast<char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  int32_t* s_phys = reinterpret_cast<int32_t*>(smem + C::OFF_PHYS);
  int16_t* s_valid = reinterpret_cast<int16_t*>(smem + C::OFF_VALID);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int Hkv = d.num_kv_heads, Hq = Hkv * G, PS = d.page_size;
  pdl_trigger();
  if (tid == 0) {
    for (int i = 0; i <= C::NSTAGE; ++i) mbar_init(&bars[i], 1);   // stages + row copies
    fence_mbar_init();
  }
  __syncthreads();                           // the barriers are initialised for every thread
  pdl_wait();
  const long grp = (long)b * Hkv + g;
  const int32_t* table = d.page_table + (long)b * d.page_table_stride;
  uint32_t* ring = reinterpret_cast<uint32_t*>(smem + C::OFF_STAGES);
  // Step mode: the group's score row, and where it fits beside it the page-table row
  // (page_table_stride entries each, of which the first n_pages are used), are copied into
  // the ring in bulk at once, before the sequence length is known, where the rows allow it.
  const float* srow = sa.scores != nullptr ? sa.scores + grp * sa.scores_stride : nullptr;
  const int KW = cta_key_words(d.page_table_stride);
  const bool keys_bulk = srow != nullptr && KW <= C::MAX_SELECT_PAGES &&
                         cta_row_bulk_ok(srow, sa.scores_stride);
  const bool table_bulk = keys_bulk && 2 * KW <= C::MAX_SELECT_PAGES &&
                          cta_row_bulk_ok(table, d.page_table_stride);
  if (keys_bulk && tid == 0) {
    mbar_arrive_expect_tx(&bars[C::NSTAGE], (table_bulk ? 8u : 4u) * (uint32_t)KW);
    cta_bulk_copy(ring, srow, 4u * (uint32_t)KW, &bars[C::NSTAGE]);
    if (table_bulk) cta_bulk_copy(ring + KW, table, 4u * (uint32_t)KW, &bars[C::NSTAGE]);
  }
  const int len = checked_len(ctx, d, b);
  const int n_pages = ceil_div(len, PS);

  // ---- this split's run of the page list ------------------------------------------------
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int32_t* tab = table;                // the page-table row, in global or shared memory
  // resolve logical page p (list position pos) into run slot i
  auto resolve = [&](int i, int p) {
    int P = -1, valid = 0;
    if (p < 0 || p >= n_pages) {
      flag(ctx, KV_DEVERR_BAD_SEL);
    } else {
      P = tab[p];
      if (P < 0 || P >= d.num_phys_pages) {
        flag(ctx, KV_DEVERR_BAD_PAGE);
        P = -1;
      } else {
        valid = min(PS, len - p * PS);
      }
    }
    s_phys[i] = P;
    s_valid[i] = (int16_t)valid;
  };
  int cnt = n_pages;
  if (sa.scores != nullptr) {
    cnt = keep_rule(n_pages, nullptr, b, sa.keep_ratio, sa.budget);
    if (cnt > sa.k_max) {
      if (s == 0 && tid == 0) flag(ctx, KV_DEVERR_KEEP);
      cnt = sa.k_max;
    }
    if (s == 0 && tid == 0 && sa.cnt_out != nullptr) sa.cnt_out[grp] = cnt;
  } else if (sel_idx != nullptr) {
    cnt = sel_cnt[grp];
    if (cnt < 0 || cnt > sel_stride) {
      if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      cnt = cnt < 0 ? 0 : sel_stride;
    }
  }
  // split s takes whole 64-token tiles [s T / S, (s + 1) T / S) of the list's T tiles, so
  // the splits differ by at most one tile and only the last tile of the list is partial
  const int ppt = kTileTokens / PS;
  const long n_tl = ceil_div(cnt, ppt);
  const int pos0 = min(cnt, (int)((long)s * n_tl / S) * ppt);
  int np = min(cnt, (int)((long)(s + 1) * n_tl / S) * ppt) - pos0;
  if (np > kMaxSplitPages) {
    if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
    np = kMaxSplitPages;
  }
  uint32_t qa0[C::KSTEPS], qa2[C::KSTEPS];
  bool rows_waited = false;
  if (sa.scores != nullptr && cnt > 0 && cnt < n_pages && n_pages <= C::MAX_SELECT_PAGES) {
    // select this CTA's run from the group's scores (the ring is free until the first copy);
    // q is fetched meanwhile
    load_q_frags<D, G>(q, (long)b * Hq + g * G, qa0, qa2);
    if (!table_bulk)
      for (int j = tid; j * 32 < n_pages; j += C::THREADS) prefetch_l2(table + j * 32);
    int used;
    if (keys_bulk) {
      if (!mbar_wait_bounded(&bars[C::NSTAGE], 0u, ctx.wait_ns) && tid == 0)
        flag(ctx, KV_DEVERR_TIMEOUT);
      rows_waited = true;
      used = table_bulk ? 2 * KW : KW;
    } else {
      cta_fill_loads<C::THREADS>(ring, srow, n_pages);
      used = cta_key_words(n_pages);
    }
    const CtaKeys K = cta_keys_finish<C::THREADS>(ring, n_pages, misc + 8);
    uint32_t T, take_eq;
    CtaCand list;
    cta_threshold<C::THREADS, LONG>(K, cnt, ring + used, misc, ring + used + kHistWords,
                                    C::RING_WORDS - used - kHistWords, T, take_eq, &list);
    // this CTA's run only; each CTA also writes its run's part of the selection output.
    // After a prefilter, from its page-ordered candidates; else a short run (many splits):
    // per-thread counts and one warp walking from the run's start; a long one (few splits,
    // where that walk would cover most of the list): every warp walking its own segment
    int32_t* sel_out = sa.sel_out;
    auto emit = [&](int p, int pos) {
      if (sel_out != nullptr) sel_out[grp * sa.k_max + pos] = p;
      s_phys[pos - pos0] = p;
    };
    uint64_t* wtot = reinterpret_cast<uint64_t*>(smem + C::OFF_WTOT);
    if (LONG && list.n >= 0)
      cta_compact_list<C::THREADS>(list, T, take_eq, wtot, pos0, pos0 + np, emit);
    else if (4 * np < cnt)
      cta_compact_window<C::THREADS>(K, T, take_eq, wtot, misc, pos0, pos0 + np, emit);
    else
      cta_compact<C::THREADS>(K, T, take_eq, wtot, pos0, pos0 + np, emit);
    __syncthreads();
    if (table_bulk) tab = reinterpret_cast<const int32_t*>(ring + KW);
    for (int i = tid; i < np; i += C::THREADS) resolve(i, s_phys[i]);
  } else {
    if (sa.scores != nullptr && cnt > 0 && cnt < n_pages) {   // group too long to select here
      if (tid == 0) flag(ctx, KV_DEVERR_BAD_SEL);
      np = 0;
    }
    for (int i = tid; i < np; i += C::THREADS)
      resolve(i, sel_idx != nullptr ? sel_idx[grp * sel_stride + pos0 + i] : pos0 + i);
    if (sa.scores != nullptr && s == 0 && sa.sel_out != nullptr)
      for (int i = tid; i < cnt; i += C::THREADS) sa.sel_out[grp * sa.k_max + i] = i;
    load_q_frags<D, G>(q, (long)b * Hq + g * G, qa0, qa2);
  }
  if (keys_bulk && !rows_waited &&                // the ring is reused for the pages next
      !mbar_wait_bounded(&bars[C::NSTAGE], 0u, ctx.wait_ns) && tid == 0)
    flag(ctx, KV_DEVERR_TIMEOUT);
  __syncthreads();

  WarpAcc<D> acc;
  acc.init();
  const bool ok = attend_run<D, G, C::NSTAGE, !LONG>(&tmK, &tmV, smem + C::OFF_STAGES, bars, 0u,
                                              s_phys, s_valid, np, g, Hkv, PS, qa0, qa2,
                                              qk_scale_log2, acc, ctx.wait_ns);
  const long out_row = ((long)b * Hq + g * G) * S + s;
  if (!ok) {
    if (tid == 0) flag(ctx, KV_DEVERR_TIMEOUT);
    for (int i = tid; i < G * D; i += C::THREADS) {
      const int hl = i / D, dd = i % D;
      part_acc[(out_row + (long)hl * S) * D + dd] = 0.f;
      if (dd == 0) {
        part_ml[(out_row + (long)hl * S) * 2 + 0] = -INFINITY;
        part_ml[(out_row + (long)hl * S) * 2 + 1] = 0.f;
      }
    }
  } else {
    float* scratch = reinterpret_cast<float*>(smem + C::OFF_STAGES);
    float* part = scratch + 4 * G * (D + 2);
    cta_partial<D, G>(acc, scratch, part);
    for (int i = tid; i < G * D; i += C::THREADS) {
      const int hl = i / D, dd = i % D;
      part_acc[(out_row + (long)hl * S) * D + dd] = part[hl * D + dd];
      if (dd == 0) {
        const float M = part[G * D + hl];
        part_ml[(out_row + (long)hl * S) * 2 + 0] = M == -INFINITY ? -INFINITY : M * kLn2;
        part_ml[(out_row + (long)hl * S) * 2 + 1] = part[G * D + G + hl];
      }
    }
  }
  if (sa.counters == nullptr) return;

  // ---- the group's last CTA merges its S partials (log-sum-exp) -------------------------
  __syncthreads();                                         // this CTA's partials are written
  if (tid == 0) {
    // one acquire-release atomic: the partials this CTA wrote (ordered before it by the
    // barrier above) are visible to whoever counts after it, and the others' to this CTA
    int done;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                 : "=r"(done) : "l"(&sa.counters[grp]) : "memory");
    misc[3] = (done == S - 1) ? 1u : 0u;
  }
  __syncthreads();                                         // orders every thread after it
  if (misc[3] == 0u) return;
  float* wts = reinterpret_cast<float*>(smem + C::OFF_STAGES);   // [G][S] weights, M[G],
  float* Ms = wts + G * S;                                        // L[G], l values [G][S]
  float* Ls = Ms + G;
  float* lv = Ls + G;
  const int warp = tid >> 5, lane = tid & 31;
  // The first splits' partial sums of this thread's first output columns do not depend on the
  // weights: their loads go out now and land while the weights are computed.
  constexpr int D4 = D / 4;
  constexpr int PB = 40;
  float4 pre[PB];
  if (tid < G * D4) {
    const int hl = tid / D4, d4 = tid - hl * D4;
    const float4* a = reinterpret_cast<const float4*>(part_acc + ((long)b * Hq + g * G + hl) * S * D) + d4;
#pragma unroll
    for (int u = 0; u < PB; ++u)
      pre[u] = u < S ? __ldcg(a + (long)u * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int hl = warp; hl < G; hl += C::THREADS / 32) {
    // the (m, l) pairs, two per lane in flight; M = max m by shuffles alone, then one
    // exponential per split and a plain sum (a short dependency chain)
    const float2* ml = reinterpret_cast<const float2*>(part_ml) + ((long)b * Hq + g * G + hl) * S;
    float M = -INFINITY;
    for (int x0 = lane; x0 < S; x0 += 64) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int x = x0 + 32 * u;
        if (x < S) {
          const float2 v = __ldcg(ml + x);
          wts[hl * S + x] = v.x;                          // m for now, the weight below
          lv[hl * S + x] = v.y;
          M = fmaxf(M, v.x);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    __syncwarp();
    float L = 0.f;
    for (int x = lane; x < S; x += 32) {
      const float m = wts[hl * S + x];
      const float w = (m == -INFINITY || M == -INFINITY) ? 0.f : expf(m - M);
      wts[hl * S + x] = w;
      L = fmaf(lv[hl * S + x], w, L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      Ms[hl] = M;
      Ls[hl] = L;
    }
  }
  __syncthreads();
  // out = sum_s w_s acc_s / L, four columns per thread, sixteen splits' loads in flight
  for (int o = tid; o < G * D4; o += C::THREADS) {
    const int hl = o / D4, d4 = o - hl * D4;
    const long row = (long)b * Hq + g * G + hl;
    const float4* a = reinterpret_cast<const float4*>(part_acc + row * S * D) + d4;
    const float* w = wts + hl * S;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    int x0 = 0;
    if (o == tid) {                                    // the prefetched first splits
#pragma unroll
      for (int u = 0; u < PB; ++u) {
        if (u < S) {
          const float ww = w[u];
          A.x = fmaf(pre[u].x, ww, A.x);
          A.y = fmaf(pre[u].y, ww, A.y);
          A.z = fmaf(pre[u].z, ww, A.z);
          A.w = fmaf(pre[u].w, ww, A.w);
        }
      }
      x0 = PB;
    }
    for (int x = x0; x < S; x += 16) {                 // no serial remainder: guarded lanes
      float4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u)
        v[u] = x + u < S ? __ldcg(a + (long)(x + u) * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        if (x + u < S) {
          const float ww = w[x + u];
          A.x = fmaf(v[u].x, ww, A.x);
          A.y = fmaf(v[u].y, ww, A.y);
          A.z = fmaf(v[u].z, ww, A.z);
          A.w = fmaf(v[u].w, ww, A.w);
        }
      }
    }
    const float M = Ms[hl], L = Ls[hl];
    float* op = sa.out + row * D + d4 * 4;
    const bool empty = M == -INFINITY;
    op[0] = empty ? 0.f : A.x / L;
    op[1] = empty ? 0.f : A.y / L;
    op[2] = empty ? 0.f : A.z / L;
    op[3] = empty ? 0.f : A.w / L;
    if (d4 == 0 && sa.lse != nullptr) sa.lse[row] = empty ? -INFINITY : M + logf(L);
  }
  if (tid == 0) sa.counters[grp] = 0;                      // ready for the next step
}

}  // namespace skv
