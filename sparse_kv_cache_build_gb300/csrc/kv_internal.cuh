// Internal device helpers and launcher declarations shared by the library's CUDA files.
// Not part of the public interface (include/sparsekv.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sparsekv.h"

namespace skv {

// ------------------------------------------------------------------------------------
// Limits of this build
// ------------------------------------------------------------------------------------
constexpr int kTileTokens = 64;        // tokens per pipeline stage of the attention kernel
constexpr int kWarpTokens = 16;        // tokens per warp per stage
constexpr int kMaxSplitPages = 2048;   // pages one split may cover (index list in smem)
constexpr int kSelectThreads = 1024;   // threads of the top-k block
constexpr int kSelectChunk = 8192;     // keys staged in shared memory per compaction pass

// Everything a kernel needs to report data faults without trapping.
struct DevCtx {
  int32_t* err;                 // per-device error word (KV_DEVERR_* bits)
  unsigned long long wait_ns;   // bound of every wait on an asynchronous copy
};

__device__ __forceinline__ void flag(const DevCtx& c, int32_t bits) { atomicOr(c.err, bits); }

// ------------------------------------------------------------------------------------
// Element access: bf16 is the upper half of an IEEE float, so widening is a shift.
// ------------------------------------------------------------------------------------
struct bf16_t { uint16_t bits; };

template <typename T> struct ElemTraits;
template <> struct ElemTraits<bf16_t> { static constexpr int bytes = 2; };
template <> struct ElemTraits<float>  { static constexpr int bytes = 4; };

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Widen one 16-byte chunk (8 bf16 or 4 fp32) to floats.
template <typename T> __device__ __forceinline__ void chunk_to_f32(uint4 v, float* f);
template <> __device__ __forceinline__ void chunk_to_f32<bf16_t>(uint4 v, float* f) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}
template <> __device__ __forceinline__ void chunk_to_f32<float>(uint4 v, float* f) {
  f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}

// Load `n` consecutive elements (n * bytes a multiple of 4) from shared or global memory.
// D += A * B, m16n8k16, bf16 inputs, f32 accumulators.
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <typename T> __device__ __forceinline__ float load_elem(const void* base, long i);
template <> __device__ __forceinline__ float load_elem<bf16_t>(const void* base, long i) {
  const uint16_t v = reinterpret_cast<const uint16_t*>(base)[i];
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}
template <> __device__ __forceinline__ float load_elem<float>(const void* base, long i) {
  return reinterpret_cast<const float*>(base)[i];
}

// ------------------------------------------------------------------------------------
// mbarrier + bulk asynchronous copy (global -> shared), with bounded waits.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count the current phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`, for at most `limit_ns` of the global timer.
// Returns false if the limit ran out first (the caller flags KV_DEVERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// One bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from global
// memory into this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// L2 policy for data read exactly once per step (K/V pages): evict first.
// Hint: bring the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel of the library lets the next kernel on the
// stream start launching as soon as all of its own blocks are running (pdl_trigger), and
// waits for the previous kernel to finish and flush (pdl_wait) before its first access to
// global memory, so only launch latency and on-chip set-up overlap. Both are no-ops when the
// kernel was launched without the programmatic-serialisation attribute.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kern` on `s` with the programmatic-serialisation attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// Small math helpers
// ------------------------------------------------------------------------------------
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Order-preserving key of a page score: the unsigned order of keys is the float order
// (-0 and +0 give one key; NaN is not a valid score).
__device__ __forceinline__ uint32_t score_order_key(float s) {
  const uint32_t u = __float_as_uint(s + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Pages kept of a group of n: keep[b] if given, else min(n, budget) if budget > 0, else n
// if ratio >= 1, else min(n, max(1, ceil(ratio * n - 1e-9))) in double; 0 when n == 0.
__device__ __forceinline__ int keep_rule(int n, const int32_t* keep, int b, double ratio,
                                         int budget) {
  if (n <= 0) return 0;
  if (keep != nullptr) {
    const int k = keep[b];
    return k < 0 ? 0 : (k > n ? n : k);
  }
  if (budget > 0) return budget < n ? budget : n;
  if (ratio >= 1.0) return n;
  int k = (int)ceil(ratio * (double)n - 1e-9);
  k = k < 1 ? 1 : k;
  return k < n ? k : n;
}

// Sequence length of b, clamped into [0, stride * page_size] (flags a bad length).
__device__ __forceinline__ int checked_len(const DevCtx& c, const kv_cache_desc& d, int b) {
  int len = d.seq_lens[b];
  const int cap = d.page_table_stride * d.page_size;
  if (len < 0 || len > cap) {
    flag(c, KV_DEVERR_BAD_LEN);
    len = len < 0 ? 0 : cap;
  }
  return len;
}

// ------------------------------------------------------------------------------------
// Launchers (one per kernel family; each returns cudaGetLastError()).
// ------------------------------------------------------------------------------------
// stats_exp == NULL: statistics in the cache's dtype; otherwise FP8 bytes in stats and one
// int8 exponent per (page, KV head) in stats_exp (fp8_stats.cuh). subset != NULL: only the
// mapped pages whose physical index is in subset[0, n_subset) (strictly ascending).
cudaError_t launch_page_stats(const kv_cache_desc& d, void* stats, int8_t* stats_exp,
                              const int32_t* subset, int n_subset, DevCtx ctx, cudaStream_t s);
// Entmax decoding (entmax.cu). Moments: zb/cz/vz [B][Hq][stride]. Selection: one block per
// group writes the kept pages ascending. Attention: logits [B][Hq][cap_slots] scratch, then
// out [B][Hq][D] and tau [B][Hq] (in z = logit/2 units).
cudaError_t launch_entmax_moments(const kv_cache_desc& d, int G, const void* q,
                                  const void* stats, float scale, float* zb, float* cz,
                                  float* vz, int stride, int sms, DevCtx ctx, cudaStream_t s);
cudaError_t launch_entmax_select(const int32_t* seq_lens, int page_size, int batch, int Hq,
                                 int Hkv, int table_stride, const float* zb, const float* cz,
                                 const float* vz, int stride, int k_max, int32_t* sel_idx,
                                 int32_t* sel_cnt, float* tau_hat, DevCtx ctx, cudaStream_t s);
// Entmax attention scratch: logits, candidate z and slot ([B][Hq][cap_slots] each), and per
// split the largest logit and the candidate count ([B][Hq][entmax_max_splits()] each).
struct EntmaxScratch {
  float* cand_z;        // [batch * Hq][slots]: candidates' z, per split from its first slot
  uint32_t* cand_row;   // same layout: the candidate's row in the V pool
  float* split_floor;   // [batch * Hq][kMaxEntSplits]: lower bounds on tau
  int* split_cnt;       // same layout: candidates per split
};
int entmax_max_splits();
cudaError_t launch_entmax_attn(const kv_cache_desc& d, int G, const void* q, float scale,
                               const int32_t* sel, const int32_t* cnt, int sel_stride, int S,
                               const EntmaxScratch& w, int cap_slots, float* out, float* tau,
                               DevCtx ctx, cudaStream_t s);
cudaError_t launch_score_pages(const kv_cache_desc& d, const void* q, int Hq,
                               const void* stats, const int8_t* stats_exp, float* scores,
                               int scores_stride, DevCtx ctx, cudaStream_t s);
// kv_score_pages and the group's top-k (keep ratio / budget) in one launch; counters
// [batch][Hkv] start at zero and are returned to zero. score_select_smem: dynamic shared
// bytes the launch needs for a table stride (the caller checks it against the device).
size_t score_select_smem(int page_table_stride);
cudaError_t launch_score_select(const kv_cache_desc& d, const void* q, int Hq,
                                const void* stats, const int8_t* stats_exp, float* scores,
                                int scores_stride, double keep_ratio, int budget, int k_max,
                                int32_t* counters, int32_t* sel_idx, int32_t* sel_cnt,
                                DevCtx ctx, cudaStream_t s);
cudaError_t launch_select_topk(const float* scores, int scores_stride, const int32_t* seq_lens,
                               int page_size, int batch, int Hkv, const int32_t* keep,
                               double keep_ratio, int budget_pages, int k_max, int sink,
                               int local, int32_t* sel_idx, int32_t* sel_cnt,
                               int page_table_stride, DevCtx ctx, cudaStream_t s);
cudaError_t launch_split_attn(const kv_cache_desc& d, const void* q, int Hq, float sm_scale,
                              const int32_t* sel_idx, const int32_t* sel_cnt, int sel_stride,
                              int num_splits, float* part_acc, float* part_ml, DevCtx ctx,
                              cudaStream_t s, int num_sms);
cudaError_t launch_merge(const float* part_acc, const float* part_ml, int batch, int Hq,
                         int num_splits, int D, float* out, float* lse, cudaStream_t s);
cudaError_t launch_dropped_mass(const kv_cache_desc& d, const void* q, int Hq,
                                float sm_scale, const int32_t* sel_idx,
                                const int32_t* sel_cnt, int sel_stride, int num_splits,
                                float* partials, float* delta, DevCtx ctx, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, DevCtx ctx, cudaStream_t s);
cudaError_t launch_append(const kv_cache_desc& d, const void* k_new, const void* v_new,
                          void* stats, DevCtx ctx, cudaStream_t s);

// The single-launch decode step (bf16): cluster size for this shape on this device
// (0 = use the four-kernel path), and its launcher.
int fused_cluster_size(const kv_cache_desc& d, int G, int num_sms);
cudaError_t launch_fused_step(const kv_cache_desc& d, int G, int CL, const void* q,
                              const void* stats, float sm_scale, double keep_ratio, int budget,
                              int k_max, int dense, int32_t* sel_out, int32_t* cnt_out,
                              float* out, float* lse, DevCtx ctx, cudaStream_t s);

// The 2-D TMA tensor map of a bf16 pool ([NP*Hkv*PS rows][D columns], boxes of 64 columns x
// PS rows, 128-byte swizzle) for the current device, from a small cache of encoded maps
// (thread-safe); false if it cannot be encoded.
bool pool_tensor_map(CUtensorMap* map, const void* pool, const kv_cache_desc& d);

// Dynamic shared memory bytes of the attention kernel for this shape (0 = unsupported).
size_t split_attn_smem_bytes(int dtype, int head_dim, int group_size);

}  // namespace skv
