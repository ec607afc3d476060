// Host side of the C interface declared in include/sparsekv.h: argument checks, the
// per-device error word, split-count choice, workspace carving and kernel launches.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <map>
#include <new>
#include <mutex>
#include <tuple>

#include "attn_impl.cuh"
#include "attn_mma.cuh"
#include "kv_internal.cuh"

namespace skv {
namespace {

// Device-side error word (one per device context). Kernels receive its device address.
__device__ int32_t g_kv_error_word = 0;

constexpr int kMaxDevices = 64;
constexpr int kDroppedSplits = 64;          // page ranges per group in the dropped-mass probe
// Longest group (pages) whose selection kv_decode_step leaves to the attention kernel's CTAs;
// longer groups select once, in the score launch. Measured with the bulk-copied rows, 11-bit
// digits and the one-wave score pass: 70.8 against 88.3 us a step at 8192 pages (128K
// context), 66.7 against 97.4 us at 16384 pages (1M context, page size 64).
constexpr int kInAttnSelectPages = 16384;
// Split count from which the step merges in a separate kernel (chained by programmatic
// dependent launch) rather than in the attention kernel's last CTA per group. Measured on
// this part: with 38 splits the separate merge saved 2.0 us at 32K and 128K and 5.1 us at 1M
// context; with one split per group (batched serving) it cost 2.0 us.
constexpr int kSeparateMergeMinSplits = 8;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int smem_per_sm = 0;
  int smem_optin = 0;          // largest dynamic shared memory one block may opt into
  int32_t* err = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
unsigned long long g_wait_ns = 2000000000ull;

kv_status device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kv_error_word) != cudaSuccess) return KV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return KV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&st.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                               dev) != cudaSuccess)
      return KV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               dev) != cudaSuccess)
      return KV_ERR_CUDA;
    st.err = static_cast<int32_t*>(p);
    st.ready = true;
  }
  *out = &st;
  return KV_OK;
}

kv_status ctx_for_call(DevCtx* ctx, DeviceState** st_out = nullptr) {
  DeviceState* st = nullptr;
  kv_status r = device_state(&st);
  if (r != KV_OK) return r;
  ctx->err = st->err;
  ctx->wait_ns = g_wait_ns;
  if (st_out) *st_out = st;
  return KV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kv_status check_desc(const kv_cache_desc* d) {
  if (d == nullptr || d->k_pool == nullptr || d->v_pool == nullptr ||
      d->page_table == nullptr || d->seq_lens == nullptr)
    return KV_ERR_INVALID_ARG;
  if (d->num_phys_pages <= 0 || d->num_kv_heads <= 0 || d->batch <= 0 ||
      d->page_table_stride <= 0 || d->batch > 65535 || d->num_kv_heads > 65535)
    return KV_ERR_INVALID_ARG;
  if (d->dtype != KV_BF16 && d->dtype != KV_FP32) return KV_ERR_UNSUPPORTED;
  if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64) return KV_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return KV_ERR_UNSUPPORTED;
  if ((long long)d->page_table_stride * d->page_size > INT32_MAX) return KV_ERR_INVALID_ARG;
  if (!aligned16(d->k_pool) || !aligned16(d->v_pool)) return KV_ERR_MISALIGNED;
  return KV_OK;
}

kv_status check_heads(const kv_cache_desc* d, const void* q, int32_t num_q_heads) {
  if (q == nullptr || num_q_heads <= 0 || num_q_heads % d->num_kv_heads != 0)
    return KV_ERR_INVALID_ARG;
  const int G = num_q_heads / d->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KV_ERR_UNSUPPORTED;
  if (!aligned16(q)) return KV_ERR_MISALIGNED;
  return KV_OK;
}

kv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KV_OK : KV_ERR_CUDA; }

size_t attn_smem(const kv_cache_desc* d, int G) {
  return d->dtype == KV_BF16 ? split_attn_smem_bf16(d->head_dim, G)
                             : split_attn_smem_fp32(d->head_dim, G);
}

int min_splits_for(int pages) { return (pages + kMaxSplitPages - 1) / kMaxSplitPages; }

constexpr long kBatchRunPages = 256;           // pages per split at most, batches of several

int auto_splits(const kv_cache_desc* d, int G, int pages_per_group, const DeviceState* st) {
  const size_t smem = attn_smem(d, G);
  int per_sm = smem > 0 ? (int)(st->smem_per_sm / (smem + 1024)) : 1;
  per_sm = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
  const long groups = (long)d->batch * d->num_kv_heads;
  const long target = (long)st->sms * per_sm;
  // as many splits as fill the resident CTA slots without starting a partial second wave
  // (rounding up had 256 groups run 512 CTAs in 1.7 waves: 176.3 against 167.1 us a step
  // for one CTA per group, each of which also repeats the group's selection)
  long S = target / groups;
  // with several sequences the lengths differ and the grid is sized by the longest: runs of
  // at most kBatchRunPages pages let a long sequence's CTAs spread over several waves while
  // the short ones finish (dense over the batched-serving shape: 1576 us a step at 2 splits,
  // 1158 us at 16)
  if (d->batch > 1) {
    const long by_len = (pages_per_group + kBatchRunPages - 1) / kBatchRunPages;
    if (S < by_len) S = by_len;
  }
  const int ppt = kTileTokens / d->page_size;
  const long cap = pages_per_group / (2 * ppt);            // at least two tiles per split
  if (S > cap) S = cap;
  if (S < 1) S = 1;
  const int lo = min_splits_for(pages_per_group);
  if (S < lo) S = lo;
  return (int)S;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

struct StepLayout {
  size_t scores, sel, cnt, acc, ml, ctr, ctr2, total;
};

// Row stride of the step's scores: page_table_stride rounded up to four floats, so that every
// row starts 16-byte aligned and can be copied into shared memory in bulk.
size_t step_scores_stride(const kv_cache_desc* d) {
  return ((size_t)d->page_table_stride + 3) & ~(size_t)3;
}

// The per-group counters come first, at offsets that depend only on batch * num_kv_heads,
// so calls of different shapes (sparse and dense, other k_max or split counts) on one
// workspace keep finding them where the previous call returned them to zero.
StepLayout step_layout(const kv_cache_desc* d, int Hq, int k_max, int S) {
  StepLayout L;
  const size_t groups = (size_t)d->batch * d->num_kv_heads;
  L.ctr = 0;
  L.ctr2 = L.ctr + round256(groups * sizeof(int32_t));
  L.scores = L.ctr2 + round256(groups * sizeof(int32_t));
  L.sel = L.scores + round256(groups * step_scores_stride(d) * sizeof(float));
  L.cnt = L.sel + round256(groups * (size_t)(k_max > 0 ? k_max : 1) * sizeof(int32_t));
  L.acc = L.cnt + round256(groups * sizeof(int32_t));
  L.ml = L.acc + round256((size_t)d->batch * Hq * S * d->head_dim * sizeof(float));
  L.total = L.ml + round256((size_t)d->batch * Hq * S * 2 * sizeof(float));
  return L;
}

// Cluster size of the one-launch step per (device, shape), decided once (outside any
// stream capture that follows) and reused.
int cached_cluster_size(const kv_cache_desc* d, int G, const DeviceState* st) {
  int dev = -1;
  cudaGetDevice(&dev);
  using Key = std::tuple<int, int, int, int, int, int, int, int, int>;
  static std::map<Key, int> memo;
  const Key key{dev, d->dtype, d->head_dim, G, d->page_size, d->batch, d->num_kv_heads,
                d->page_table_stride, d->num_phys_pages};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  const int CL = fused_cluster_size(*d, G, st->sms);
  std::lock_guard<std::mutex> lock(g_mu);
  memo[key] = CL;
  return CL;
}

bool is_dense(double keep_ratio, int budget_pages) {
  return budget_pages <= 0 && keep_ratio >= 1.0;
}

// The fused score + select launch fits this device for this table stride (its static
// shared memory is a few KB on top of the dynamic part).
bool score_select_fits(const kv_cache_desc* d, const DeviceState* st) {
  // + the kernel's static shared memory (histogram, q-side vector, scratch): under 16 KB
  return score_select_smem(d->page_table_stride) + 16 * 1024 <= (size_t)st->smem_optin;
}

__global__ void wait_selftest_kernel(unsigned long long limit_ns, DevCtx ctx) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);          // expects one arrival that never comes
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
  if (!ok && threadIdx.x == 0) flag(ctx, KV_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_split_attn(const kv_cache_desc& d, const void* q, int Hq, float sm_scale,
                              const int32_t* sel_idx, const int32_t* sel_cnt, int sel_stride,
                              int num_splits, float* part_acc, float* part_ml, DevCtx ctx,
                              cudaStream_t s, int /*num_sms*/) {
  const int G = Hq / d.num_kv_heads;
  return d.dtype == KV_BF16
             ? launch_split_attn_bf16(d, q, G, sm_scale, sel_idx, sel_cnt, sel_stride,
                                      num_splits, part_acc, part_ml, ctx, s)
             : launch_split_attn_fp32(d, q, G, sm_scale, sel_idx, sel_cnt, sel_stride,
                                      num_splits, part_acc, part_ml, ctx, s);
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, DevCtx ctx, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, ctx);
  return cudaGetLastError();
}

}  // namespace skv

using namespace skv;

extern "C" {

const char* kv_status_string(int32_t status) {
  switch (status) {
    case KV_OK: return "ok";
    case KV_ERR_INVALID_ARG: return "invalid argument";
    case KV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KV_ERR_CUDA: return "CUDA error";
    case KV_ERR_WORKSPACE: return "workspace missing or too small";
    case KV_ERR_BAD_INDEX: return "device detected a bad page, length, index or keep count";
    case KV_ERR_TIMEOUT: return "device wait timed out";
    case KV_ERR_MISALIGNED: return "buffer not 16-byte aligned";
    default: return "unknown status";
  }
}

int32_t kv_version(void) { return 101; }

kv_status kv_build_page_stats(const kv_cache_desc* cache, void* stats,
                              const int32_t* phys_pages, int32_t n_phys, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if (stats == nullptr) return KV_ERR_INVALID_ARG;
  if (phys_pages != nullptr && (n_phys < 0 || n_phys > cache->num_phys_pages))
    return KV_ERR_INVALID_ARG;
  if (!aligned16(stats)) return KV_ERR_MISALIGNED;
  if (phys_pages != nullptr && n_phys == 0) return KV_OK;     // nothing to rebuild
  DevCtx ctx;
  if ((r = ctx_for_call(&ctx)) != KV_OK) return r;
  return from_cuda(launch_page_stats(*cache, stats, nullptr, phys_pages, n_phys, ctx, stream));
}

kv_status kv_build_page_stats_fp8(const kv_cache_desc* cache, void* stats_fp8,
                                  int8_t* stats_exp, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if (stats_fp8 == nullptr || stats_exp == nullptr) return KV_ERR_INVALID_ARG;
  if (!aligned16(stats_fp8)) return KV_ERR_MISALIGNED;
  DevCtx ctx;
  if ((r = ctx_for_call(&ctx)) != KV_OK) return r;
  return from_cuda(launch_page_stats(*cache, stats_fp8, stats_exp, nullptr, 0, ctx, stream));
}

kv_status kv_append_token(const kv_cache_desc* cache, const void* k_new, const void* v_new,
                          void* stats, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if (k_new == nullptr || v_new == nullptr || stats == nullptr) return KV_ERR_INVALID_ARG;
  if (!aligned16(stats) || !aligned16(k_new) || !aligned16(v_new)) return KV_ERR_MISALIGNED;
  DevCtx ctx;
  if ((r = ctx_for_call(&ctx)) != KV_OK) return r;
  return from_cuda(launch_append(*cache, k_new, v_new, stats, ctx, stream));
}

kv_status kv_score_pages(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                         const void* stats, float* scores, int32_t scores_stride,
                         cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (stats == nullptr || scores == nullptr || scores_stride < cache->page_table_stride)
    return KV_ERR_INVALID_ARG;
  if (!aligned16(stats)) return KV_ERR_MISALIGNED;
  DevCtx ctx;
  if ((r = ctx_for_call(&ctx)) != KV_OK) return r;
  return from_cuda(launch_score_pages(*cache, q, num_q_heads, stats, nullptr, scores,
                                      scores_stride, ctx, stream));
}

kv_status kv_score_pages_fp8(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                             const void* stats_fp8, const int8_t* stats_exp, float* scores,
                             int32_t scores_stride, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (stats_fp8 == nullptr || stats_exp == nullptr || scores == nullptr ||
      scores_stride < cache->page_table_stride)
    return KV_ERR_INVALID_ARG;
  if (!aligned16(stats_fp8)) return KV_ERR_MISALIGNED;
  DevCtx ctx;
  if ((r = ctx_for_call(&ctx)) != KV_OK) return r;
  return from_cuda(launch_score_pages(*cache, q, num_q_heads, stats_fp8, stats_exp, scores,
                                      scores_stride, ctx, stream));
}

kv_status kv_select_topk(const float* scores, int32_t scores_stride, const int32_t* seq_lens,
                         int32_t page_size, int32_t batch, int32_t num_kv_heads,
                         const int32_t* keep, double keep_ratio, int32_t budget_pages,
                         int32_t k_max, int32_t* sel_idx, int32_t* sel_cnt,
                         cudaStream_t stream) {
  if (scores == nullptr || seq_lens == nullptr || sel_idx == nullptr || sel_cnt == nullptr)
    return KV_ERR_INVALID_ARG;
  if (scores_stride <= 0 || page_size <= 0 || batch <= 0 || batch > 65535 ||
      num_kv_heads <= 0 || num_kv_heads > 65535 || k_max <= 0)
    return KV_ERR_INVALID_ARG;
  if (keep == nullptr && budget_pages <= 0 && !(keep_ratio > 0.0)) return KV_ERR_INVALID_ARG;
  if ((long long)scores_stride * page_size > INT32_MAX) return KV_ERR_INVALID_ARG;
  DevCtx ctx;
  kv_status r = ctx_for_call(&ctx);
  if (r != KV_OK) return r;
  // The row stride bounds every sequence: a longer seq_len is flagged by the kernel.
  return from_cuda(launch_select_topk(scores, scores_stride, seq_lens, page_size, batch,
                                      num_kv_heads, keep, keep_ratio, budget_pages, k_max, 0, 0,
                                      sel_idx, sel_cnt, scores_stride, ctx, stream));
}

kv_status kv_select_structured(const float* scores, int32_t scores_stride,
                               const int32_t* seq_lens, int32_t page_size, int32_t batch,
                               int32_t num_kv_heads, const int32_t* keep, double keep_ratio,
                               int32_t budget_pages, int32_t sink_pages, int32_t local_pages,
                               int32_t k_max, int32_t* sel_idx, int32_t* sel_cnt,
                               cudaStream_t stream) {
  if (seq_lens == nullptr || sel_idx == nullptr || sel_cnt == nullptr) return KV_ERR_INVALID_ARG;
  if (scores_stride <= 0 || page_size <= 0 || batch <= 0 || batch > 65535 ||
      num_kv_heads <= 0 || num_kv_heads > 65535 || k_max <= 0 || sink_pages < 0 ||
      local_pages < 0)
    return KV_ERR_INVALID_ARG;
  if (keep == nullptr && budget_pages <= 0 && !(keep_ratio > 0.0) &&
      sink_pages + local_pages == 0)
    return KV_ERR_INVALID_ARG;
  if ((long long)scores_stride * page_size > INT32_MAX) return KV_ERR_INVALID_ARG;
  DevCtx ctx;
  kv_status r = ctx_for_call(&ctx);
  if (r != KV_OK) return r;
  return from_cuda(launch_select_topk(scores, scores_stride, seq_lens, page_size, batch,
                                      num_kv_heads, keep, keep_ratio, budget_pages, k_max,
                                      sink_pages, local_pages, sel_idx, sel_cnt, scores_stride,
                                      ctx, stream));
}

kv_status kv_sparse_decode_attn(const kv_cache_desc* cache, const void* q,
                                int32_t num_q_heads, float sm_scale, const int32_t* sel_idx,
                                const int32_t* sel_cnt, int32_t sel_stride,
                                int32_t num_splits, float* part_acc, float* part_ml,
                                cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (part_acc == nullptr || part_ml == nullptr || num_splits < 1 || num_splits > 65535 ||
      !(sm_scale > 0.f) || !isfinite(sm_scale))
    return KV_ERR_INVALID_ARG;
  if (sel_idx != nullptr && (sel_cnt == nullptr || sel_stride <= 0)) return KV_ERR_INVALID_ARG;
  const int bound = sel_idx != nullptr ? sel_stride : cache->page_table_stride;
  if (num_splits < min_splits_for(bound)) return KV_ERR_INVALID_ARG;
  DevCtx ctx;
  DeviceState* st = nullptr;
  if ((r = ctx_for_call(&ctx, &st)) != KV_OK) return r;
  return from_cuda(launch_split_attn(*cache, q, num_q_heads, sm_scale, sel_idx, sel_cnt,
                                     sel_stride, num_splits, part_acc, part_ml, ctx, stream,
                                     st->sms));
}

kv_status kv_score_select(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                          const void* stats, double keep_ratio, int32_t budget_pages,
                          int32_t k_max, float* scores, int32_t scores_stride,
                          int32_t* counters, int32_t* sel_idx, int32_t* sel_cnt,
                          cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (stats == nullptr || scores == nullptr || counters == nullptr || sel_idx == nullptr ||
      sel_cnt == nullptr || scores_stride < cache->page_table_stride || k_max <= 0 ||
      !(keep_ratio > 0.0 || budget_pages > 0))
    return KV_ERR_INVALID_ARG;
  if (!aligned16(stats)) return KV_ERR_MISALIGNED;
  DevCtx ctx;
  DeviceState* st = nullptr;
  if ((r = ctx_for_call(&ctx, &st)) != KV_OK) return r;
  if (!score_select_fits(cache, st)) return KV_ERR_UNSUPPORTED;
  return from_cuda(launch_score_select(*cache, q, num_q_heads, stats, nullptr, scores,
                                       scores_stride,
                                       keep_ratio, budget_pages, k_max, counters, sel_idx,
                                       sel_cnt, ctx, stream));
}

kv_status kv_decode_attn_merge(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                               float sm_scale, const int32_t* sel_idx, const int32_t* sel_cnt,
                               int32_t sel_stride, int32_t num_splits, float* part_acc,
                               float* part_ml, int32_t* counters, float* out, float* lse,
                               cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (cache->dtype != KV_BF16) return KV_ERR_UNSUPPORTED;
  if (part_acc == nullptr || part_ml == nullptr || counters == nullptr || out == nullptr ||
      num_splits < 1 || num_splits > 65535 || !(sm_scale > 0.f) || !isfinite(sm_scale))
    return KV_ERR_INVALID_ARG;
  if (sel_idx != nullptr && (sel_cnt == nullptr || sel_stride <= 0)) return KV_ERR_INVALID_ARG;
  if (!aligned16(part_acc) || (reinterpret_cast<uintptr_t>(part_ml) & 7u) != 0)
    return KV_ERR_MISALIGNED;
  const int G = num_q_heads / cache->num_kv_heads;
  int max_sel = 0, max_S = 0;
  step_attn_limits_bf16(cache->head_dim, G, &max_sel, &max_S);
  if (num_splits > max_S) return KV_ERR_UNSUPPORTED;
  if (num_splits < min_splits_for(sel_idx != nullptr ? sel_stride : cache->page_table_stride))
    return KV_ERR_INVALID_ARG;
  DevCtx ctx;
  if ((r = ctx_for_call(&ctx)) != KV_OK) return r;
  StepArgs sa{};
  sa.counters = counters;
  sa.out = out;
  sa.lse = lse;
  return from_cuda(launch_step_attn_bf16(*cache, q, G, sm_scale, sel_idx, sel_cnt, sel_stride,
                                         num_splits, part_acc, part_ml, ctx, stream, sa));
}

kv_status kv_select_decode_attn(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                float sm_scale, const float* scores, int32_t scores_stride,
                                double keep_ratio, int32_t budget_pages, int32_t k_max,
                                int32_t num_splits, float* part_acc, float* part_ml,
                                int32_t* counters, float* out, float* lse, int32_t* sel_idx,
                                int32_t* sel_cnt, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (cache->dtype != KV_BF16) return KV_ERR_UNSUPPORTED;
  if (part_acc == nullptr || part_ml == nullptr || (counters != nullptr && out == nullptr) ||
      num_splits < 1 || num_splits > 65535 || !(sm_scale > 0.f) || !isfinite(sm_scale))
    return KV_ERR_INVALID_ARG;
  if (!aligned16(part_acc) || (reinterpret_cast<uintptr_t>(part_ml) & 7u) != 0)
    return KV_ERR_MISALIGNED;
  const bool dense = scores == nullptr;
  if (!dense && (scores_stride < cache->page_table_stride || k_max <= 0 ||
                 !(keep_ratio > 0.0 || budget_pages > 0)))
    return KV_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  int max_sel = 0, max_S = 0;
  step_attn_limits_bf16(cache->head_dim, G, &max_sel, &max_S);
  if ((!dense && cache->page_table_stride > max_sel) || num_splits > max_S)
    return KV_ERR_UNSUPPORTED;
  if (num_splits < min_splits_for(dense ? cache->page_table_stride : k_max))
    return KV_ERR_INVALID_ARG;
  DevCtx ctx;
  if ((r = ctx_for_call(&ctx)) != KV_OK) return r;
  StepArgs sa{};
  sa.scores = scores;
  sa.scores_stride = scores_stride;
  sa.keep_ratio = keep_ratio;
  sa.budget = budget_pages;
  sa.k_max = dense ? 1 : k_max;
  sa.sel_out = dense ? nullptr : sel_idx;
  sa.cnt_out = dense ? nullptr : sel_cnt;
  sa.counters = counters;
  sa.out = out;
  sa.lse = lse;
  return from_cuda(launch_step_attn_bf16(*cache, q, G, sm_scale, nullptr, nullptr, 0,
                                         num_splits, part_acc, part_ml, ctx, stream, sa));
}

kv_status kv_merge_splits(const float* part_acc, const float* part_ml, int32_t batch,
                          int32_t num_q_heads, int32_t num_splits, int32_t head_dim,
                          float* out, float* lse, cudaStream_t stream) {
  if (part_acc == nullptr || part_ml == nullptr || out == nullptr) return KV_ERR_INVALID_ARG;
  if (batch <= 0 || num_q_heads <= 0 || num_splits < 1) return KV_ERR_INVALID_ARG;
  if ((long long)batch * num_q_heads > INT32_MAX) return KV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return KV_ERR_UNSUPPORTED;
  return from_cuda(
      launch_merge(part_acc, part_ml, batch, num_q_heads, num_splits, head_dim, out, lse, stream));
}

int32_t kv_auto_num_splits(const kv_cache_desc* cache, int32_t num_q_heads,
                           int32_t pages_per_group) {
  if (cache == nullptr || cache->num_kv_heads <= 0 || cache->batch <= 0 ||
      num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0 || pages_per_group < 0)
    return KV_ERR_INVALID_ARG;
  if (cache->page_size != 16 && cache->page_size != 32 && cache->page_size != 64)
    return KV_ERR_UNSUPPORTED;
  DeviceState* st = nullptr;
  kv_status r = device_state(&st);
  if (r != KV_OK) return r;
  return auto_splits(cache, num_q_heads / cache->num_kv_heads, pages_per_group, st);
}

size_t kv_dropped_mass_workspace_size(const kv_cache_desc* cache, int32_t num_q_heads) {
  if (cache == nullptr || cache->batch <= 0 || num_q_heads <= 0) return 0;
  return (size_t)cache->batch * num_q_heads * kDroppedSplits * 3 * sizeof(float);
}

kv_status kv_dropped_mass(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                          float sm_scale, const int32_t* sel_idx, const int32_t* sel_cnt,
                          int32_t sel_stride, float* delta, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (sel_idx == nullptr || sel_cnt == nullptr || sel_stride <= 0 || delta == nullptr ||
      !(sm_scale > 0.f) || !isfinite(sm_scale))
    return KV_ERR_INVALID_ARG;
  if ((long long)cache->page_table_stride > (long long)kDroppedSplits * 65536)
    return KV_ERR_UNSUPPORTED;
  if (workspace == nullptr ||
      workspace_bytes < kv_dropped_mass_workspace_size(cache, num_q_heads))
    return KV_ERR_WORKSPACE;
  DevCtx ctx;
  if ((r = ctx_for_call(&ctx)) != KV_OK) return r;
  return from_cuda(launch_dropped_mass(*cache, q, num_q_heads, sm_scale, sel_idx, sel_cnt,
                                       sel_stride, kDroppedSplits,
                                       static_cast<float*>(workspace), delta, ctx, stream));
}

size_t kv_decode_step_workspace_size(const kv_cache_desc* cache, int32_t num_q_heads,
                                     int32_t k_max, int32_t num_splits) {
  if (cache == nullptr || num_q_heads <= 0 || cache->num_kv_heads <= 0 || cache->batch <= 0 ||
      num_q_heads % cache->num_kv_heads != 0 || cache->head_dim <= 0 ||
      cache->page_table_stride <= 0 || k_max < 0)
    return 0;
  int S = num_splits;
  if (S <= 0) {
    DeviceState* st = nullptr;
    if (device_state(&st) != KV_OK) return 0;
    const int G = num_q_heads / cache->num_kv_heads;
    // the larger of the sparse and the dense split counts, so either mode fits
    const int s1 = auto_splits(cache, G, k_max > 0 ? k_max : 1, st);
    const int s2 = auto_splits(cache, G, cache->page_table_stride, st);
    S = s1 > s2 ? s1 : s2;
  }
  return step_layout(cache, num_q_heads, k_max, S).total;
}

}  // extern "C"

namespace {

// The kernels kv_decode_step launches for a shape (KV_PLAN_*), and its split count.
struct StepPlan {
  int plan = KV_PLAN_FOUR_KERNELS;
  int S = 1;
  int CL = 0;          // cluster size of the one-launch plan
};

kv_status plan_step(const kv_cache_desc* cache, int num_q_heads, double keep_ratio,
                    int budget_pages, int k_max, int num_splits, DeviceState* st,
                    StepPlan* out) {
  const bool dense = is_dense(keep_ratio, budget_pages);
  const int G = num_q_heads / cache->num_kv_heads;
  const int stride = cache->page_table_stride;
  StepPlan P;
  if (num_splits == KV_SPLITS_ONE_LAUNCH) {
    // one launch for the whole step when the shape allows it (bf16, one wave of clusters);
    // otherwise the plans below with the automatic split count
    P.CL = cached_cluster_size(cache, G, st);
    if (P.CL > 0) {
      P.plan = KV_PLAN_ONE_LAUNCH;
      P.S = P.CL;
      *out = P;
      return KV_OK;
    }
    num_splits = 0;
  }
  int S = num_splits;
  if (S <= 0) S = auto_splits(cache, G, dense ? stride : k_max, st);
  if (S < min_splits_for(dense ? stride : k_max)) return KV_ERR_INVALID_ARG;
  P.S = S;
  P.plan = dense ? KV_PLAN_DENSE_TWO_KERNELS : KV_PLAN_FOUR_KERNELS;
  if (cache->dtype == KV_BF16) {
    // Two launches at most, the merge in the attention kernel's last CTA per group. Short
    // groups: the scores, then an attention kernel whose CTAs each select their own run
    // (redoing a small top-k per CTA is cheaper than a kernel boundary). Long groups: the
    // scores with the top-k in each group's last score block, then attention over the list.
    // Dense: the attention kernel alone.
    int max_sel = 0, max_S = 0;
    step_attn_limits_bf16(cache->head_dim, G, &max_sel, &max_S);
    if (S <= max_S) {
      if (dense)
        P.plan = KV_PLAN_DENSE_ATTN_MERGE;
      else if (stride <= kInAttnSelectPages && stride <= max_sel)
        P.plan = KV_PLAN_SCORE_THEN_SELECT_ATTN;
      else if (score_select_fits(cache, st))
        P.plan = KV_PLAN_SCORE_SELECT_THEN_ATTN;
    }
    if (S >= kSeparateMergeMinSplits) {
      if (P.plan == KV_PLAN_DENSE_ATTN_MERGE) P.plan = KV_PLAN_DENSE_TWO_KERNELS;
      else if (P.plan == KV_PLAN_SCORE_THEN_SELECT_ATTN)
        P.plan = KV_PLAN_SCORE_THEN_SELECT_ATTN_THEN_MERGE;
      else if (P.plan == KV_PLAN_SCORE_SELECT_THEN_ATTN)
        P.plan = KV_PLAN_SCORE_SELECT_THEN_ATTN_THEN_MERGE;
    }
  }
  *out = P;
  return KV_OK;
}

}  // namespace

extern "C" {

int32_t kv_decode_step_plan(const kv_cache_desc* cache, int32_t num_q_heads, double keep_ratio,
                            int32_t budget_pages, int32_t k_max, int32_t num_splits,
                            int32_t* splits) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0) return KV_ERR_INVALID_ARG;
  const int G = num_q_heads / cache->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KV_ERR_UNSUPPORTED;
  if (!is_dense(keep_ratio, budget_pages) && (k_max <= 0 || !(keep_ratio > 0.0 || budget_pages > 0)))
    return KV_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  if ((r = device_state(&st)) != KV_OK) return r;
  StepPlan P;
  if ((r = plan_step(cache, num_q_heads, keep_ratio, budget_pages, k_max, num_splits, st, &P)) !=
      KV_OK)
    return r;
  if (splits != nullptr) *splits = P.S;
  return P.plan;
}

}  // extern "C"

namespace {

// kv_decode_step with the statistics in the cache's dtype (stats_exp == NULL) or as FP8
// bytes with per-row exponents.
kv_status decode_step_impl(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                           float sm_scale, const void* stats, const int8_t* stats_exp,
                           double keep_ratio, int32_t budget_pages, int32_t k_max,
                           int32_t num_splits, float* out, float* lse, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (out == nullptr || !(sm_scale > 0.f) || !isfinite(sm_scale)) return KV_ERR_INVALID_ARG;
  const bool dense = is_dense(keep_ratio, budget_pages);
  if (!dense && (stats == nullptr || k_max <= 0 || !(keep_ratio > 0.0 || budget_pages > 0)))
    return KV_ERR_INVALID_ARG;
  if (!dense && !aligned16(stats)) return KV_ERR_MISALIGNED;
  if (!dense && stats_exp != nullptr && num_splits == KV_SPLITS_ONE_LAUNCH)
    num_splits = 0;                        // the one-launch kernel reads cache-dtype stats
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return KV_ERR_WORKSPACE;
  DevCtx ctx;
  DeviceState* st = nullptr;
  if ((r = ctx_for_call(&ctx, &st)) != KV_OK) return r;
  StepPlan P;
  if ((r = plan_step(cache, num_q_heads, keep_ratio, budget_pages, k_max, num_splits, st, &P)) !=
      KV_OK)
    return r;
  const int G = num_q_heads / cache->num_kv_heads;
  const int stride = (int)step_scores_stride(cache);     // of the scores rows
  const StepLayout L = step_layout(cache, num_q_heads, dense ? 1 : k_max, P.S);
  if (workspace_bytes < L.total) return KV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  float* scores = reinterpret_cast<float*>(ws + L.scores);
  int32_t* sel = dense ? nullptr : reinterpret_cast<int32_t*>(ws + L.sel);
  int32_t* cnt = dense ? nullptr : reinterpret_cast<int32_t*>(ws + L.cnt);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  float* ml = reinterpret_cast<float*>(ws + L.ml);
  StepArgs sa{};
  sa.counters = reinterpret_cast<int32_t*>(ws + L.ctr2);
  sa.out = out;
  sa.lse = lse;
  cudaError_t e = cudaSuccess;
  switch (P.plan) {
    case KV_PLAN_ONE_LAUNCH:
      return from_cuda(launch_fused_step(*cache, G, P.CL, q, stats, sm_scale, keep_ratio,
                                         budget_pages, dense ? 1 : k_max, dense ? 1 : 0, sel,
                                         cnt, out, lse, ctx, stream));
    case KV_PLAN_DENSE_ATTN_MERGE:
      return from_cuda(launch_step_attn_bf16(*cache, q, G, sm_scale, nullptr, nullptr, 0, P.S,
                                             acc, ml, ctx, stream, sa));
    case KV_PLAN_SCORE_THEN_SELECT_ATTN:
      e = launch_score_pages(*cache, q, num_q_heads, stats, stats_exp, scores, stride, ctx,
                             stream);
      if (e != cudaSuccess) return KV_ERR_CUDA;
      sa.scores = scores;
      sa.scores_stride = stride;
      sa.keep_ratio = keep_ratio;
      sa.budget = budget_pages;
      sa.k_max = k_max;
      sa.sel_out = sel;
      sa.cnt_out = cnt;
      return from_cuda(launch_step_attn_bf16(*cache, q, G, sm_scale, nullptr, nullptr, 0, P.S,
                                             acc, ml, ctx, stream, sa));
    case KV_PLAN_SCORE_SELECT_THEN_ATTN:
      e = launch_score_select(*cache, q, num_q_heads, stats, stats_exp, scores, stride,
                              keep_ratio,
                              budget_pages, k_max, reinterpret_cast<int32_t*>(ws + L.ctr), sel,
                              cnt, ctx, stream);
      if (e != cudaSuccess) return KV_ERR_CUDA;
      return from_cuda(launch_step_attn_bf16(*cache, q, G, sm_scale, sel, cnt, k_max, P.S, acc,
                                             ml, ctx, stream, sa));
    case KV_PLAN_SCORE_THEN_SELECT_ATTN_THEN_MERGE:
      // as plan 1, but the attention kernel only writes the partials (no counters) and the
      // merge is a kernel of its own
      e = launch_score_pages(*cache, q, num_q_heads, stats, stats_exp, scores, stride, ctx,
                             stream);
      if (e != cudaSuccess) return KV_ERR_CUDA;
      sa.scores = scores;
      sa.scores_stride = stride;
      sa.keep_ratio = keep_ratio;
      sa.budget = budget_pages;
      sa.k_max = k_max;
      sa.sel_out = sel;
      sa.cnt_out = cnt;
      sa.counters = nullptr;
      e = launch_step_attn_bf16(*cache, q, G, sm_scale, nullptr, nullptr, 0, P.S, acc, ml, ctx,
                                stream, sa);
      if (e != cudaSuccess) return KV_ERR_CUDA;
      return from_cuda(launch_merge(acc, ml, cache->batch, num_q_heads, P.S, cache->head_dim,
                                    out, lse, stream));
    case KV_PLAN_SCORE_SELECT_THEN_ATTN_THEN_MERGE:
      e = launch_score_select(*cache, q, num_q_heads, stats, stats_exp, scores, stride,
                              keep_ratio, budget_pages, k_max,
                              reinterpret_cast<int32_t*>(ws + L.ctr), sel, cnt, ctx, stream);
      if (e != cudaSuccess) return KV_ERR_CUDA;
      e = launch_split_attn(*cache, q, num_q_heads, sm_scale, sel, cnt, k_max, P.S, acc, ml, ctx,
                            stream, st->sms);
      if (e != cudaSuccess) return KV_ERR_CUDA;
      return from_cuda(launch_merge(acc, ml, cache->batch, num_q_heads, P.S, cache->head_dim,
                                    out, lse, stream));
    default:
      break;
  }
  // four kernels (sparse) or two (dense)
  if (!dense) {
    e = launch_score_pages(*cache, q, num_q_heads, stats, stats_exp, scores, stride, ctx,
                           stream);
    if (e != cudaSuccess) return KV_ERR_CUDA;
    e = launch_select_topk(scores, stride, cache->seq_lens, cache->page_size, cache->batch,
                           cache->num_kv_heads, nullptr, keep_ratio, budget_pages, k_max, 0, 0,
                           sel, cnt, cache->page_table_stride, ctx, stream);
    if (e != cudaSuccess) return KV_ERR_CUDA;
  }
  e = launch_split_attn(*cache, q, num_q_heads, sm_scale, sel, cnt, dense ? 0 : k_max, P.S, acc,
                        ml, ctx, stream, st->sms);
  if (e != cudaSuccess) return KV_ERR_CUDA;
  return from_cuda(
      launch_merge(acc, ml, cache->batch, num_q_heads, P.S, cache->head_dim, out, lse, stream));
}

}  // namespace

extern "C" {

kv_status kv_decode_step(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                         float sm_scale, const void* stats, double keep_ratio,
                         int32_t budget_pages, int32_t k_max, int32_t num_splits,
                         float* out, float* lse, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
  return decode_step_impl(cache, q, num_q_heads, sm_scale, stats, nullptr, keep_ratio,
                          budget_pages, k_max, num_splits, out, lse, workspace, workspace_bytes,
                          stream);
}

// ----------------------------------------------------------------- captured decode step

struct kv_step_graph {
  cudaGraphExec_t exec = nullptr;
};

}  // extern "C"

namespace {

// The device's address of a page-locked host buffer it can read and write in place (unified
// addressing), or nullptr (then the buffer is reached by copies).
void* mapped_device_ptr(const void* host) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();                          // not a CUDA pointer: clear the error
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace

extern "C" {

kv_status kv_decode_step_graph_create(const kv_cache_desc* cache, const void* q,
                                      int32_t num_q_heads, float sm_scale, const void* stats,
                                      double keep_ratio, int32_t budget_pages, int32_t k_max,
                                      int32_t num_splits, float* out, float* lse,
                                      void* workspace, size_t workspace_bytes,
                                      const void* q_host, float* out_host,
                                      kv_step_graph** graph) {
  if (graph == nullptr) return KV_ERR_INVALID_ARG;
  *graph = nullptr;
  if (cache == nullptr || cache->batch <= 0 || num_q_heads <= 0 || cache->head_dim <= 0)
    return KV_ERR_INVALID_ARG;
  const size_t elems = (size_t)cache->batch * num_q_heads * cache->head_dim;
  const size_t q_bytes = elems * (cache->dtype == KV_BF16 ? 2 : 4);
  // host buffers the device addresses in place are read and written by the kernels over the
  // host link (no copy node); others are copied in and out around the step
  const void* q_in = q_host != nullptr ? mapped_device_ptr(q_host) : nullptr;
  float* out_to = out_host != nullptr ? static_cast<float*>(mapped_device_ptr(out_host)) : nullptr;
  const void* q_step = q_in != nullptr ? q_in : q;
  float* out_step = out_to != nullptr ? out_to : out;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return KV_ERR_CUDA;
  // one uncaptured call first: it checks the arguments and does every first-use set-up
  // (device state, kernel attributes, tensor maps) outside the capture
  kv_status r = kv_decode_step(cache, q_step, num_q_heads, sm_scale, stats, keep_ratio,
                               budget_pages, k_max, num_splits, out_step, lse, workspace,
                               workspace_bytes, s);
  if (r == KV_OK && cudaStreamSynchronize(s) != cudaSuccess) r = KV_ERR_CUDA;
  cudaGraph_t g = nullptr;
  if (r == KV_OK) {
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      r = KV_ERR_CUDA;
    } else {
      if (q_host != nullptr && q_in == nullptr &&
          cudaMemcpyAsync(const_cast<void*>(q), q_host, q_bytes, cudaMemcpyHostToDevice, s) !=
              cudaSuccess)
        r = KV_ERR_CUDA;
      if (r == KV_OK)
        r = kv_decode_step(cache, q_step, num_q_heads, sm_scale, stats, keep_ratio,
                           budget_pages, k_max, num_splits, out_step, lse, workspace,
                           workspace_bytes, s);
      if (r == KV_OK && out_host != nullptr && out_to == nullptr &&
          cudaMemcpyAsync(out_host, out, elems * sizeof(float), cudaMemcpyDeviceToHost, s) !=
              cudaSuccess)
        r = KV_ERR_CUDA;
      const cudaError_t e = cudaStreamEndCapture(s, &g);
      if (r == KV_OK && e != cudaSuccess) r = KV_ERR_CUDA;
    }
  }
  kv_step_graph* h = nullptr;
  if (r == KV_OK) {
    h = new (std::nothrow) kv_step_graph;
    if (h == nullptr) r = KV_ERR_CUDA;
    else if (cudaGraphInstantiate(&h->exec, g, 0) != cudaSuccess) r = KV_ERR_CUDA;
  }
  if (g != nullptr) cudaGraphDestroy(g);
  cudaStreamDestroy(s);
  if (r != KV_OK) {
    delete h;
    return r;
  }
  *graph = h;
  return KV_OK;
}

kv_status kv_decode_step_graph_launch(kv_step_graph* graph, cudaStream_t stream) {
  if (graph == nullptr || graph->exec == nullptr) return KV_ERR_INVALID_ARG;
  return from_cuda(cudaGraphLaunch(graph->exec, stream));
}

kv_status kv_decode_step_graph_destroy(kv_step_graph* graph) {
  if (graph == nullptr) return KV_OK;
  const cudaError_t e = graph->exec != nullptr ? cudaGraphExecDestroy(graph->exec) : cudaSuccess;
  delete graph;
  return from_cuda(e);
}

kv_status kv_decode_step_fp8(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                             float sm_scale, const void* stats_fp8, const int8_t* stats_exp,
                             double keep_ratio, int32_t budget_pages, int32_t k_max,
                             int32_t num_splits, float* out, float* lse, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  if (!is_dense(keep_ratio, budget_pages) && stats_exp == nullptr) return KV_ERR_INVALID_ARG;
  return decode_step_impl(cache, q, num_q_heads, sm_scale, stats_fp8, stats_exp, keep_ratio,
                          budget_pages, k_max, num_splits, out, lse, workspace, workspace_bytes,
                          stream);
}

// ------------------------------------------------------------------------- entmax (f4)

kv_status kv_entmax_page_moments(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                 const void* stats, float sm_scale, float* zb, float* cz,
                                 float* vz, int32_t stride, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (stats == nullptr || zb == nullptr || cz == nullptr || vz == nullptr ||
      stride < cache->page_table_stride || !(sm_scale > 0.f) || !isfinite(sm_scale))
    return KV_ERR_INVALID_ARG;
  if (!aligned16(stats)) return KV_ERR_MISALIGNED;
  DevCtx ctx;
  DeviceState* st = nullptr;
  if ((r = ctx_for_call(&ctx, &st)) != KV_OK) return r;
  return from_cuda(launch_entmax_moments(*cache, num_q_heads / cache->num_kv_heads, q, stats,
                                         sm_scale, zb, cz, vz, stride, st->sms, ctx, stream));
}

kv_status kv_entmax_select(const float* zb, const float* cz, const float* vz, int32_t stride,
                           const int32_t* seq_lens, int32_t page_size, int32_t batch,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t k_max,
                           int32_t* sel_idx, int32_t* sel_cnt, float* tau_hat,
                           cudaStream_t stream) {
  if (zb == nullptr || cz == nullptr || vz == nullptr || seq_lens == nullptr ||
      sel_idx == nullptr || sel_cnt == nullptr)
    return KV_ERR_INVALID_ARG;
  if (stride <= 0 || page_size <= 0 || batch <= 0 || batch > 65535 || num_kv_heads <= 0 ||
      num_kv_heads > 65535 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || k_max <= 0)
    return KV_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > 8) return KV_ERR_UNSUPPORTED;
  if ((long long)stride * page_size > INT32_MAX) return KV_ERR_INVALID_ARG;
  DevCtx ctx;
  kv_status r = ctx_for_call(&ctx);
  if (r != KV_OK) return r;
  return from_cuda(launch_entmax_select(seq_lens, page_size, batch, num_q_heads, num_kv_heads,
                                        stride, zb, cz, vz, stride, k_max, sel_idx, sel_cnt,
                                        tau_hat, ctx, stream));
}

size_t kv_entmax_attn_workspace_size(const kv_cache_desc* cache, int32_t num_q_heads,
                                     int32_t sel_stride) {
  if (cache == nullptr || cache->batch <= 0 || num_q_heads <= 0 || cache->page_size <= 0)
    return 0;
  const long long pages = sel_stride > 0 ? sel_stride : cache->page_table_stride;
  const size_t slots = (size_t)cache->batch * num_q_heads * pages * cache->page_size;
  const size_t splits = (size_t)cache->batch * num_q_heads * entmax_max_splits();
  return 2 * round256(slots * 4) + 2 * round256(splits * 4);
}

}  // extern "C"

namespace {

// The candidate lists hold a token's V-pool row as 32 bits.
bool entmax_rows_fit(const kv_cache_desc* cache) {
  return (long long)cache->num_phys_pages * cache->num_kv_heads * cache->page_size <= UINT32_MAX;
}

int entmax_splits(const kv_cache_desc* cache, int pages, const DeviceState* st) {
  const long groups = (long)cache->batch * cache->num_kv_heads;
  long S = (4L * st->sms + groups - 1) / groups;
  const long cap = pages / 4 > 1 ? pages / 4 : 1;
  if (S > cap) S = cap;
  if (S > entmax_max_splits()) S = entmax_max_splits();
  return S < 1 ? 1 : (int)S;
}

// Carves the entmax attention scratch (kv_entmax_attn_workspace_size's layout).
EntmaxScratch entmax_scratch(void* base, const kv_cache_desc* cache, int Hq, int pages) {
  const size_t slots = (size_t)cache->batch * Hq * pages * cache->page_size;
  const size_t splits = (size_t)cache->batch * Hq * entmax_max_splits();
  char* p = static_cast<char*>(base);
  EntmaxScratch w;
  w.cand_z = reinterpret_cast<float*>(p);
  w.cand_row = reinterpret_cast<uint32_t*>(p + round256(slots * 4));
  w.split_floor = reinterpret_cast<float*>(p + 2 * round256(slots * 4));
  w.split_cnt = reinterpret_cast<int*>(p + 2 * round256(slots * 4) + round256(splits * 4));
  return w;
}

}  // namespace

extern "C" {

kv_status kv_entmax_decode_attn(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                float sm_scale, const int32_t* sel_idx, const int32_t* sel_cnt,
                                int32_t sel_stride, float* out, float* tau, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (!entmax_rows_fit(cache)) return KV_ERR_UNSUPPORTED;
  if (out == nullptr || !(sm_scale > 0.f) || !isfinite(sm_scale)) return KV_ERR_INVALID_ARG;
  if (sel_idx != nullptr && (sel_cnt == nullptr || sel_stride <= 0)) return KV_ERR_INVALID_ARG;
  const int stride = sel_idx != nullptr ? sel_stride : cache->page_table_stride;
  if ((long long)stride * cache->page_size > INT32_MAX) return KV_ERR_INVALID_ARG;
  if (workspace == nullptr ||
      workspace_bytes < kv_entmax_attn_workspace_size(cache, num_q_heads,
                                                      sel_idx != nullptr ? sel_stride : 0))
    return KV_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KV_ERR_MISALIGNED;
  DevCtx ctx;
  DeviceState* st = nullptr;
  if ((r = ctx_for_call(&ctx, &st)) != KV_OK) return r;
  return from_cuda(launch_entmax_attn(*cache, num_q_heads / cache->num_kv_heads, q, sm_scale,
                                      sel_idx, sel_cnt, sel_idx != nullptr ? sel_stride : 0,
                                      entmax_splits(cache, stride, st),
                                      entmax_scratch(workspace, cache, num_q_heads, stride),
                                      stride * cache->page_size, out, tau, ctx, stream));
}

size_t kv_entmax_decode_step_workspace_size(const kv_cache_desc* cache, int32_t num_q_heads,
                                            int32_t k_max) {
  if (cache == nullptr || cache->batch <= 0 || num_q_heads <= 0 || cache->num_kv_heads <= 0 ||
      cache->page_table_stride <= 0 || k_max <= 0)
    return 0;
  const size_t B = cache->batch, Hq = num_q_heads, Hkv = cache->num_kv_heads;
  return 3 * round256(B * Hq * cache->page_table_stride * sizeof(float)) +
         round256(B * Hkv * k_max * sizeof(int32_t)) + round256(B * Hkv * sizeof(int32_t)) +
         kv_entmax_attn_workspace_size(cache, num_q_heads, k_max);
}

kv_status kv_entmax_decode_step(const kv_cache_desc* cache, const void* q, int32_t num_q_heads,
                                float sm_scale, const void* stats, int32_t k_max, float* out,
                                float* tau, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  kv_status r = check_desc(cache);
  if (r != KV_OK) return r;
  if ((r = check_heads(cache, q, num_q_heads)) != KV_OK) return r;
  if (!entmax_rows_fit(cache)) return KV_ERR_UNSUPPORTED;
  if (stats == nullptr || out == nullptr || k_max <= 0 || !(sm_scale > 0.f) ||
      !isfinite(sm_scale))
    return KV_ERR_INVALID_ARG;
  if (!aligned16(stats)) return KV_ERR_MISALIGNED;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < kv_entmax_decode_step_workspace_size(cache, num_q_heads, k_max))
    return KV_ERR_WORKSPACE;
  DevCtx ctx;
  DeviceState* st = nullptr;
  if ((r = ctx_for_call(&ctx, &st)) != KV_OK) return r;
  const size_t B = cache->batch, Hq = num_q_heads, Hkv = cache->num_kv_heads;
  const int stride = cache->page_table_stride;
  const size_t mom = round256(B * Hq * stride * sizeof(float));
  char* ws = static_cast<char*>(workspace);
  float* zb = reinterpret_cast<float*>(ws);
  float* cz = reinterpret_cast<float*>(ws + mom);
  float* vz = reinterpret_cast<float*>(ws + 2 * mom);
  int32_t* sel = reinterpret_cast<int32_t*>(ws + 3 * mom);
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + 3 * mom + round256(B * Hkv * k_max * 4));
  void* scratch = ws + 3 * mom + round256(B * Hkv * k_max * 4) + round256(B * Hkv * 4);
  const int G = num_q_heads / cache->num_kv_heads;
  cudaError_t e = launch_entmax_moments(*cache, G, q, stats, sm_scale, zb, cz, vz, stride,
                                        st->sms, ctx, stream);
  if (e != cudaSuccess) return KV_ERR_CUDA;
  e = launch_entmax_select(cache->seq_lens, cache->page_size, cache->batch, num_q_heads,
                           cache->num_kv_heads, stride, zb, cz, vz, stride, k_max, sel, cnt,
                           nullptr, ctx, stream);
  if (e != cudaSuccess) return KV_ERR_CUDA;
  return from_cuda(launch_entmax_attn(*cache, G, q, sm_scale, sel, cnt, k_max,
                                      entmax_splits(cache, k_max, st),
                                      entmax_scratch(scratch, cache, num_q_heads, k_max),
                                      k_max * cache->page_size, out, tau, ctx, stream));
}

size_t kv_workspace_size(int32_t op, const kv_cache_desc* cache, int32_t num_q_heads,
                         int32_t k_max, int32_t num_splits) {
  switch (op) {
    case KV_OP_DECODE_STEP:
      return kv_decode_step_workspace_size(cache, num_q_heads, k_max, num_splits);
    case KV_OP_DROPPED_MASS:
      return kv_dropped_mass_workspace_size(cache, num_q_heads);
    case KV_OP_ENTMAX_DECODE_ATTN:
      return kv_entmax_attn_workspace_size(cache, num_q_heads, k_max);
    case KV_OP_ENTMAX_DECODE_STEP:
      return kv_entmax_decode_step_workspace_size(cache, num_q_heads, k_max);
    default:
      return 0;
  }
}

kv_status kv_check_device_errors(cudaStream_t stream, int32_t* flags) {
  DeviceState* st = nullptr;
  kv_status r = device_state(&st);
  if (r != KV_OK) return r;
  int32_t h = 0;
  const int32_t zero = 0;
  if (cudaMemcpyAsync(&h, st->err, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return KV_ERR_CUDA;
  if (cudaMemcpyAsync(st->err, &zero, sizeof(zero), cudaMemcpyHostToDevice, stream) !=
      cudaSuccess)
    return KV_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KV_ERR_CUDA;
  if (flags != nullptr) *flags = h;
  if (h == 0) return KV_OK;
  return (h & KV_DEVERR_TIMEOUT) ? KV_ERR_TIMEOUT : KV_ERR_BAD_INDEX;
}

kv_status kv_set_wait_limit_ns(uint64_t limit_ns) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_wait_ns = (unsigned long long)limit_ns;
  return KV_OK;
}

kv_status kv_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  DevCtx ctx;
  kv_status r = ctx_for_call(&ctx);
  if (r != KV_OK) return r;
  return from_cuda(launch_wait_selftest((unsigned long long)limit_ns, ctx, stream));
}

}  // extern "C"
