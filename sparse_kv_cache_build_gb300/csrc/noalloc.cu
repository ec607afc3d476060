// kv_decode_step_static: the decode step of kv_decode_step, on a scratch buffer that lives
// in the library itself instead of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory on the decode path -- a plain C
// or plugin host with no device allocator of its own, or a serving loop that must not call
// cudaMalloc per token (it can synchronise the device, or fail under memory pressure, in the
// middle of a step). They still pass inputs and outputs; only the scratch moves here.
//
// The scratch is one file-scope __device__ array of KV_STATIC_SCRATCH_BYTES (8 MiB). Every
// GPU that loads the library holds it until the process exits. In host code the array's name
// is only a host-side stand-in, never a device address, so the first call on each device
// looks the address up with cudaGetSymbolAddress (with that device current) and keeps it.
// CUDA loads this file's module lazily, so that first lookup is also when the module is
// loaded and the array reserved on the device (it can fail under memory pressure, or
// synchronise): the first call belongs at start-up, before any stream capture. All calls
// share the one array and it keeps the previous call's contents: calls that overlap on the
// GPU (other streams, other host threads) race on it and must be serialised by the caller.
// Nothing in it needs to start at zero -- every call writes each scratch byte before reading
// it.
//
// The step runs the four public calls (score, select, split-K attention, merge) on
// sub-buffers carved from the array like kv_decode_step's workspace, without its per-group
// counters, so no value has to survive from one call to the next; the limit checked is this
// layout's size. num_splits <= 0 takes kv_auto_num_splits' count. The selection matches
// kv_decode_step's bit for bit and the outputs match up to float32 rounding of the merge
// (kv_decode_step merges inside its attention kernel for bf16 caches).
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "sparsekv.h"

namespace {

static __device__ __align__(256) unsigned char g_kv_static_scratch[KV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDev] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
kv_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return KV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_kv_static_scratch) != cudaSuccess || ptr == nullptr)
      return KV_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return KV_OK;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" kv_status kv_decode_step_static(const kv_cache_desc* cache, const void* q,
                                           int32_t num_q_heads, float sm_scale,
                                           const void* stats, double keep_ratio,
                                           int32_t budget_pages, int32_t k_max,
                                           int32_t num_splits, float* out, float* lse,
                                           cudaStream_t stream) {
  if (cache == nullptr || q == nullptr || out == nullptr || num_q_heads <= 0 ||
      cache->num_kv_heads <= 0 || cache->batch <= 0 || cache->page_table_stride <= 0 ||
      cache->head_dim <= 0 || num_q_heads % cache->num_kv_heads != 0)
    return KV_ERR_INVALID_ARG;
  const bool dense = budget_pages <= 0 && keep_ratio >= 1.0;
  if (!dense && (stats == nullptr || k_max <= 0 || !(keep_ratio > 0.0 || budget_pages > 0)))
    return KV_ERR_INVALID_ARG;
  int S = num_splits;
  if (S <= 0) {
    S = kv_auto_num_splits(cache, num_q_heads, dense ? cache->page_table_stride : k_max);
    if (S < 0) return (kv_status)S;
  }
  // carved like kv_decode_step's workspace, less its per-group counters
  const size_t groups = (size_t)cache->batch * cache->num_kv_heads;
  const size_t off_sel = up256(groups * cache->page_table_stride * sizeof(float));
  const size_t off_cnt = off_sel + up256(groups * (size_t)(dense ? 1 : k_max) * sizeof(int32_t));
  const size_t off_acc = off_cnt + up256(groups * sizeof(int32_t));
  const size_t off_ml =
      off_acc + up256((size_t)cache->batch * num_q_heads * S * cache->head_dim * sizeof(float));
  const size_t total = off_ml + up256((size_t)cache->batch * num_q_heads * S * 2 * sizeof(float));
  if (total > (size_t)KV_STATIC_SCRATCH_BYTES) return KV_ERR_WORKSPACE;   // above the limit

  void* base = nullptr;
  kv_status r = scratch_address(&base);
  if (r != KV_OK) return r;
  char* ws = static_cast<char*>(base);
  float* scores = reinterpret_cast<float*>(ws);
  int32_t* sel = reinterpret_cast<int32_t*>(ws + off_sel);
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + off_cnt);
  float* acc = reinterpret_cast<float*>(ws + off_acc);
  float* ml = reinterpret_cast<float*>(ws + off_ml);
  if (!dense) {
    r = kv_score_pages(cache, q, num_q_heads, stats, scores, cache->page_table_stride, stream);
    if (r != KV_OK) return r;
    r = kv_select_topk(scores, cache->page_table_stride, cache->seq_lens, cache->page_size,
                       cache->batch, cache->num_kv_heads, nullptr, keep_ratio, budget_pages,
                       k_max, sel, cnt, stream);
    if (r != KV_OK) return r;
  }
  r = kv_sparse_decode_attn(cache, q, num_q_heads, sm_scale, dense ? nullptr : sel,
                            dense ? nullptr : cnt, dense ? 0 : k_max, S, acc, ml, stream);
  if (r != KV_OK) return r;
  return kv_merge_splits(acc, ml, cache->batch, num_q_heads, S, cache->head_dim, out, lse,
                         stream);
}
