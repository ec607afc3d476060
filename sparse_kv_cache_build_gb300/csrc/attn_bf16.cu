// Split-K decode attention for bf16 caches: the tensor-core kernel of attn_mma.cuh, fed by
// TMA tensor copies. This file builds the two tensor maps (K and V pools seen as 2-D
// [NP*Hkv*PS rows][D columns] bf16 arrays, boxes of 64 columns x PS rows, 128-byte swizzle),
// keeps the maps of recently used pools so that a launch does not re-encode them, and
// launches the kernel.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "attn_impl.cuh"
#include "attn_mma.cuh"

namespace skv {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_pool_map(CUtensorMap* map, const void* pool, const kv_cache_desc& d) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
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

// Encoded maps of recently used pools: a map depends only on the pool's address and shape,
// so a decode loop over one cache encodes its two maps once instead of on every launch.
struct MapEntry {
  bool used = false;
  int device = -1;
  const void* pool = nullptr;
  int head_dim = 0, page_size = 0;
  long long rows = 0;
  CUtensorMap map;
};
constexpr int kMapCacheEntries = 32;
std::mutex g_map_mu;
MapEntry g_maps[kMapCacheEntries];
int g_map_next = 0;

}  // namespace

bool pool_tensor_map(CUtensorMap* map, const void* pool, const kv_cache_desc& d) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const long long rows = (long long)d.num_phys_pages * d.num_kv_heads * d.page_size;
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (const MapEntry& e : g_maps) {
      if (e.used && e.device == dev && e.pool == pool && e.head_dim == d.head_dim &&
          e.page_size == d.page_size && e.rows == rows) {
        *map = e.map;
        return true;
      }
    }
  }
  CUtensorMap m;
  if (!encode_pool_map(&m, pool, d)) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry& e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCacheEntries;
  e.used = true;
  e.device = dev;
  e.pool = pool;
  e.head_dim = d.head_dim;
  e.page_size = d.page_size;
  e.rows = rows;
  e.map = m;
  *map = m;
  return true;
}

namespace {

template <int D, int G>
cudaError_t launch_mma(const kv_cache_desc& d, const CUtensorMap& mk, const CUtensorMap& mv,
                       const void* q, float sm_scale, const int32_t* sel_idx,
                       const int32_t* sel_cnt, int sel_stride, int S, float* part_acc,
                       float* part_ml, DevCtx ctx, cudaStream_t st, const StepArgs& sa) {
  using C = MmaCfg<D, G>;
  // the filtering instantiation only where the in-kernel selection can use it: long tables
  // keeping at most a sixteenth of their pages (cta_threshold)
  const bool is_long = sa.scores != nullptr &&
                       d.page_table_stride >= topk_detail::kPrefilterMinPages &&
                       16L * sa.k_max <= (long)d.page_table_stride;
  auto kern = is_long ? split_attn_mma_kernel<D, G, true> : split_attn_mma_kernel<D, G, false>;
  // set once per device and instantiation; atomic so that concurrent first calls from several
  // host threads are well defined (both may set the attribute, which is idempotent)
  static std::atomic<int> attr_set_for_device[2][64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 &&
      !attr_set_for_device[is_long][dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set_for_device[is_long][dev].store(1, std::memory_order_release);
  }
  dim3 grid(S, d.num_kv_heads, d.batch);
  return launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, st, mk, mv, d,
                    static_cast<const uint16_t*>(q), sm_scale * kLog2e, sel_idx, sel_cnt,
                    sel_stride, S, part_acc, part_ml, ctx, sa);
}

template <int D>
cudaError_t launch_mma_d(const kv_cache_desc& d, const CUtensorMap& mk, const CUtensorMap& mv,
                         const void* q, int G, float sm_scale, const int32_t* sel_idx,
                         const int32_t* sel_cnt, int sel_stride, int S, float* part_acc,
                         float* part_ml, DevCtx ctx, cudaStream_t st, const StepArgs& sa) {
  switch (G) {
    case 1: return launch_mma<D, 1>(d, mk, mv, q, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx, st, sa);
    case 2: return launch_mma<D, 2>(d, mk, mv, q, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx, st, sa);
    case 4: return launch_mma<D, 4>(d, mk, mv, q, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx, st, sa);
    case 8: return launch_mma<D, 8>(d, mk, mv, q, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc, part_ml, ctx, st, sa);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bf16_common(const kv_cache_desc& d, const void* q, int G, float sm_scale,
                               const int32_t* sel_idx, const int32_t* sel_cnt, int sel_stride,
                               int S, float* part_acc, float* part_ml, DevCtx ctx,
                               cudaStream_t st, const StepArgs& sa) {
  if ((long long)d.num_phys_pages * d.num_kv_heads * d.page_size >= (1ll << 31))
    return cudaErrorInvalidValue;                 // TMA row coordinates are 32-bit
  CUtensorMap mk, mv;
  if (!pool_tensor_map(&mk, d.k_pool, d) || !pool_tensor_map(&mv, d.v_pool, d))
    return cudaErrorInvalidValue;
  if (d.head_dim == 128)
    return launch_mma_d<128>(d, mk, mv, q, G, sm_scale, sel_idx, sel_cnt, sel_stride, S,
                             part_acc, part_ml, ctx, st, sa);
  return launch_mma_d<64>(d, mk, mv, q, G, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc,
                          part_ml, ctx, st, sa);
}

}  // namespace

cudaError_t launch_split_attn_bf16(const kv_cache_desc& d, const void* q, int G, float sm_scale,
                                   const int32_t* sel_idx, const int32_t* sel_cnt,
                                   int sel_stride, int S, float* part_acc, float* part_ml,
                                   DevCtx ctx, cudaStream_t st) {
  const StepArgs none{};
  return launch_bf16_common(d, q, G, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc,
                            part_ml, ctx, st, none);
}

cudaError_t launch_step_attn_bf16(const kv_cache_desc& d, const void* q, int G, float sm_scale,
                                  const int32_t* sel_idx, const int32_t* sel_cnt,
                                  int sel_stride, int S, float* part_acc, float* part_ml,
                                  DevCtx ctx, cudaStream_t st, const StepArgs& sa) {
  return launch_bf16_common(d, q, G, sm_scale, sel_idx, sel_cnt, sel_stride, S, part_acc,
                            part_ml, ctx, st, sa);
}

void step_attn_limits_bf16(int head_dim, int G, int* max_select_pages, int* max_splits) {
  int sel = 0, ring = 0;
#define SKV_LIM_CASE(DD, GG)                                                               \
  if (head_dim == DD && G == GG) {                                                         \
    sel = MmaCfg<DD, GG>::MAX_SELECT_PAGES;                                                \
    ring = MmaCfg<DD, GG>::NSTAGE * MmaCfg<DD, GG>::STAGE_BYTES;                           \
  }
  SKV_LIM_CASE(64, 1) SKV_LIM_CASE(64, 2) SKV_LIM_CASE(64, 4) SKV_LIM_CASE(64, 8)
  SKV_LIM_CASE(128, 1) SKV_LIM_CASE(128, 2) SKV_LIM_CASE(128, 4) SKV_LIM_CASE(128, 8)
#undef SKV_LIM_CASE
  *max_select_pages = sel;
  *max_splits = G > 0 ? (ring / 4 - 2 * G) / (2 * G) : 0;   // merge: [G][S] weights and l
}

size_t split_attn_smem_bf16(int head_dim, int G) {
#define SKV_SMEM_CASE(DD, GG) if (head_dim == DD && G == GG) return MmaCfg<DD, GG>::SMEM;
  SKV_SMEM_CASE(64, 1) SKV_SMEM_CASE(64, 2) SKV_SMEM_CASE(64, 4) SKV_SMEM_CASE(64, 8)
  SKV_SMEM_CASE(128, 1) SKV_SMEM_CASE(128, 2) SKV_SMEM_CASE(128, 4) SKV_SMEM_CASE(128, 8)
#undef SKV_SMEM_CASE
  return 0;
}

}  // namespace skv
