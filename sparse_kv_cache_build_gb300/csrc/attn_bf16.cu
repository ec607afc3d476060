// Split-K decode attention kernels for bf16 caches (see attn_impl.cuh).
#include "attn_impl.cuh"

namespace skv {

cudaError_t launch_split_attn_bf16(const kv_cache_desc& d, const void* q, int G, float sm_scale,
                                   const int32_t* sel_idx, const int32_t* sel_cnt,
                                   int sel_stride, int S, float* part_acc, float* part_ml,
                                   DevCtx ctx, cudaStream_t st) {
  if (d.head_dim == 128)
    return launch_split_attn_d<bf16_t, 128>(d, q, G, sm_scale, sel_idx, sel_cnt, sel_stride, S,
                                          part_acc, part_ml, ctx, st);
  return launch_split_attn_d<bf16_t, 64>(d, q, G, sm_scale, sel_idx, sel_cnt, sel_stride, S,
                                       part_acc, part_ml, ctx, st);
}

size_t split_attn_smem_bf16(int head_dim, int G) { return split_attn_smem_t<bf16_t>(head_dim, G); }

}  // namespace skv
