"""Sparse paged-KV decode attention for GB300: a C-ABI CUDA library and a thin binding.

``binding`` wraps ``libsparsekv.so`` (``include/sparsekv.h``) call for call; ``inputs``
draws seeded synthetic caches. Importing the package does not load the library: the first
call does, and raises if it has not been built.
"""

from . import inputs  # noqa: F401
from .binding import (  # noqa: F401
    ONE_LAUNCH,
    PLANS,
    DecodeStepGraph,
    PagedKV,
    kv_append_token,
    kv_auto_num_splits,
    kv_build_page_stats,
    kv_build_page_stats_fp8,
    kv_check_device_errors,
    kv_decode_attn_merge,
    kv_decode_step,
    kv_decode_step_fp8,
    kv_decode_step_plan,
    kv_decode_step_workspace_size,
    kv_dropped_mass,
    kv_entmax_decode_attn,
    kv_entmax_decode_step,
    kv_entmax_decode_step_workspace_size,
    kv_entmax_page_moments,
    kv_entmax_select,
    kv_dropped_mass_workspace_size,
    kv_merge_splits,
    kv_score_pages,
    kv_score_pages_fp8,
    kv_score_select,
    kv_select_decode_attn,
    kv_select_structured,
    kv_select_topk,
    kv_selftest_wait_timeout,
    kv_set_wait_limit_ns,
    kv_sparse_decode_attn,
    kv_version,
    kv_workspace_size,
    max_keep_pages,
)
