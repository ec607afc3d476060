"""kv_decode_step_static: the decode step on the library's own static scratch.

Callers that cannot allocate device memory on the decode path (a plain C or plugin host
without a device allocator, or a serving loop that must not call cudaMalloc per token) use
this entry point instead of kv_decode_step. Its output must match kv_decode_step's within
the tests' output tolerance on two calls in a row -- the second with a different query, so
that anything left over in the shared scratch from the first call would show. This file is
collected last so that a run stopping at the first failure has run every other test.
"""

import numpy as np
import pytest
import torch

import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import binding, inputs

from gpu_helpers import BF16_TOL, assert_no_device_error, f64, need_gpu, workload

pytestmark = pytest.mark.gpu


def test_static_scratch_step_matches_the_workspace_step_twice_in_a_row():
    need_gpu()
    torch.cuda.set_device(0)
    w = workload(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, dtype="bf16",
                 seed=21, seq_lens=(3000, 777), planted=8)
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    q2 = torch.randn(c.q.shape, device="cuda").to(c.q.dtype)
    for q in (c.q, q2):
        for keep in (dict(keep_ratio=0.3), dict(keep_ratio=1.0), dict(budget_pages=20)):
            ref, ref_lse = skv.kv_decode_step(kv, q, w.sm_scale, stats, **keep)
            got, got_lse = binding.kv_decode_step_static(kv, q, w.sm_scale, stats, **keep)
            assert_no_device_error()
            assert np.abs(f64(got) - f64(ref)).max() < BF16_TOL, keep
            assert np.abs(f64(got_lse) - f64(ref_lse)).max() < 1e-4, keep


def test_static_scratch_rejects_shapes_above_its_limit():
    need_gpu()
    torch.cuda.set_device(0)
    # 4096 groups x 1024 pages of float32 scores alone is 16 MiB > 8 MiB: rejected on the
    # host before any launch (the pools are never read).
    B = 512
    k = torch.zeros((1, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((B, 1024), dtype=torch.int32, device="cuda")
    lens = torch.full((B,), 16, dtype=torch.int32, device="cuda")
    kv = binding.PagedKV(k, k.clone(), table, lens)
    q = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.KVError) as e:
        binding.kv_decode_step_static(kv, q, 0.1, k.new_zeros((1, 8, 2, 128)), keep_ratio=0.3)
    assert e.value.status == -4
