"""The C-ABI library on the host: it builds, loads, exports every declared symbol, and
rejects bad arguments before touching a GPU. No compute call runs here."""

import ctypes
import math
import os
import re

import pytest

import oracle
from sparse_kv_cache_build_gb300 import binding
from sparse_kv_cache_build_gb300 import build as builder

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparsekv.h")


@pytest.fixture(scope="module")
def lib():
    builder.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(kv_[a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kv_build_page_stats", "kv_score_pages", "kv_select_topk",
                 "kv_sparse_decode_attn", "kv_merge_splits", "kv_dropped_mass"):
        assert must in names
    assert sorted(binding.EXPORTS) == names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    assert lib.kv_version() == 101
    for code in range(-7, 1):
        s = lib.kv_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.kv_status_string(-99).decode() == "unknown status"


def desc(**kw):
    base = dict(k_pool=16 * 1000, v_pool=16 * 2000, dtype=0, num_phys_pages=4,
                num_kv_heads=2, page_size=16, head_dim=128, batch=1, page_table=4096,
                page_table_stride=4, seq_lens=8192)
    base.update(kw)
    return binding.KVCacheDesc(**base)


def test_invalid_arguments_are_rejected_on_the_host(lib):
    d = desc()
    null = None
    assert lib.kv_build_page_stats(None, 256, None, 0, null) == -1
    assert lib.kv_build_page_stats(ctypes.byref(desc(k_pool=None)), 256, None, 0, null) == -1
    assert lib.kv_build_page_stats(ctypes.byref(desc(head_dim=96)), 256, None, 0, null) == -2
    assert lib.kv_build_page_stats(ctypes.byref(desc(page_size=8)), 256, None, 0, null) == -2
    assert lib.kv_build_page_stats(ctypes.byref(desc(dtype=7)), 256, None, 0, null) == -2
    assert lib.kv_build_page_stats(ctypes.byref(desc(k_pool=16 * 1000 + 2)), 256, None, 0, null) == -7
    assert lib.kv_build_page_stats(ctypes.byref(d), None, None, 0, null) == -1
    assert lib.kv_build_page_stats(ctypes.byref(d), 258, None, 0, null) == -7
    # a physical-page subset: its length must lie in [0, num_phys_pages]; an empty list
    # has nothing to rebuild and launches nothing
    assert lib.kv_build_page_stats(ctypes.byref(d), 256, 4096, -1, null) == -1
    assert lib.kv_build_page_stats(ctypes.byref(d), 256, 4096, 5, null) == -1
    assert lib.kv_build_page_stats(ctypes.byref(d), 256, 4096, 0, null) == 0
    # group size 3 is outside {1, 2, 4, 8}; 7 heads do not divide into 2 KV heads
    assert lib.kv_score_pages(ctypes.byref(d), 512, 6, 256, 1024, 4, null) == -2
    assert lib.kv_score_pages(ctypes.byref(d), 512, 7, 256, 1024, 4, null) == -1
    assert lib.kv_score_pages(ctypes.byref(d), 512, 8, 256, 1024, 3, null) == -1  # stride
    assert lib.kv_score_pages(ctypes.byref(d), 520, 8, 256, 1024, 4, null) == -7  # q align
    # select: no keep rule at all, k_max 0
    assert lib.kv_select_topk(1024, 4, 2048, 16, 1, 2, None, 0.0, 0, 4, 64, 128, null) == -1
    assert lib.kv_select_topk(1024, 4, 2048, 16, 1, 2, None, 0.3, 0, 0, 64, 128, null) == -1
    # attention: zero splits, non-positive scale, splits below the page-list capacity
    assert lib.kv_sparse_decode_attn(ctypes.byref(d), 512, 8, 0.1, None, None, 0, 0,
                                     64, 128, null) == -1
    assert lib.kv_sparse_decode_attn(ctypes.byref(d), 512, 8, 0.0, None, None, 0, 1,
                                     64, 128, null) == -1
    big = desc(page_table_stride=5000)
    assert lib.kv_sparse_decode_attn(ctypes.byref(big), 512, 8, 0.1, None, None, 0, 2,
                                     64, 128, null) == -1
    assert lib.kv_merge_splits(64, 128, 1, 8, 0, 128, 256, None, null) == -1
    assert lib.kv_merge_splits(64, 128, 1, 8, 1, 96, 256, None, null) == -2
    # dropped mass without a workspace
    assert lib.kv_dropped_mass(ctypes.byref(d), 512, 8, 0.1, 64, 128, 4, 256, None, 0,
                               null) == -4
    # decode step: misaligned workspace
    assert lib.kv_decode_step(ctypes.byref(d), 512, 8, 0.1, 256, 0.3, 0, 4, 1, 1024, None,
                              4096 + 16, 1 << 20, null) == -4
    assert lib.kv_set_wait_limit_ns(2_000_000_000) == 0


def test_workspace_size_dispatches_to_each_calls_own_size(lib):
    d = desc(batch=3, page_table_stride=40)
    ref = ctypes.byref(d)
    assert lib.kv_workspace_size(0, ref, 8, 12, 5) == lib.kv_decode_step_workspace_size(ref, 8, 12, 5)
    assert lib.kv_workspace_size(0, ref, 8, 12, 5) > 0
    assert lib.kv_workspace_size(1, ref, 8, 0, 0) == lib.kv_dropped_mass_workspace_size(ref, 8)
    assert lib.kv_workspace_size(2, ref, 8, 12, 0) == lib.kv_entmax_attn_workspace_size(ref, 8, 12)
    assert lib.kv_workspace_size(2, ref, 8, 0, 0) == lib.kv_entmax_attn_workspace_size(ref, 8, 0)
    assert lib.kv_workspace_size(3, ref, 8, 12, 0) == \
        lib.kv_entmax_decode_step_workspace_size(ref, 8, 12)
    assert lib.kv_workspace_size(99, ref, 8, 12, 5) == 0
    assert lib.kv_workspace_size(0, None, 8, 12, 5) == 0


def test_dropped_mass_workspace_size_formula(lib):
    d = desc(batch=3)
    assert lib.kv_dropped_mass_workspace_size(ctypes.byref(d), 8) == 3 * 8 * 64 * 3 * 4
    assert lib.kv_dropped_mass_workspace_size(None, 8) == 0


def test_max_keep_pages_bounds_the_keep_count():
    for stride in (1, 7, 256, 2048, 16384):
        for r in (0.01, 0.02, 0.2, 0.3, 0.5, 0.999, 1.0):
            bound = binding.max_keep_pages(stride, keep_ratio=r)
            for n in {1, stride // 3 + 1, stride}:
                assert oracle.keep_count(n, ratio=r) <= bound
        assert binding.max_keep_pages(stride, budget_pages=128) == min(stride, 128)
    assert binding.max_keep_pages(16384, keep_ratio=1 / 50) == 328
    assert math.ceil(0.3 * 2048) == binding.max_keep_pages(2048, keep_ratio=0.3)


def test_binding_refuses_cpu_tensors():
    import torch
    k = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.PagedKV(k, k.clone(), torch.zeros((1, 4), dtype=torch.int32),
                        torch.zeros((1,), dtype=torch.int32))
