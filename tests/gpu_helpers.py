"""Shared plumbing of the GPU parity tests: run the library's path on a cache, and hand the
oracle byte copies of the same inputs (never a value computed by the library)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import binding, inputs

BF16_TOL = 2e-3     # max abs output error for bf16 caches
FP32_TOL = 1e-5     # max abs output error for fp32 caches


def out_tol(w: inputs.Workload) -> float:
    return FP32_TOL if w.dtype == "fp32" else BF16_TOL


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_build_gb300 import build as builder
    builder.build()
    binding.lib()


def f64(t) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def f32(t) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float32).numpy()


def workload(**kw) -> inputs.Workload:
    base = dict(name="t", batch=1, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                dtype="bf16", seed=0, planted=0)
    base.update(kw)
    if "seq_lens" in base:
        base["batch"] = len(base["seq_lens"])
    return inputs.Workload(**base)


def assert_no_device_error():
    st, flags = skv.kv_check_device_errors()
    assert st == 0, f"device error word {flags:#x}"


def group_inputs(c: inputs.KVCache, b: int, g: int):
    """Oracle inputs of one (sequence, KV head) group: the group's query heads and the
    sequence's pages of KV head g, copied to the host with a compact page table."""
    w = c.workload
    G = w.group_size
    n = oracle.num_pages(int(c.seq_lens[b]), w.page_size)
    phys = c.page_table[b, :n].to(torch.int64)
    K = f32(c.k_pool.index_select(0, phys)[:, g:g + 1])          # [n][1][PS][D]
    V = f32(c.v_pool.index_select(0, phys)[:, g:g + 1])
    q = f64(c.q[b:b + 1, g * G:(g + 1) * G])                      # [1][G][D]
    table = np.arange(max(n, 1), dtype=np.int64)[None, :]
    lens = np.array([int(c.seq_lens[b])])
    return q, K, V, table, lens


def oracle_group(c, b, g, ratio=None, budget_tokens=None, keep_pages=None, selected=None):
    """Oracle stats, scores, keep count and selection of one group."""
    w = c.workload
    q, K, V, table, lens = group_inputs(c, b, g)
    mn, mx = oracle.page_stats(K, table, lens, w.page_size)
    s = oracle.page_scores(q, mn, mx, table, lens, w.page_size)[0][0]
    n = s.shape[0]
    if keep_pages is not None:
        k = min(n, keep_pages)
    elif budget_tokens is not None:
        k = oracle.keep_count(n, budget_tokens=budget_tokens, page_size=w.page_size)
    else:
        k = oracle.keep_count(n, ratio=ratio)
    return dict(q=q, K=K, V=V, table=table, lens=lens, mn=mn, mx=mx, scores=s, k=k)


def round256(x: int) -> int:
    return (x + 255) // 256 * 256


def round4(x: int) -> int:
    return (x + 3) // 4 * 4


def step_selection(workspace, B, Hkv, stride, k_max):
    """sel_idx and sel_cnt of a sparse kv_decode_step, read from its workspace at the
    offsets include/sparsekv.h documents."""
    a = 2 * round256(B * Hkv * 4) + round256(B * Hkv * round4(stride) * 4)
    c = a + round256(B * Hkv * k_max * 4)
    sel = workspace[a: a + B * Hkv * k_max * 4].view(torch.int32).view(B, Hkv, k_max)
    cnt = workspace[c: c + B * Hkv * 4].view(torch.int32).view(B, Hkv)
    return sel.cpu().numpy(), cnt.cpu().numpy()


def step_score_region(workspace, B, Hkv, stride):
    """The byte range of a kv_decode_step workspace that holds the step's scores (after the
    two per-group counter arrays)."""
    a = 2 * round256(B * Hkv * 4)
    return workspace[a: a + round256(B * Hkv * round4(stride) * 4)]
