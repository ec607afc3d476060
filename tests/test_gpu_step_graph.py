"""kv_decode_step_graph_*: the decode step captured once and launched per token gives
kv_decode_step's result for every new query and length written into the captured buffers."""

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import inputs

from gpu_helpers import BF16_TOL, assert_no_device_error, f64, need_gpu, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("keep", [dict(keep_ratio=0.3), dict(keep_ratio=1.0),
                                  dict(budget_pages=24)])
def test_captured_step_equals_the_call_across_tokens(keep):
    w = workload(num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=16, dtype="bf16",
                 seed=5, seq_lens=(2000, 1500), planted=8)
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    q_buf = c.q.clone()
    lens_full = c.seq_lens.clone()
    # the captured cache descriptor points at the same lengths tensor, updated in place
    c.seq_lens.copy_(lens_full - 300)
    k_max = skv.max_keep_pages(kv.stride, keep.get("keep_ratio"), keep.get("budget_pages"))
    g = skv.DecodeStepGraph(kv, q_buf, w.sm_scale, stats, k_max=k_max, **keep)
    gen = torch.Generator(device="cuda").manual_seed(3)
    for step in range(3):
        q_new = torch.randn(c.q.shape, generator=gen, device="cuda").to(c.q.dtype)
        q_buf.copy_(q_new)
        c.seq_lens.copy_(lens_full - 300 + 100 * step)
        skv.kv_build_page_stats(kv, stats)
        out, lse = g.launch()
        ref, ref_lse = skv.kv_decode_step(kv, q_buf, w.sm_scale, stats, k_max=k_max, **keep)
        assert_no_device_error()
        np.testing.assert_allclose(f64(out), f64(ref), rtol=0, atol=1e-6)
        np.testing.assert_allclose(f64(lse), f64(ref_lse), rtol=0, atol=1e-6)
        if keep.get("keep_ratio") == 1.0:
            dense, _ = oracle.attend(f64(q_buf), f64(c.k_pool), f64(c.v_pool),
                                     c.page_table.cpu().numpy(), c.seq_lens.cpu().numpy(),
                                     w.page_size, w.sm_scale)
            assert np.abs(f64(out) - dense).max() < BF16_TOL
    g.close()


def test_captured_step_rejects_bad_arguments_without_a_graph():
    w = workload(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, dtype="bf16",
                 seed=6, seq_lens=(500,))
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    with pytest.raises(skv.binding.KVError):
        skv.DecodeStepGraph(kv, c.q, -1.0, keep_ratio=1.0)        # non-positive scale


def test_captured_step_with_host_buffers():
    """The query taken from q_host and the output left in out_host by the same launch (page-
    locked buffers: the kernels read and write them in place under unified addressing)."""
    w = workload(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, dtype="bf16",
                 seed=8, seq_lens=(3000,), planted=4)
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    q_dev = torch.empty_like(c.q)
    q_host = torch.empty(c.q.shape, dtype=c.q.dtype).pin_memory()
    out_host = torch.empty((1, 8, 128), dtype=torch.float32).pin_memory()
    g = skv.DecodeStepGraph(kv, q_dev, w.sm_scale, stats, keep_ratio=0.3, q_host=q_host,
                            out_host=out_host)
    gen = torch.Generator().manual_seed(4)
    for _ in range(2):
        q_host.copy_(torch.randn(c.q.shape, generator=gen).to(c.q.dtype))
        g.launch()
        torch.cuda.synchronize()
        ref, _ = skv.kv_decode_step(kv, q_host.cuda(), w.sm_scale, stats, keep_ratio=0.3)
        assert_no_device_error()
        np.testing.assert_allclose(out_host.numpy().astype(np.float64), f64(ref), rtol=0,
                                   atol=1e-6)
    g.close()
