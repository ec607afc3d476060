"""FP8 (E4M3) page statistics through the C ABI, against the float64 oracle.

Bytes and exponents bit-exact; scores to float32 rounding of the oracle's score from the
decoded statistics, and never below the score from exact statistics; the decode step's
selection exactly the oracle's rule on the GPU's own scores, and its output within the bf16
bar of the oracle's attention over that selection.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8stats
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import inputs

from gpu_helpers import (BF16_TOL, FP32_TOL, assert_no_device_error, f64, need_gpu, out_tol,
                         workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


SHAPES = [("bf16", 128, 4, 16), ("bf16", 64, 2, 64), ("fp32", 128, 8, 32), ("fp32", 64, 1, 16)]


def make(dtype, D, G, PS, lens=(1000, 4097, 37), seed=9, Hkv=2, edge=True):
    w = workload(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=PS, dtype=dtype,
                 seed=seed, seq_lens=lens, planted=4)
    c = inputs.make_cache(w, "cuda", extra_phys_pages=3)
    if edge:
        k = c.k_pool
        P = c.page_table[0, :6].long()
        k[P[0]] *= 1e4                                   # a large exponent
        k[P[1]] *= 1e-4                                  # a small one
        k[P[2], 0, 0, :] = 448.0                         # a row whose max sits on the limit
        k[P[2], 0, 1:, :] = -1.0
        k[P[3], 1, :, : D // 2] = 0.0                    # zeros of both signs
        k[P[3], 1, 0, : D // 4] = -0.0
        k[P[4]] = torch.round(k[P[4]] * 4) / 4           # on-grid values
    return w, c


def oracle_fp8(c):
    K = f64(c.k_pool)
    return fp8stats.page_stats_fp8(K, c.page_table.cpu().numpy(), c.seq_lens.cpu().numpy(),
                                   c.workload.page_size)


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
def test_fp8_stats_bit_exact(dtype, D, G, PS):
    w, c = make(dtype, D, G, PS)
    kv = skv.PagedKV.from_cache(c)
    stats = torch.full((c.num_phys_pages, 2, 2, D), 0xAB, dtype=torch.uint8, device="cuda")
    exps = torch.full((c.num_phys_pages, 2), 99, dtype=torch.int8, device="cuda")
    skv.kv_build_page_stats_fp8(kv, stats, exps)
    assert_no_device_error()
    cmn, cmx, e, mapped = oracle_fp8(c)
    got = stats.cpu().numpy()
    np.testing.assert_array_equal(got[mapped, :, 0, :], cmn[mapped])
    np.testing.assert_array_equal(got[mapped, :, 1, :], cmx[mapped])
    np.testing.assert_array_equal(exps.cpu().numpy()[mapped], e[mapped])
    assert (got[~mapped] == 0xAB).all() and (exps.cpu().numpy()[~mapped] == 99).all()
    assert e[mapped].max() > 5 and e[mapped].min() < -15           # the edge rows took effect


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
def test_fp8_scores_match_oracle_and_bound_exact_scores(dtype, D, G, PS):
    w, c = make(dtype, D, G, PS)
    kv = skv.PagedKV.from_cache(c)
    stats8, exps = skv.kv_build_page_stats_fp8(kv)
    got = f64(skv.kv_score_pages_fp8(kv, c.q, stats8, exps))
    exact = f64(skv.kv_score_pages(kv, c.q, skv.kv_build_page_stats(kv)))
    assert_no_device_error()
    cmn, cmx, e, mapped = oracle_fp8(c)
    dmn, dmx = fp8stats.decode_stats_fp8(cmn, cmx, e, mapped)
    ref = oracle.page_scores(f64(c.q), dmn, dmx, c.page_table.cpu().numpy(),
                             c.seq_lens.cpu().numpy(), PS)
    for b in range(w.batch):
        n = ref[b].shape[1]
        scale = np.abs(ref[b]).max(axis=1, keepdims=True) + 1.0
        assert (np.abs(got[b, :, :n] - ref[b]) <= 2e-6 * scale).all()
        assert (got[b, :, :n] >= exact[b, :, :n] - 4e-6 * scale).all()


@pytest.mark.parametrize("dtype,D,G,PS,lens", [
    ("bf16", 128, 4, 16, (1000, 4097, 37)),        # plan 1
    ("bf16", 128, 8, 16, (8200 * 16, 500)),         # plan 2
    ("fp32", 64, 4, 16, (3000, 77)),                # four kernels
])
@pytest.mark.parametrize("keep", [dict(keep_ratio=0.3), dict(budget_pages=25)], ids=["r0.3", "b25"])
def test_fp8_decode_step_matches_oracle(dtype, D, G, PS, lens, keep):
    w, c = make(dtype, D, G, PS, lens=lens, edge=False)
    kv = skv.PagedKV.from_cache(c)
    stats8, exps = skv.kv_build_page_stats_fp8(kv)
    ratio, budget = keep.get("keep_ratio", 0.0), keep.get("budget_pages", 0)
    k_max = skv.max_keep_pages(kv.stride, ratio if not budget else None, budget or None)
    ws = torch.zeros((skv.kv_decode_step_workspace_size(kv, w.num_q_heads, k_max),),
                     dtype=torch.uint8, device="cuda")
    out, lse = skv.kv_decode_step_fp8(kv, c.q, w.sm_scale, stats8, exps, keep_ratio=ratio or 1.0,
                                      budget_pages=budget, k_max=k_max, workspace=ws)
    assert_no_device_error()
    scores = f64(skv.kv_score_pages_fp8(kv, c.q, stats8, exps))
    sel, cnt = skv.kv_select_topk(torch.from_numpy(scores).float().cuda(), c.seq_lens, PS,
                                  keep_ratio=ratio, budget_pages=budget, k_max=k_max)
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt)
    out2, _ = skv.kv_merge_splits(acc, ml)
    np.testing.assert_allclose(f64(out), f64(out2), rtol=0, atol=1e-6)
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    q, Kp, Vp = f64(c.q), f64(c.k_pool), f64(c.v_pool)
    table, L = c.page_table.cpu().numpy(), c.seq_lens.cpu().numpy()
    for b in range(w.batch):
        n = oracle.num_pages(int(L[b]), PS)
        k = (oracle.keep_count(n, budget_tokens=budget * PS, page_size=PS) if budget
             else oracle.keep_count(n, ratio=ratio))
        for g in range(w.num_kv_heads):
            assert cnt[b, g] == k
            np.testing.assert_array_equal(sel[b, g, :k], oracle.select_pages(scores[b, g, :n], k))
        chosen = [[sel[b, g, : cnt[b, g]] for g in range(w.num_kv_heads)]]
        ref, ref_lse = oracle.attend(q[b:b + 1], Kp, Vp, table[b:b + 1], L[b:b + 1], PS,
                                     w.sm_scale, selected=chosen)
        assert np.abs(f64(out)[b] - ref[0]).max() < out_tol(w)
        assert np.abs(f64(lse)[b] - ref_lse[0]).max() < 1e-4
