"""kv_select_decode_attn: selection, split-K attention and merge in one kernel (bf16).

Its selection must equal kv_select_topk's on the same scores bit for bit, its output must
match the separate calls (select, attention, merge kernel) within float32 rounding and the
oracle within the bf16 bar, the dense call must equal dense attention, and the per-group
counters must be back at zero after every call.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import inputs

from gpu_helpers import BF16_TOL, assert_no_device_error, f64, need_gpu, oracle_group, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


SHAPES = [(128, 4, 16), (128, 8, 64), (128, 1, 32), (64, 2, 16), (64, 8, 64)]
LENS = [(1000, 4097, 37), (0, 1, 17, 65, 3000), (30000,)]


@pytest.mark.parametrize("D,G,PS", SHAPES)
@pytest.mark.parametrize("lens", LENS)
@pytest.mark.parametrize("keep", [dict(keep_ratio=0.3), dict(budget_pages=20),
                                  dict(keep_ratio=0.02)], ids=["r0.3", "budget20", "r0.02"])
@pytest.mark.parametrize("S", [1, 5, 40])
def test_select_attend_merge_in_one_kernel(D, G, PS, lens, keep, S):
    Hkv = 2
    w = workload(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=PS, dtype="bf16",
                 seed=13, seq_lens=lens, planted=6)
    c = inputs.make_cache(w, "cuda", extra_phys_pages=3)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    scores = skv.kv_score_pages(kv, c.q, stats)
    ratio, budget = keep.get("keep_ratio", 0.0), keep.get("budget_pages", 0)
    k_max = skv.max_keep_pages(kv.stride, ratio if not budget else None, budget or None)
    B = w.batch
    sel = torch.full((B, Hkv, k_max), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, Hkv), -7, dtype=torch.int32, device="cuda")
    ctr = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
    outs = []
    for rep in range(2):                               # counters must be reusable
        out, lse = skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores, keep_ratio=ratio,
                                             budget_pages=budget, k_max=k_max, num_splits=S,
                                             counters=ctr, sel_idx=sel, sel_cnt=cnt)
        assert_no_device_error()
        assert int(ctr.abs().sum()) == 0
        outs.append(f64(out))
    assert (outs[0] == outs[1]).all()
    out, lse = outs[0], f64(lse)
    # selection: identical to the separate top-k kernel
    sel2, cnt2 = skv.kv_select_topk(scores, c.seq_lens, PS, keep_ratio=ratio,
                                    budget_pages=budget, k_max=k_max)
    sel, cnt, sel2, cnt2 = (x.cpu().numpy() for x in (sel, cnt, sel2, cnt2))
    np.testing.assert_array_equal(cnt, cnt2)
    for b in range(B):
        for g in range(Hkv):
            np.testing.assert_array_equal(sel[b, g, : cnt[b, g]], sel2[b, g, : cnt2[b, g]])
    # output: the separate calls with the same split count, and the oracle
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, torch.from_numpy(sel2).cuda(),
                                        torch.from_numpy(cnt2).cuda(), num_splits=S)
    out2, lse2 = skv.kv_merge_splits(acc, ml)
    np.testing.assert_allclose(out, f64(out2), rtol=0, atol=1e-6)
    for b, L in enumerate(lens):
        if L == 0:                                     # nothing to attend to
            assert (cnt[b] == 0).all() and (out[b] == 0).all() and np.isneginf(lse[b]).all()
            continue
        for g in range(Hkv):
            o = oracle_group(c, b, g, ratio=ratio if not budget else None,
                             budget_tokens=budget * PS if budget else None)
            k = int(cnt[b, g])
            assert k == o["k"]
            got = sel[b, g, :k]
            ok, msg = oracle.check_selection(got, o["scores"], k)
            assert ok, msg
            ref, ref_lse = oracle.attend(o["q"], o["K"], o["V"], o["table"], o["lens"], PS,
                                         w.sm_scale, selected=[[got]])
            hs = slice(g * G, (g + 1) * G)
            assert np.abs(out[b, hs] - ref[0]).max() < BF16_TOL
            assert np.abs(lse[b, hs] - ref_lse[0]).max() < 1e-4


@pytest.mark.parametrize("S", [1, 7, 38])
def test_dense_call_is_dense_attention(S):
    w = workload(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, dtype="bf16",
                 seed=14, seq_lens=(5000, 33, 0), planted=4)
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    ctr = torch.zeros((w.batch, 2), dtype=torch.int32, device="cuda")
    out, lse = skv.kv_select_decode_attn(kv, c.q, w.sm_scale, None, num_splits=S, counters=ctr)
    assert_no_device_error()
    assert int(ctr.abs().sum()) == 0
    ref, _ = oracle.attend(f64(c.q), f64(c.k_pool), f64(c.v_pool), c.page_table.cpu().numpy(),
                           c.seq_lens.cpu().numpy(), 16, w.sm_scale)
    assert np.abs(f64(out) - ref).max() < BF16_TOL
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, num_splits=S)
    out2, _ = skv.kv_merge_splits(acc, ml)
    np.testing.assert_allclose(f64(out), f64(out2), rtol=0, atol=1e-6)


def _score_rows(kind, n, gen):
    if kind == "coarse":                       # many exact ties, both signs, both zeros
        s = torch.round(torch.randn(n, generator=gen, dtype=torch.float64) * 4) / 4
        s[: min(n, 40)] = -0.0
        return s.float()
    if kind == "tied":                         # every page equal
        return torch.full((n,), 1.5)
    if kind == "outliers":                     # a few huge scores over a narrow band
        s = 100.0 + torch.rand(n, generator=gen) * 1e-3
        s[torch.randint(0, n, (min(n, 7),), generator=gen)] = 1e6
        return s
    if kind == "ramp":                         # distinct, ascending
        return torch.arange(n, dtype=torch.float32) * 0.5 - n / 4
    if kind == "sampled_high":                 # the largest scores sit exactly on the pages
        s = torch.randn(n, generator=gen)      # a strided 512-key sample of the row reads, so
        st = (n // 512) | 1                    # the sample puts its bound L too high: fewer
        idx = torch.tensor(sorted({(j * st) % n for j in range(512)}))   # than k keys >= L
        s[idx] = 1000.0 + torch.arange(len(idx), dtype=torch.float32)
        return s
    if kind == "tied_low":                     # a few distinct high scores over a floor of
        s = torch.full((n,), 1.0)              # ties: every key >= L, too many to gather
        s[torch.randint(0, n, (20,), generator=gen)] = 5.0 + torch.rand(20, generator=gen)
        return s
    return torch.randn(n, generator=gen)


@pytest.mark.parametrize("n", [5, 300, 2047, 2048, 8192, 9003, 21440])
@pytest.mark.parametrize("kind", ["coarse", "tied", "outliers", "ramp", "normal",
                                  "sampled_high", "tied_low"])
def test_in_kernel_selection_is_exact_on_given_scores(n, kind):
    """Arbitrary score rows through the in-kernel selection: the oracle's rule exactly
    (score descending, lower page first on ties, ascending output). At 8192 and 21440 pages
    with keep ratio 0.02 the attention kernel's sample filter runs and its runs come from the
    page-ordered candidates; sampled_high and tied_low defeat the filter, so those runs come
    from the search over every key instead."""
    PS, D, G, Hkv = 16, 128, 4, 2
    w = workload(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=PS, dtype="bf16",
                 seed=n, seq_lens=(n * PS, n * PS - 5))
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    gen = torch.Generator().manual_seed(n * 7 + len(kind))
    scores = torch.stack([torch.stack([_score_rows(kind, kv.stride, gen) for _ in range(Hkv)])
                          for _ in range(w.batch)]).contiguous()
    sh = scores.double().numpy()
    scores = scores.cuda()
    for kw in (dict(keep_ratio=0.3), dict(keep_ratio=0.02), dict(budget_pages=max(1, n // 3))):
        ratio, budget = kw.get("keep_ratio", 0.0), kw.get("budget_pages", 0)
        k_max = skv.max_keep_pages(kv.stride, ratio if not budget else None, budget or None)
        sel = torch.full((w.batch, Hkv, k_max), -1, dtype=torch.int32, device="cuda")
        cnt = torch.full((w.batch, Hkv), -1, dtype=torch.int32, device="cuda")
        S_auto = skv.kv_auto_num_splits(kv, w.num_q_heads, k_max)
        S = min(8, S_auto)
        out, _ = skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores, keep_ratio=ratio,
                                           budget_pages=budget, k_max=k_max, num_splits=S,
                                           sel_idx=sel, sel_cnt=cnt)
        assert_no_device_error()
        # the automatic split count: short runs per CTA (each CTA writes its run's part)
        sel_a = torch.full_like(sel, -1)
        skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores, keep_ratio=ratio,
                                  budget_pages=budget, k_max=k_max, num_splits=S_auto,
                                  sel_idx=sel_a, sel_cnt=torch.empty_like(cnt))
        assert_no_device_error()
        sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
        np.testing.assert_array_equal(sel_a.cpu().numpy(), sel)
        for b in range(w.batch):
            nb = oracle.num_pages(int(c.seq_lens[b]), PS)
            k = (oracle.keep_count(nb, budget_tokens=budget * PS, page_size=PS) if budget
                 else oracle.keep_count(nb, ratio=ratio))
            for g in range(Hkv):
                assert cnt[b, g] == k
                np.testing.assert_array_equal(sel[b, g, :k], oracle.select_pages(sh[b, g, :nb], k))
        # the output is the separate calls' on the same selection
        acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, torch.from_numpy(sel).cuda(),
                                            torch.from_numpy(cnt).cuda(), num_splits=S)
        out2, _ = skv.kv_merge_splits(acc, ml)
        np.testing.assert_allclose(f64(out), f64(out2), rtol=0, atol=1e-6)


@pytest.mark.parametrize("n", [4096, 9001, 20000])
@pytest.mark.parametrize("kind", ["coarse", "outliers", "ramp", "normal", "sampled_high",
                                  "tied_low"])
def test_select_topk_long_groups_keeping_few(n, kind):
    """Groups of 4096 pages or more keeping at most a sixteenth, where the block top-k first
    filters the keys by a sample: the oracle's rule exactly (score descending, lower page
    first on ties, ascending output), ties, outliers and ramps included. sampled_high and
    tied_low defeat the sample (too few keys at or above its bound; too many to gather), so
    the search takes its path over every key."""
    PS, Hkv, B = 16, 2, 2
    gen = torch.Generator().manual_seed(n + 31 * len(kind))
    scores = torch.stack([torch.stack([_score_rows(kind, n, gen) for _ in range(Hkv)])
                          for _ in range(B)]).contiguous()
    lens = torch.tensor([n * PS, n * PS - 7 * PS - 3], dtype=torch.int32)
    sh = scores.double().numpy()
    for kw in (dict(keep_ratio=0.02), dict(budget_pages=max(1, n // 40))):
        ratio, budget = kw.get("keep_ratio", 0.0), kw.get("budget_pages", 0)
        k_max = skv.max_keep_pages(n, ratio if not budget else None, budget or None)
        sel, cnt = skv.kv_select_topk(scores.cuda(), lens.cuda(), PS, keep_ratio=ratio,
                                      budget_pages=budget, k_max=k_max)
        assert_no_device_error()
        sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
        for b in range(B):
            nb = oracle.num_pages(int(lens[b]), PS)
            k = (oracle.keep_count(nb, budget_tokens=budget * PS, page_size=PS) if budget
                 else oracle.keep_count(nb, ratio=ratio))
            for g in range(Hkv):
                assert cnt[b, g] == k
                np.testing.assert_array_equal(sel[b, g, :k], oracle.select_pages(sh[b, g, :nb], k))
