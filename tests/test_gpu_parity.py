"""GPU parity of every step of the path against the float64 oracle, through the C-ABI.

Sizes span several 64-token tiles, several splits and ragged last pages. Bars: page
statistics and all index work bit-exact; scores to float32 rounding; selections identical
except inside the 1e-4 relative tie band (and exactly the oracle's rule applied to the GPU's
own float32 scores); outputs within 2e-3 (bf16) or 1e-5 (fp32) max abs error.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import inputs

from gpu_helpers import (assert_no_device_error, f32, f64, group_inputs, need_gpu,
                         oracle_group, out_tol, workload)

pytestmark = pytest.mark.gpu

SHAPES = [  # dtype, D, G, PS
    ("bf16", 128, 4, 16), ("bf16", 128, 8, 64), ("bf16", 128, 1, 32), ("bf16", 64, 2, 16),
    ("fp32", 64, 4, 16), ("fp32", 128, 8, 32), ("bf16", 64, 8, 64), ("fp32", 64, 1, 64),
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


def make(dtype="bf16", D=128, G=4, PS=16, lens=(1000, 4097, 37), Hkv=2, planted=6, seed=3,
         extra=5):
    w = workload(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=PS, dtype=dtype,
                 seed=seed, seq_lens=tuple(lens), planted=planted)
    return inputs.make_cache(w, "cuda", extra_phys_pages=extra)


# ------------------------------------------------------------------------------ stats

@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
def test_page_stats_bit_exact(dtype, D, G, PS):
    c = make(dtype, D, G, PS)
    kv = skv.PagedKV.from_cache(c)
    stats = torch.full((c.num_phys_pages, 2, 2, D), float("nan"), dtype=c.k_pool.dtype,
                       device="cuda")
    skv.kv_build_page_stats(kv, stats)
    assert_no_device_error()
    K, table, lens = f64(c.k_pool), c.page_table.cpu().numpy(), c.seq_lens.cpu().numpy()
    mn, mx = oracle.page_stats(K, table, lens, PS)
    got = f64(stats)
    mapped = ~np.isnan(mn[:, 0, 0])
    assert mapped.sum() == sum(c.pages_per_seq)
    np.testing.assert_array_equal(got[mapped, :, 0, :], mn[mapped])
    np.testing.assert_array_equal(got[mapped, :, 1, :], mx[mapped])
    assert np.isnan(got[~mapped]).all()          # unmapped pages are never written


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES[:4])
def test_page_stats_rebuild_of_a_physical_page_subset(dtype, D, G, PS):
    """A strictly ascending list of physical pages: exactly the mapped ones among them are
    rebuilt, bit-exact; every other row keeps what it held; listed unmapped pages stay
    unwritten; an out-of-order list is flagged."""
    c = make(dtype, D, G, PS)
    kv = skv.PagedKV.from_cache(c)
    NP = c.num_phys_pages
    K, table, lens = f64(c.k_pool), c.page_table.cpu().numpy(), c.seq_lens.cpu().numpy()
    mn, mx = oracle.page_stats(K, table, lens, PS)
    mapped = ~np.isnan(mn[:, 0, 0])
    rng = np.random.default_rng(11)
    subset = np.sort(rng.choice(NP, size=NP // 3, replace=False))
    unmapped = np.nonzero(~mapped)[0]
    subset = np.unique(np.concatenate([subset, unmapped[:2]]))   # two listed unmapped pages
    stats = torch.full((NP, 2, 2, D), float("nan"), dtype=c.k_pool.dtype, device="cuda")
    skv.kv_build_page_stats(kv, stats,
                            phys_pages=torch.tensor(subset, dtype=torch.int32, device="cuda"))
    assert_no_device_error()
    got = f64(stats)
    want = np.zeros(NP, dtype=bool)
    want[subset] = True
    rebuilt = want & mapped
    assert rebuilt.sum() > 0 and (mapped & ~want).sum() > 0
    np.testing.assert_array_equal(got[rebuilt, :, 0, :], mn[rebuilt])
    np.testing.assert_array_equal(got[rebuilt, :, 1, :], mx[rebuilt])
    assert np.isnan(got[~rebuilt]).all()
    # an empty list rebuilds nothing; the full build then matches the oracle everywhere
    skv.kv_build_page_stats(kv, stats, phys_pages=torch.zeros((0,), dtype=torch.int32,
                                                              device="cuda"))
    assert np.isnan(f64(stats)[~rebuilt]).all()
    skv.kv_build_page_stats(kv, stats)
    got = f64(stats)
    np.testing.assert_array_equal(got[mapped, :, 0, :], mn[mapped])
    # a list out of order is flagged as a bad page
    bad = torch.tensor([3, 1, 2], dtype=torch.int32, device="cuda")
    skv.kv_build_page_stats(kv, stats, phys_pages=bad)
    st, flags = skv.kv_check_device_errors()
    assert flags & 1


# ------------------------------------------------------------------------------ score

@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
def test_page_scores_match_oracle_and_bound_qk(dtype, D, G, PS):
    c = make(dtype, D, G, PS)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    scores = skv.kv_score_pages(kv, c.q, stats)
    assert_no_device_error()
    got = f64(scores)
    for b in range(c.workload.batch):
        for g in range(2):
            o = oracle_group(c, b, g, ratio=0.3)
            n = o["scores"].shape[0]
            ref = o["scores"]
            scale = np.abs(ref).max() + 1.0
            np.testing.assert_allclose(got[b, g, :n], ref, rtol=2e-6, atol=2e-6 * scale)
            # upper bound of the group-summed q.k of every valid token of each page
            qsum = o["q"][0].sum(axis=0)
            K = o["K"][:, 0].astype(np.float64)
            for p in range(n):
                v = oracle.valid_tokens(o["lens"][0], PS, p)
                true = (K[p, :v] @ qsum).max()
                assert got[b, g, p] >= true - 1e-5 * scale


# ------------------------------------------------------------------------------ select

def gpu_select(scores, lens, PS, **kw):
    sel, cnt = skv.kv_select_topk(scores, lens, PS, **kw)
    assert_no_device_error()
    return sel.cpu().numpy(), cnt.cpu().numpy()


@pytest.mark.parametrize("n,k", [(1, 1), (5, 2), (300, 7), (2048, 615), (8192, 1639),
                                 (16384, 328), (65536, 5000), (3000, 2999)])
def test_select_is_exact_on_given_scores_with_heavy_ties(n, k):
    torch.manual_seed(n + k)
    B, Hkv = 2, 3
    # coarse values: many exact ties, negative values, and both signed zeros
    s = torch.round(torch.randn((B, Hkv, n)) * 4) / 4
    s[0, 0, : min(n, 50)] = -0.0
    s[0, 1, :] = 1.5                             # a fully tied row
    scores = s.cuda()
    lens = torch.full((B,), n * 16, dtype=torch.int32, device="cuda")
    keep = torch.full((B,), k, dtype=torch.int32, device="cuda")
    sel, cnt = gpu_select(scores, lens, 16, keep=keep, k_max=k)
    sh = s.double().numpy()
    for b in range(B):
        for g in range(Hkv):
            assert cnt[b, g] == k
            want = oracle.select_pages(sh[b, g], k)
            np.testing.assert_array_equal(sel[b, g, :k], want)


def test_select_keep_rules_ratio_budget_and_edges():
    torch.manual_seed(0)
    lens_list = [0, 1, 15, 16, 17, 1000, 32768, 5 * 16]
    B = len(lens_list)
    stride = 2048
    s = torch.randn((B, 2, stride)).cuda()
    lens = torch.tensor(lens_list, dtype=torch.int32, device="cuda")
    sh = s.double().cpu().numpy()
    for kw, rule in [(dict(keep_ratio=0.3), dict(ratio=0.3)),
                     (dict(keep_ratio=0.2), dict(ratio=0.2)),
                     (dict(keep_ratio=1 / 50), dict(ratio=1 / 50)),
                     (dict(keep_ratio=1.0), dict(ratio=1.0)),
                     (dict(budget_pages=128), dict(budget_tokens=2048, page_size=16))]:
        sel, cnt = gpu_select(s, lens, 16, k_max=stride, **kw)
        for b, L in enumerate(lens_list):
            n = oracle.num_pages(L, 16)
            k = oracle.keep_count(n, **rule)
            for g in range(2):
                assert cnt[b, g] == k, (kw, L)
                np.testing.assert_array_equal(sel[b, g, :k], oracle.select_pages(sh[b, g, :n], k))


def test_select_flags_keep_above_k_max():
    s = torch.randn((1, 1, 100)).cuda()
    lens = torch.tensor([1600], dtype=torch.int32, device="cuda")
    sel, cnt = skv.kv_select_topk(s, lens, 16, keep_ratio=0.5, k_max=10)
    st, flags = skv.kv_check_device_errors()
    assert st == -5 and flags & 8
    assert cnt.item() == 10
    want = oracle.select_pages(s.double().cpu().numpy()[0, 0], 10)
    np.testing.assert_array_equal(sel.cpu().numpy()[0, 0], want)


# ------------------------------------------------------------------------------ attention

def run_sparse(c, ratio=None, budget_pages=0, S=None, keep=None):
    w = c.workload
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    scores = skv.kv_score_pages(kv, c.q, stats)
    sel, cnt = skv.kv_select_topk(scores, c.seq_lens, w.page_size, keep=keep,
                                  keep_ratio=ratio or 0.0, budget_pages=budget_pages)
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=S)
    out, lse = skv.kv_merge_splits(acc, ml)
    assert_no_device_error()
    return dict(kv=kv, stats=stats, scores=scores, sel=sel.cpu().numpy(), cnt=cnt.cpu().numpy(),
                acc=acc, ml=ml, out=f64(out), lse=f64(lse), S=acc.shape[2])


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
@pytest.mark.parametrize("S", [1, 3, 16])
def test_sparse_step_matches_oracle(dtype, D, G, PS, S):
    c = make(dtype, D, G, PS, planted=6)
    w = c.workload
    r = run_sparse(c, ratio=0.3, S=S)
    tol = out_tol(w)
    for b in range(w.batch):
        for g in range(w.num_kv_heads):
            o = oracle_group(c, b, g, ratio=0.3)
            k = o["k"]
            got_sel = r["sel"][b, g, : r["cnt"][b, g]]
            ok, msg = oracle.check_selection(got_sel, o["scores"], k)
            assert ok, msg
            # the index work is exact: the oracle's rule on the GPU's own float32 scores
            gs = f64(r["scores"][b, g, : o["scores"].shape[0]])
            np.testing.assert_array_equal(got_sel, oracle.select_pages(gs, k))
            # attention over the GPU's selected set
            out, lse = oracle.attend(o["q"], o["K"], o["V"], o["table"], o["lens"],
                                     w.page_size, w.sm_scale, selected=[[got_sel]])
            hs = slice(g * w.group_size, (g + 1) * w.group_size)
            assert np.abs(r["out"][b, hs] - out[0]).max() < tol
            assert np.abs(r["lse"][b, hs] - lse[0]).max() < 1e-4
            # split partials, split by split, against the oracle on the same partition
            toks = np.concatenate([[0], np.cumsum([oracle.valid_tokens(o["lens"][0], w.page_size, p)
                                                   for p in got_sel])]).astype(int)
            Kt = oracle.gather_tokens(o["K"], o["table"], o["lens"][0], w.page_size, 0, 0, got_sel)
            Vt = oracle.gather_tokens(o["V"], o["table"], o["lens"][0], w.page_size, 0, 0, got_sel)
            tsplits = [(toks[a], toks[e])
                       for a, e in oracle.split_ranges(len(got_sel), r["S"], w.page_size)]
            acc, ml = f64(r["acc"][b, hs]), f64(r["ml"][b, hs])
            for hi in range(w.group_size):
                m, l, a = oracle.split_partials(o["q"][0, hi], Kt, Vt, w.sm_scale, tsplits)
                live = np.isfinite(m)
                assert (np.isfinite(ml[hi, :, 0]) == live).all()
                np.testing.assert_allclose(ml[hi, live, 0], m[live], rtol=1e-5, atol=1e-5)
                np.testing.assert_allclose(ml[hi, :, 1], l, rtol=1e-4, atol=1e-6)
                np.testing.assert_allclose(acc[hi], a, rtol=1e-4, atol=1e-4 * (1 + np.abs(a).max()))


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES[:5])
def test_dense_is_the_same_kernel_with_every_page(dtype, D, G, PS):
    c = make(dtype, D, G, PS)
    w = c.workload
    kv = skv.PagedKV.from_cache(c)
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, num_splits=5)
    out, lse = skv.kv_merge_splits(acc, ml)
    # the same pages listed explicitly give bit-identical results
    n = c.pages_per_seq
    sel = torch.zeros((w.batch, w.num_kv_heads, max(n)), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32, device="cuda")
    for b in range(w.batch):
        sel[b, :, : n[b]] = torch.arange(n[b], dtype=torch.int32)
        cnt[b] = n[b]
    acc2, ml2 = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=5)
    out2, _ = skv.kv_merge_splits(acc2, ml2)
    assert_no_device_error()
    assert torch.equal(out, out2)
    q, K, V = f64(c.q), f64(c.k_pool), f64(c.v_pool)
    ref, ref_lse = oracle.attend(q, K, V, c.page_table.cpu().numpy(), c.seq_lens.cpu().numpy(),
                                 PS, w.sm_scale)
    assert np.abs(f64(out) - ref).max() < out_tol(w)
    assert np.abs(f64(lse) - ref_lse).max() < 1e-4


def test_merge_kernel_matches_oracle_merge():
    torch.manual_seed(1)
    B, Hq, S, D = 3, 4, 9, 128
    m = torch.randn((B, Hq, S)) * 5
    m[0, 0, :4] = float("-inf")
    m[1, 2, :] = float("-inf")                   # every split empty
    l = torch.rand((B, Hq, S)) * 10 + 0.1
    l[torch.isinf(m)] = 0
    acc = torch.randn((B, Hq, S, D))
    acc[torch.isinf(m)] = 0
    ml = torch.stack([m, l], dim=-1).cuda().contiguous()
    out, lse = skv.kv_merge_splits(acc.cuda().contiguous(), ml)
    out, lse = f64(out), f64(lse)
    for b in range(B):
        for h in range(Hq):
            o, e = oracle.merge_partials(m[b, h].double().numpy(), l[b, h].double().numpy(),
                                         acc[b, h].double().numpy())
            np.testing.assert_allclose(out[b, h], o, rtol=1e-5, atol=1e-6)
            if np.isfinite(e):
                assert lse[b, h] == pytest.approx(e, rel=1e-6, abs=1e-6)
            else:
                assert lse[b, h] == -np.inf


def test_fused_decode_step_equals_the_separate_calls():
    c = make("bf16", 128, 4, 16, planted=6)
    w = c.workload
    r = run_sparse(c, ratio=0.3, S=7)
    out, lse = skv.kv_decode_step(r["kv"], c.q, w.sm_scale, r["stats"], keep_ratio=0.3,
                                  num_splits=7)
    dense, _ = skv.kv_decode_step(r["kv"], c.q, w.sm_scale, keep_ratio=1.0, num_splits=7)
    acc, ml = skv.kv_sparse_decode_attn(r["kv"], c.q, w.sm_scale, num_splits=7)
    dense2, _ = skv.kv_merge_splits(acc, ml)
    assert_no_device_error()
    # same selection and partials; the merge runs in the attention kernel's last CTA
    np.testing.assert_allclose(f64(out), r["out"], rtol=0, atol=1e-6)
    np.testing.assert_allclose(f64(lse), r["lse"], rtol=0, atol=1e-6)
    np.testing.assert_allclose(f64(dense), f64(dense2), rtol=0, atol=1e-6)


def test_physical_placement_is_bit_identical():
    c = make("bf16", 128, 8, 16, planted=6)
    c2 = inputs.permute_physical(c, seed=99)
    r1 = run_sparse(c, ratio=0.3, S=4)
    r2 = run_sparse(c2, ratio=0.3, S=4)
    np.testing.assert_array_equal(r1["sel"], r2["sel"])
    np.testing.assert_array_equal(r1["out"], r2["out"])
    np.testing.assert_array_equal(r1["lse"], r2["lse"])


def test_split_count_changes_only_rounding():
    c = make("bf16", 128, 4, 16, lens=(20000,), planted=10)
    w = c.workload
    kv = skv.PagedKV.from_cache(c)
    outs = []
    for S in (1, 2, 5, 17, 64, 400):
        acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, num_splits=S)
        outs.append(f64(skv.kv_merge_splits(acc, ml)[0]))
    assert_no_device_error()
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() < 1e-5


# ------------------------------------------------------------------------------ edges

def test_edge_cases_empty_one_token_and_keep_zero():
    c = make("bf16", 128, 4, 16, lens=(0, 1, 17, 64, 65), planted=0)
    w = c.workload
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    scores = skv.kv_score_pages(kv, c.q, stats)
    keep = torch.tensor([3, 3, 0, 100, 2], dtype=torch.int32, device="cuda")
    sel, cnt = skv.kv_select_topk(scores, c.seq_lens, 16, keep=keep, k_max=8)
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=6)
    out, lse = skv.kv_merge_splits(acc, ml)
    assert_no_device_error()
    out, lse, cnt = f64(out), f64(lse), cnt.cpu().numpy()
    assert list(cnt[:, 0]) == [0, 1, 0, 4, 2]
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()      # empty sequence
    assert (out[2] == 0).all() and np.isneginf(lse[2]).all()      # nothing kept
    for b in (1, 3, 4):
        for g in range(2):
            s = sel.cpu().numpy()[b, g, : cnt[b, g]]
            o = oracle_group(c, b, g, keep_pages=int(keep[b]))
            ok, msg = oracle.check_selection(s, o["scores"], o["k"])
            assert ok, msg
            ref, ref_lse = oracle.attend(o["q"], o["K"], o["V"], o["table"], o["lens"], 16,
                                         w.sm_scale, selected=[[s]])
            hs = slice(g * 4, g * 4 + 4)
            assert np.abs(out[b, hs] - ref[0]).max() < 2e-3
    # one token: the output is that token's value row exactly (weight 1)
    P = int(c.page_table[1, 0])
    for h in range(8):
        np.testing.assert_allclose(out[1, h], f64(c.v_pool[P, h // 4, 0]), rtol=0, atol=1e-6)


def test_bad_page_table_entry_is_flagged_not_faulted():
    c = make("bf16", 128, 4, 16, lens=(500,), planted=0)
    c.page_table[0, 3] = c.num_phys_pages + 7
    c.page_table[0, 9] = -2
    w = c.workload
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    st, flags = skv.kv_check_device_errors()
    assert st == -5 and flags & 1
    skv.kv_score_pages(kv, c.q, stats)
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, num_splits=3)
    skv.kv_merge_splits(acc, ml)
    st, flags = skv.kv_check_device_errors()
    assert st == -5 and flags & 1
    # the context is still usable
    c.page_table[0, 3] = 0
    c.page_table[0, 9] = 1
    c.seq_lens[0] = 10 ** 6                      # longer than the table row
    skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, num_splits=3)
    st, flags = skv.kv_check_device_errors()
    assert st == -5 and flags & 2


def test_bounded_wait_reports_timeout_and_context_survives():
    skv.kv_selftest_wait_timeout(1_000_000)      # 1 ms on a barrier nothing completes
    st, flags = skv.kv_check_device_errors()
    assert st == -6 and flags & 16
    c = make("fp32", 64, 4, 16, lens=(300,))
    kv = skv.PagedKV.from_cache(c)
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, c.workload.sm_scale, num_splits=2)
    skv.kv_merge_splits(acc, ml)
    assert_no_device_error()


# ------------------------------------------------------------------------------ probe

@pytest.mark.parametrize("dtype,D,G,PS", SHAPES[:4])
def test_dropped_mass_matches_oracle(dtype, D, G, PS):
    c = make(dtype, D, G, PS, planted=6)
    w = c.workload
    r = run_sparse(c, ratio=0.3, S=4)
    sel_t = torch.from_numpy(r["sel"]).cuda()
    cnt_t = torch.from_numpy(r["cnt"]).cuda()
    delta = f64(skv.kv_dropped_mass(r["kv"], c.q, w.sm_scale, sel_t, cnt_t))
    assert_no_device_error()
    for b in range(w.batch):
        for g in range(w.num_kv_heads):
            q, K, V, table, lens = group_inputs(c, b, g)
            s = r["sel"][b, g, : r["cnt"][b, g]]
            ref = oracle.dropped_mass(q, K, table, lens, PS, w.sm_scale, [[s]])
            hs = slice(g * G, (g + 1) * G)
            np.testing.assert_allclose(delta[b, hs], ref[0], rtol=1e-4, atol=1e-6)
