"""kv_score_select (score + top-k in one launch) and kv_decode_attn_merge (split-K attention
+ merge in one launch), through the C ABI.

kv_score_select must write the scores kv_score_pages writes and the selection kv_select_topk
makes from them, bit for bit; kv_decode_attn_merge must give the outputs of
kv_sparse_decode_attn + kv_merge_splits up to float32 rounding of the merge, and the oracle's
within the bf16 bar. Both return their per-group counters to zero after every call.
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


SHAPES = [  # dtype, D, G, PS
    ("bf16", 128, 4, 16), ("bf16", 128, 8, 64), ("bf16", 128, 1, 32), ("bf16", 64, 2, 16),
    ("fp32", 64, 4, 16), ("fp32", 128, 8, 32),
]
LENS = [(1000, 4097, 37), (0, 1, 17, 65, 3000), (30000,)]
KEEPS = [dict(keep_ratio=0.3), dict(keep_ratio=0.02), dict(budget_pages=20),
         dict(keep_ratio=1.0), dict(budget_pages=100000)]


def _make(dtype, D, G, PS, lens, seed=21, Hkv=2):
    w = workload(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=PS, dtype=dtype,
                 seed=seed, seq_lens=lens, planted=5)
    return w, inputs.make_cache(w, "cuda", extra_phys_pages=2)


def _compare_with_separate_calls(kv, q, stats, lens, PS, keep, reps=2):
    ratio, budget = keep.get("keep_ratio", 0.0), keep.get("budget_pages", 0)
    k_max = skv.max_keep_pages(kv.stride, ratio if not budget else None, budget or None)
    B, Hkv = kv.batch, kv.num_kv_heads
    ctr = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
    got = None
    for _ in range(reps):                            # counters must be reusable
        scores = torch.full((B, Hkv, kv.stride), float("nan"), device="cuda")
        sel = torch.full((B, Hkv, k_max), -3, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, Hkv), -3, dtype=torch.int32, device="cuda")
        skv.kv_score_select(kv, q, stats, keep_ratio=ratio, budget_pages=budget, k_max=k_max,
                            scores=scores, counters=ctr, sel_idx=sel, sel_cnt=cnt)
        assert_no_device_error()
        assert int(ctr.abs().sum()) == 0
        now = (scores.cpu().numpy(), sel.cpu().numpy(), cnt.cpu().numpy())
        if got is not None:
            np.testing.assert_array_equal(now[1], got[1])
        got = now
    scores, sel, cnt = got
    ref_scores = skv.kv_score_pages(kv, q, stats).cpu().numpy()
    ref_sel, ref_cnt = skv.kv_select_topk(torch.from_numpy(ref_scores).cuda(), lens, PS,
                                          keep_ratio=ratio, budget_pages=budget, k_max=k_max)
    ref_sel, ref_cnt = ref_sel.cpu().numpy(), ref_cnt.cpu().numpy()
    np.testing.assert_array_equal(cnt, ref_cnt)
    lens_h = lens.cpu().numpy()
    for b in range(B):
        n = oracle.num_pages(int(lens_h[b]), PS)
        np.testing.assert_array_equal(scores[b, :, :n], ref_scores[b, :, :n])
        assert np.isnan(scores[b, :, n:]).all()         # pages past the sequence untouched
        for g in range(Hkv):
            k = int(cnt[b, g])
            np.testing.assert_array_equal(sel[b, g, :k], ref_sel[b, g, :k])
            # and the oracle's rule on these scores
            np.testing.assert_array_equal(sel[b, g, :k],
                                          oracle.select_pages(scores[b, g, :n].astype(np.float64), k))
    return scores, sel, cnt, k_max


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
@pytest.mark.parametrize("lens", LENS)
@pytest.mark.parametrize("keep", KEEPS, ids=["r0.3", "r0.02", "budget20", "all", "budget_big"])
def test_score_select_equals_the_separate_calls(dtype, D, G, PS, lens, keep):
    w, c = _make(dtype, D, G, PS, lens)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    _compare_with_separate_calls(kv, c.q, stats, c.seq_lens, PS, keep)


def test_score_select_on_tied_scores():
    """A zero query ties every page (all scores 0); a table that maps many logical pages to a
    few physical ones ties them in groups: the lower page index wins every tie."""
    w, c = _make("bf16", 128, 4, 16, (16 * 3000, 16 * 700 - 3))
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    for keep in KEEPS[:3]:
        _compare_with_separate_calls(kv, torch.zeros_like(c.q), stats, c.seq_lens, 16, keep)
    table = c.page_table.clone()
    table[:, :] = table[:, :7].repeat(1, (table.shape[1] + 6) // 7)[:, : table.shape[1]]
    kv2 = skv.PagedKV(c.k_pool, c.v_pool, table.contiguous(), c.seq_lens)
    stats2 = skv.kv_build_page_stats(kv2)
    for keep in KEEPS[:3]:
        _compare_with_separate_calls(kv2, c.q, stats2, c.seq_lens, 16, keep)


def test_score_select_long_group():
    """A 24448-page group: its keys (98 KB) in one 512-thread block's shared memory."""
    w, c = _make("bf16", 128, 4, 16, (24448 * 16, 1000 * 16 + 1), Hkv=1)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    for keep in (dict(keep_ratio=0.3), dict(budget_pages=2048)):
        _compare_with_separate_calls(kv, c.q, stats, c.seq_lens, 16, keep, reps=1)


def test_score_select_long_group_keeping_few():
    """A 5000-page group keeping 2 %: the last score block's top-k filters the keys by a
    sample first; the separate calls and the oracle's rule on the same scores agree."""
    w, c = _make("bf16", 128, 4, 16, (5000 * 16, 4500 * 16 - 5), Hkv=2)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    for keep in (dict(keep_ratio=0.02), dict(budget_pages=200)):
        _compare_with_separate_calls(kv, c.q, stats, c.seq_lens, 16, keep, reps=1)


@pytest.mark.parametrize("pages", [8191, 8192, 8193])
def test_selection_at_the_shared_memory_default(pages):
    """Groups whose keys and candidate scratch take 48 KB of dynamic shared memory, the
    per-block default (the kernels' static shared memory then needs the opt-in as well), next
    to strides that are no multiple of four (per-thread loads instead of one bulk copy)."""
    w, c = _make("bf16", 128, 4, 16, (pages * 16, 1000 * 16 + 3), Hkv=1)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    _compare_with_separate_calls(kv, c.q, stats, c.seq_lens, 16, dict(keep_ratio=0.3), reps=1)


@pytest.mark.parametrize("D,G,PS", [(128, 4, 16), (128, 8, 64), (128, 1, 32), (64, 2, 16),
                                    (64, 8, 64)])
@pytest.mark.parametrize("lens", LENS)
@pytest.mark.parametrize("S", [1, 5, 40])
@pytest.mark.parametrize("sparse", [True, False], ids=["sparse", "dense"])
def test_attn_merge_equals_the_separate_calls(D, G, PS, lens, S, sparse):
    w, c = _make("bf16", D, G, PS, lens, seed=22)
    kv = skv.PagedKV.from_cache(c)
    sel = cnt = None
    if sparse:
        stats = skv.kv_build_page_stats(kv)
        _, sel, cnt = skv.kv_score_select(kv, c.q, stats, keep_ratio=0.3)
    ctr = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        out, lse = skv.kv_decode_attn_merge(kv, c.q, w.sm_scale, sel, cnt, num_splits=S,
                                            counters=ctr)
        assert_no_device_error()
        assert int(ctr.abs().sum()) == 0
        outs.append((f64(out), f64(lse)))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    out, lse = outs[0]
    acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=S)
    out2, lse2 = skv.kv_merge_splits(acc, ml)
    np.testing.assert_allclose(out, f64(out2), rtol=0, atol=1e-6)
    fin = np.isfinite(f64(lse2))
    assert (np.isfinite(lse) == fin).all()
    np.testing.assert_allclose(lse[fin], f64(lse2)[fin], rtol=0, atol=1e-5)
    # the oracle, group by group
    sel_h = sel.cpu().numpy() if sparse else None
    cnt_h = cnt.cpu().numpy() if sparse else None
    for b, L in enumerate(lens):
        if L == 0:
            assert (out[b] == 0).all() and np.isneginf(lse[b]).all()
            continue
        for g in range(w.num_kv_heads):
            o = oracle_group(c, b, g, ratio=0.3)
            chosen = [sel_h[b, g, : cnt_h[b, g]]] if sparse else None
            ref, ref_lse = oracle.attend(o["q"], o["K"], o["V"], o["table"], o["lens"], PS,
                                         w.sm_scale, selected=[chosen] if sparse else None)
            hs = slice(g * G, (g + 1) * G)
            assert np.abs(out[b, hs] - ref[0]).max() < BF16_TOL
            assert np.abs(lse[b, hs] - ref_lse[0]).max() < 1e-4


def test_one_workspace_serves_sparse_dense_and_other_k_max():
    """Calls of different shapes share one decode-step workspace: the per-group counters sit
    where every shape finds them, so each call equals the same call on a fresh workspace."""
    w, c = _make("bf16", 128, 4, 16, (1000, 4097, 37, 0))
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    Hq = w.num_q_heads
    big = skv.kv_decode_step_workspace_size(kv, Hq, kv.stride)
    shared = torch.zeros((big,), dtype=torch.uint8, device="cuda")
    calls = [dict(keep_ratio=0.3), dict(keep_ratio=1.0), dict(budget_pages=20),
             dict(keep_ratio=0.02), dict(keep_ratio=1.0), dict(keep_ratio=0.3)]
    for kw in calls * 2:
        ratio, budget = kw.get("keep_ratio", 1.0), kw.get("budget_pages", 0)
        k_max = skv.max_keep_pages(kv.stride, ratio if not budget else None, budget or None)
        fresh = torch.zeros((skv.kv_decode_step_workspace_size(kv, Hq, k_max),),
                            dtype=torch.uint8, device="cuda")
        args = dict(stats=stats, keep_ratio=ratio, budget_pages=budget, k_max=k_max)
        ref, ref_lse = skv.kv_decode_step(kv, c.q, w.sm_scale, workspace=fresh, **args)
        got, got_lse = skv.kv_decode_step(kv, c.q, w.sm_scale, workspace=shared, **args)
        assert_no_device_error()
        assert torch.equal(got, ref), kw
        assert torch.equal(got_lse, ref_lse), kw
    n = 2 * ((w.batch * w.num_kv_heads * 4 + 255) // 256 * 256)
    assert int(shared[:n].abs().sum()) == 0              # every counter back at zero


def test_decode_step_plan_by_shape():
    """kv_decode_step's plan: bf16 groups of up to 16384 pages select inside the attention
    kernel, longer ones in the score launch, dense bf16 is the attention kernel alone, fp32
    keeps four kernels; with 8 splits or more the merge is a kernel of its own (plans 6, 7
    and 4 in place of 1, 2 and 3). The plan's kernels called one by one give kv_decode_step's
    output bit for bit."""
    cases = [("bf16", (1000, 4097, 37), 1), ("bf16", (8200 * 16,), 1), ("bf16", (16400 * 16,), 2),
             ("fp32", (1000, 37), 0), ("bf16", (2000,), 1)]
    seen = set()
    for dtype, lens, want in cases:
        w, c = _make(dtype, 128, 4, 16, lens)
        kv = skv.PagedKV.from_cache(c)
        plan, S = skv.kv_decode_step_plan(kv, w.num_q_heads, keep_ratio=0.3)
        separate = dtype == "bf16" and S >= 8
        assert plan == {1: 6, 2: 7}.get(want, want) if separate else plan == want, \
            (dtype, lens, plan, S)
        dplan, dS = skv.kv_decode_step_plan(kv, w.num_q_heads, keep_ratio=1.0)
        assert dplan == (4 if dtype != "bf16" or dS >= 8 else 3), (dplan, dS)
        seen.add(plan)
        if dtype != "bf16":
            continue
        stats = skv.kv_build_page_stats(kv)
        out, lse = skv.kv_decode_step(kv, c.q, w.sm_scale, stats, keep_ratio=0.3)
        k_max = skv.max_keep_pages(kv.stride, 0.3)
        if plan == 1:
            scores = skv.kv_score_pages(kv, c.q, stats)
            out2, lse2 = skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores, keep_ratio=0.3,
                                                   k_max=k_max, num_splits=S)
        elif plan == 2:
            _, sel, cnt = skv.kv_score_select(kv, c.q, stats, keep_ratio=0.3, k_max=k_max)
            out2, lse2 = skv.kv_decode_attn_merge(kv, c.q, w.sm_scale, sel, cnt, num_splits=S)
        else:
            # the same partials through the selected list, then the merge kernel
            if plan == 6:
                scores = skv.kv_score_pages(kv, c.q, stats)
                sel, cnt = skv.kv_select_topk(scores, c.seq_lens, 16, keep_ratio=0.3, k_max=k_max)
            else:
                _, sel, cnt = skv.kv_score_select(kv, c.q, stats, keep_ratio=0.3, k_max=k_max)
            acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=S)
            out2, lse2 = skv.kv_merge_splits(acc, ml)
        assert_no_device_error()
        assert torch.equal(out, out2) and torch.equal(lse, lse2), plan
    assert {0, 6, 7} <= seen or {0, 1, 2} <= seen, seen
