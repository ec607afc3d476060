"""Parity at the full sizes of the five named workloads, in the launch configuration the
benchmark times (automatic split count, the fused decode step). Every group's selection --
the standalone top-k's and the one the benchmarked step itself made, read back from its
workspace -- is checked exactly against the oracle's rule on the GPU's scores; sampled groups
are checked against the oracle end to end (statistics, scores, tie band, attention over the
step's own selection, dense, delta)."""

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import inputs

from gpu_helpers import (assert_no_device_error, f64, group_inputs, need_gpu, oracle_group,
                         out_tol, round4, step_score_region, step_selection)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


def keep_args(w):
    """(list of (label, kwargs for the library, kwargs for the oracle))."""
    if w.keep_pages is not None:
        return [("top%d" % w.keep_pages, dict(keep_pages=w.keep_pages),
                 dict(keep_pages=w.keep_pages))]
    if w.budget_tokens is not None:
        bp = w.budget_tokens // w.page_size
        return [("budget%d" % bp, dict(budget_pages=bp),
                 dict(budget_tokens=w.budget_tokens))]
    return [("r%.3g" % r, dict(keep_ratio=r), dict(ratio=r)) for r in w.keep_ratios]


def sample_groups(w):
    if w.batch == 1:
        return [(0, 0), (0, w.num_kv_heads - 1)]
    return [(0, 0), (w.batch // 2, w.num_kv_heads - 1)]


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_full_size(name):
    w = inputs.WORKLOADS[name]
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    Hq, B, Hkv, PS = w.num_q_heads, w.batch, w.num_kv_heads, w.page_size
    n_pages = c.pages_per_seq
    tol = out_tol(w)
    groups = sample_groups(w)
    if name == "llama70b_1m":
        groups = groups[:1]

    # dense through the same kernel, automatic split count
    dense, dense_lse = skv.kv_decode_step(kv, c.q, w.sm_scale, keep_ratio=1.0)
    dense = f64(dense)
    assert_no_device_error()

    for label, lib_kw, or_kw in keep_args(w):
        if "keep_pages" in lib_kw:
            keep = torch.full((B,), lib_kw["keep_pages"], dtype=torch.int32, device="cuda")
            k_max = lib_kw["keep_pages"]
            sel_kw = dict(keep=keep, k_max=k_max)
        else:
            k_max = skv.max_keep_pages(kv.stride, lib_kw.get("keep_ratio"),
                                       lib_kw.get("budget_pages"))
            sel_kw = dict(keep_ratio=lib_kw.get("keep_ratio", 0.0),
                          budget_pages=lib_kw.get("budget_pages", 0), k_max=k_max)
        S = skv.kv_auto_num_splits(kv, Hq, k_max)
        scores = skv.kv_score_pages(kv, c.q, stats)
        sel, cnt = skv.kv_select_topk(scores, c.seq_lens, PS, **sel_kw)
        acc, ml = skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=S)
        out, lse = skv.kv_merge_splits(acc, ml)
        fused = step_sel = step_cnt = step_sc = None
        if "keep" not in sel_kw:
            # the step as the benchmark times it (its selection read back from the
            # workspace), and the one-launch step
            ws = torch.zeros((skv.kv_decode_step_workspace_size(kv, Hq, k_max),),
                             dtype=torch.uint8, device="cuda")
            fused, _ = skv.kv_decode_step(kv, c.q, w.sm_scale, stats, k_max=k_max,
                                          keep_ratio=lib_kw.get("keep_ratio", 1.0),
                                          budget_pages=lib_kw.get("budget_pages", 0),
                                          workspace=ws)
            torch.cuda.synchronize()
            step_sel, step_cnt = step_selection(ws, B, Hkv, kv.stride, k_max)
            r4 = round4(kv.stride)
            step_sc = f64(step_score_region(ws, B, Hkv, kv.stride).view(torch.float32)
                          [: B * Hkv * r4].view(B, Hkv, r4))
            one, _ = skv.kv_decode_step(kv, c.q, w.sm_scale, stats, k_max=k_max,
                                        keep_ratio=lib_kw.get("keep_ratio", 1.0),
                                        budget_pages=lib_kw.get("budget_pages", 0),
                                        num_splits=skv.ONE_LAUNCH)
            assert np.abs(f64(one) - f64(fused)).max() < 1e-4
            fused = f64(fused)
        sel_t, cnt_t = sel, cnt
        delta = f64(skv.kv_dropped_mass(kv, c.q, w.sm_scale, sel_t, cnt_t))
        assert_no_device_error()
        out, sel, cnt, sc = f64(out), sel.cpu().numpy(), cnt.cpu().numpy(), f64(scores)

        # every group: exact selection rule on the GPU's own scores, and the keep count
        for b in range(B):
            n = n_pages[b]
            k = (min(n, or_kw["keep_pages"]) if "keep_pages" in or_kw else
                 oracle.keep_count(n, **({"budget_tokens": w.budget_tokens, "page_size": PS}
                                         if "budget_tokens" in or_kw else or_kw)))
            for g in range(Hkv):
                assert cnt[b, g] == k
                np.testing.assert_array_equal(sel[b, g, :k], oracle.select_pages(sc[b, g, :n], k))
                if step_sel is not None:
                    assert step_cnt[b, g] == k
                    np.testing.assert_array_equal(
                        step_sel[b, g, :k], oracle.select_pages(step_sc[b, g, :n], k))
                    np.testing.assert_array_equal(step_sel[b, g, :k], sel[b, g, :k])

        # sampled groups against the oracle end to end
        for b, g in groups:
            o = oracle_group(c, b, g, **or_kw)
            n = o["scores"].shape[0]
            ref_scale = np.abs(o["scores"]).max() + 1
            np.testing.assert_allclose(sc[b, g, :n], o["scores"], rtol=2e-6, atol=2e-6 * ref_scale)
            s = sel[b, g, : cnt[b, g]]
            ok, msg = oracle.check_selection(s, o["scores"], o["k"])
            assert ok, f"{label} b={b} g={g}: {msg}"
            ref, _ = oracle.attend(o["q"], o["K"], o["V"], o["table"], o["lens"], PS,
                                   w.sm_scale, selected=[[s]])
            hs = slice(g * w.group_size, (g + 1) * w.group_size)
            err = np.abs(out[b, hs] - ref[0]).max()
            assert err < tol, f"{label} b={b} g={g}: max err {err}"
            if fused is not None:
                s_step = step_sel[b, g, : step_cnt[b, g]]
                ref_step, _ = oracle.attend(o["q"], o["K"], o["V"], o["table"], o["lens"], PS,
                                            w.sm_scale, selected=[[s_step]])
                err = np.abs(fused[b, hs] - ref_step[0]).max()
                assert err < tol, f"{label} step b={b} g={g}: max err {err}"
            d_ref = oracle.dropped_mass(o["q"], o["K"], o["table"], o["lens"], PS, w.sm_scale,
                                        [[s]])
            np.testing.assert_allclose(delta[b, hs], d_ref[0], rtol=1e-3, atol=1e-5)

    # dense and statistics on the sampled groups
    st = f64(stats)
    for b, g in groups:
        q, K, V, table, lens = group_inputs(c, b, g)
        ref, _ = oracle.attend(q, K, V, table, lens, PS, w.sm_scale)
        hs = slice(g * w.group_size, (g + 1) * w.group_size)
        err = np.abs(dense[b, hs] - ref[0]).max()
        assert err < tol, f"dense b={b} g={g}: max err {err}"
        mn, mx = oracle.page_stats(K, table, lens, PS)
        phys = c.page_table[b, : n_pages[b]].cpu().numpy()
        np.testing.assert_array_equal(st[phys, g, 0, :], mn[:, 0, :])
        np.testing.assert_array_equal(st[phys, g, 1, :], mx[:, 0, :])
