"""The single-launch decode step (a thread-block cluster per group) against the oracle.

kv_decode_step with num_splits = KV_SPLITS_ONE_LAUNCH runs scoring, selection, attention
and the merge in one launch for bf16 caches. Its selection (read from the workspace) must equal the
oracle's rule applied to the float32 scores of kv_score_pages exactly and pass the tie band
against the float64 scores; its output must match the oracle's attention over that
selection within 2e-3 and the four-kernel path within float32 rounding. An untouched score
region of the workspace shows that the one-launch path, not the four calls, ran.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import inputs

from gpu_helpers import (BF16_TOL, assert_no_device_error, f64, need_gpu, oracle_group,
                         round256, step_score_region, step_selection, workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


SHAPES = [("bf16", 128, 4, 16), ("bf16", 128, 8, 64), ("bf16", 128, 1, 32), ("bf16", 64, 2, 16),
          ("bf16", 64, 8, 64), ("bf16", 128, 2, 16)]
LENS = [(1000, 4097, 37), (20000,), (0, 1, 17, 65, 3000)]
KEEPS = [dict(keep_ratio=0.3), dict(budget_pages=20), dict(keep_ratio=1.0), dict(keep_ratio=0.02)]


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
@pytest.mark.parametrize("lens", LENS)
@pytest.mark.parametrize("keep", KEEPS, ids=["r0.3", "budget20", "dense", "r0.02"])
def test_one_launch_step_matches_oracle(dtype, D, G, PS, lens, keep):
    Hkv = 2
    w = workload(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=PS, dtype=dtype,
                 seed=11, seq_lens=lens, planted=6)
    c = inputs.make_cache(w, "cuda", extra_phys_pages=4)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    B, Hq = w.batch, w.num_q_heads
    ratio, budget = keep.get("keep_ratio", 0.0), keep.get("budget_pages", 0)
    dense = budget <= 0 and ratio >= 1.0
    k_max = skv.max_keep_pages(kv.stride, ratio if not budget else None, budget or None)
    ws = torch.empty((skv.kv_decode_step_workspace_size(kv, Hq, k_max),), dtype=torch.uint8,
                     device="cuda")
    ws.fill_(255)
    ws[: 2 * round256(B * Hkv * 4)].zero_()           # the step's counters start at zero
    out, lse = skv.kv_decode_step(kv, c.q, w.sm_scale, stats, keep_ratio=ratio if ratio else 1.0,
                                  budget_pages=budget, k_max=k_max, workspace=ws,
                                  num_splits=skv.ONE_LAUNCH)
    assert_no_device_error()
    # one launch ran: the four-kernel path would have written the score region
    assert bool((step_score_region(ws, B, Hkv, kv.stride) == 255).all())
    out, lse = f64(out), f64(lse)

    if dense:
        ref, ref_lse = oracle.attend(f64(c.q), f64(c.k_pool), f64(c.v_pool),
                                     c.page_table.cpu().numpy(), c.seq_lens.cpu().numpy(), PS,
                                     w.sm_scale)
        assert np.abs(out - ref).max() < BF16_TOL
        fin = np.isfinite(ref_lse)
        assert (np.isfinite(lse) == fin).all()
        assert np.abs(lse[fin] - ref_lse[fin]).max() < 1e-4
        return

    sel, cnt = step_selection(ws, B, Hkv, kv.stride, k_max)
    scores = f64(skv.kv_score_pages(kv, c.q, stats))
    # the four-kernel path on the same inputs
    out4, _ = skv.kv_decode_step(kv, c.q, w.sm_scale, stats, keep_ratio=ratio if ratio else 1.0,
                                 budget_pages=budget, k_max=k_max, num_splits=3)
    assert np.abs(out - f64(out4)).max() < 1e-4
    for b, L in enumerate(lens):
        n = oracle.num_pages(L, PS)
        for g in range(Hkv):
            o = oracle_group(c, b, g, ratio=ratio if not budget else None,
                             budget_tokens=budget * PS if budget else None)
            k = o["k"]
            assert cnt[b, g] == k
            got = sel[b, g, :k]
            np.testing.assert_array_equal(got, oracle.select_pages(scores[b, g, :n], k))
            ok, msg = oracle.check_selection(got, o["scores"], k)
            assert ok, msg
            ref, ref_lse = oracle.attend(o["q"], o["K"], o["V"], o["table"], o["lens"], PS,
                                         w.sm_scale, selected=[[got]])
            hs = slice(g * G, (g + 1) * G)
            assert np.abs(out[b, hs] - ref[0]).max() < BF16_TOL
            if k > 0:
                assert np.abs(lse[b, hs] - ref_lse[0]).max() < 1e-4
            else:
                assert (out[b, hs] == 0).all() and np.isneginf(lse[b, hs]).all()
