"""Entmax decoding (1.5-entmax over selected pages, Gaussian-aware selector) through the C ABI,
against the float64 oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import entmax as E
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import inputs

from gpu_helpers import assert_no_device_error, f64, need_gpu, out_tol, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


SHAPES = [("bf16", 128, 4, 16), ("bf16", 128, 8, 64), ("bf16", 64, 1, 32), ("fp32", 64, 4, 16),
          ("fp32", 128, 2, 32)]


def make(dtype, D, G, PS, lens=(1000, 2049, 37), seed=31, Hkv=2, planted=4):
    w = workload(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=PS, dtype=dtype,
                 seed=seed, seq_lens=lens, planted=planted)
    return w, inputs.make_cache(w, "cuda", extra_phys_pages=3)


def host(c):
    return (f64(c.q), f64(c.k_pool), f64(c.v_pool), c.page_table.cpu().numpy(),
            c.seq_lens.cpu().numpy())


def G_(w):
    return w.num_q_heads // w.num_kv_heads


def step_workspace_selection(ws, B, Hq, Hkv, stride, k_max):
    """The entmax step's selection and bounds, read back from its workspace (layout of
    kv_entmax_decode_step_workspace_size: zb, cz, vz, then sel_idx, then sel_cnt)."""
    M = (B * Hq * stride * 4 + 255) // 256 * 256
    a = 3 * M
    cb = a + (B * Hkv * k_max * 4 + 255) // 256 * 256
    sel = ws[a: a + B * Hkv * k_max * 4].view(torch.int32).view(B, Hkv, k_max).cpu()
    cnt = ws[cb: cb + B * Hkv * 4].view(torch.int32).view(B, Hkv).cpu()
    zb = ws[: B * Hq * stride * 4].view(torch.float32).view(B, Hq, stride).cpu()
    return sel, cnt, zb


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
def test_page_moments_match_oracle(dtype, D, G, PS):
    w, c = make(dtype, D, G, PS)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    zb, cz, vz = (f64(t) for t in skv.kv_entmax_page_moments(kv, c.q, stats, w.sm_scale))
    assert_no_device_error()
    q, K, V, table, lens = host(c)
    mn, mx = oracle.page_stats(K, table, lens, PS)
    rzb, rc, rv, _ = E.page_moments(q, mn, mx, table, lens, PS, w.sm_scale)
    for b in range(w.batch):
        n = rzb[b].shape[1]
        for got, ref in ((zb, rzb), (cz, rc), (vz, rv)):
            scale = np.abs(ref[b]).max() + 1e-3
            assert np.abs(got[b, :, :n] - ref[b]).max() <= 2e-6 * scale
        assert np.isnan(zb[b, :, n:]).all()


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
def test_select_is_the_oracle_rule_on_gpu_moments(dtype, D, G, PS):
    check_select_rule(*make(dtype, D, G, PS, lens=(1000, 2049, 37, 0, 5)), G, PS)


@pytest.mark.parametrize("lens", [(70003, 33000, 5, 0), (16 * 4096 * 4 + 9,)],
                         ids=["4376_pages", "16385_pages"])
def test_select_over_a_cluster_of_ctas_is_the_oracle_rule(lens):
    """Long tables: every CTA of a group's cluster holds hundreds to thousands of pages (sums
    added in rank order, kept pages placed by the lower ranks' counts, several ballot passes
    in a CTA)."""
    w, c = make("bf16", 128, 4, 16, lens=lens, seed=46, Hkv=2, planted=8)
    check_select_rule(w, c, 4, 16)


def check_select_rule(w, c, G, PS):
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    zb, cz, vz = skv.kv_entmax_page_moments(kv, c.q, stats, w.sm_scale)
    sel, cnt, tau_hat = skv.kv_entmax_select(zb, cz, vz, c.seq_lens, PS, w.num_kv_heads)
    assert_no_device_error()
    sel, cnt, tau_hat = sel.cpu().numpy(), cnt.cpu().numpy(), f64(tau_hat)
    zb, cz, vz = f64(zb), f64(cz), f64(vz)
    lens = c.seq_lens.cpu().numpy()
    for b in range(w.batch):
        n = oracle.num_pages(int(lens[b]), PS)
        if n == 0:
            assert (cnt[b] == 0).all() and np.isnan(tau_hat[b]).all()
            continue
        nt = np.array([oracle.valid_tokens(int(lens[b]), PS, p) for p in range(n)], dtype=float)
        ref_sel, ref_tau = E.entmax_select(zb[b, :, :n], cz[b, :, :n], vz[b, :, :n], nt, G)
        # the GPU estimates in float (the oracle in float64): agreement to float level
        np.testing.assert_allclose(tau_hat[b], ref_tau, rtol=2e-5, atol=2e-5)
        for g in range(w.num_kv_heads):
            got = set(sel[b, g, : cnt[b, g]].tolist())
            want = set(ref_sel[g].tolist())
            assert (np.diff(sel[b, g, : cnt[b, g]]) > 0).all()
            # decisions may differ only for pages whose bound is within the band of tau_hat
            heads = range(g * G, (g + 1) * G)
            band = {p for p in range(n) for h in heads
                    if abs(zb[b, h, p] - ref_tau[h]) <= 2e-5 * (abs(ref_tau[h]) + 1.0)}
            assert got ^ want <= band, (got ^ want, band)


@pytest.mark.parametrize("dtype,D,G,PS", SHAPES)
@pytest.mark.parametrize("sparse", [True, False], ids=["selected", "dense"])
def test_entmax_attention_matches_oracle(dtype, D, G, PS, sparse):
    w, c = make(dtype, D, G, PS, lens=(1000, 2049, 37, 0, 1))
    kv = skv.PagedKV.from_cache(c)
    sel = cnt = None
    if sparse:
        stats = skv.kv_build_page_stats(kv)
        zb, cz, vz = skv.kv_entmax_page_moments(kv, c.q, stats, w.sm_scale)
        sel, cnt, _ = skv.kv_entmax_select(zb, cz, vz, c.seq_lens, PS, w.num_kv_heads)
    outs = [skv.kv_entmax_decode_attn(kv, c.q, w.sm_scale, sel, cnt) for _ in range(2)]
    assert_no_device_error()
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1].nan_to_num(7.0), outs[1][1].nan_to_num(7.0))   # NaN: empty
    out, tau = f64(outs[0][0]), f64(outs[0][1])
    q, K, V, table, lens = host(c)
    chosen = None
    if sparse:
        s_, n_ = sel.cpu().numpy(), cnt.cpu().numpy()
        chosen = [[s_[b, g, : n_[b, g]] for g in range(w.num_kv_heads)] for b in range(w.batch)]
    ref, ref_tau = E.entmax_attend(q, K, V, table, lens, PS, w.sm_scale, selected=chosen)
    for b in range(w.batch):
        if lens[b] == 0:
            assert (out[b] == 0).all() and np.isnan(tau[b]).all()
            continue
        assert np.abs(out[b] - ref[b]).max() < out_tol(w)
        assert np.abs(tau[b] - ref_tau[b]).max() < (1e-4 if dtype == "bf16" else 1e-5)


def test_selected_support_makes_sparse_entmax_exact():
    """The pages holding the dense entmax support (found by the oracle), plus unrelated
    pages, give the dense output: sparse entmax is exact once the support is selected."""
    w, c = make("bf16", 128, 4, 16, lens=(3000, 1600), seed=41, planted=16)
    q, K, V, table, lens = host(c)
    scale = w.sm_scale
    _, tau_all = E.entmax_attend(q, K, V, table, lens, 16, scale)
    B, Hkv, G = w.batch, w.num_kv_heads, w.group_size
    rng = np.random.default_rng(0)
    chosen = []
    for b in range(B):
        n = oracle.num_pages(int(lens[b]), 16)
        row = []
        for g in range(Hkv):
            keep = set(rng.choice(n, 5, replace=False).tolist())
            for h in range(g * G, (g + 1) * G):
                for p in range(n):
                    toks = K[table[b][p], g, :oracle.valid_tokens(int(lens[b]), 16, p)]
                    if (scale * toks @ q[b, h] / 2 > tau_all[b, h]).any():
                        keep.add(p)
            row.append(np.array(sorted(keep), dtype=np.int32))
        chosen.append(row)
    k_max = max(len(r) for row in chosen for r in row)
    sel = np.zeros((B, Hkv, k_max), dtype=np.int32)
    cnt = np.zeros((B, Hkv), dtype=np.int32)
    for b in range(B):
        for g in range(Hkv):
            sel[b, g, : len(chosen[b][g])] = chosen[b][g]
            cnt[b, g] = len(chosen[b][g])
    assert cnt.max() < oracle.num_pages(int(lens.max()), 16)      # a real subset
    out, tau = skv.kv_entmax_decode_attn(kv := skv.PagedKV.from_cache(c), c.q, scale,
                                         torch.from_numpy(sel).cuda(), torch.from_numpy(cnt).cuda())
    dense, dtau = skv.kv_entmax_decode_attn(kv, c.q, scale)
    assert_no_device_error()
    np.testing.assert_allclose(f64(out), f64(dense), rtol=0, atol=2e-6)
    np.testing.assert_allclose(f64(tau), f64(dtau), rtol=0, atol=2e-6)


def test_selector_adapts_to_gaussian_scores():
    """Keys whose page means vary widely with tight pages (the regime of the Gaussian reading):
    the one-call step keeps a strict subset of pages, the same set kv_entmax_select gives, and
    its output is entmax over that set."""
    w, c = make("bf16", 128, 4, 16, lens=(4000, 2500), seed=43, planted=0)
    g_ = torch.Generator(device="cuda").manual_seed(43)
    NP, Hkv, PS, D = c.k_pool.shape
    page_mean = torch.randn((NP, Hkv, 1, D), generator=g_, device="cuda")
    k = page_mean + 0.02 * torch.randn((NP, Hkv, PS, D), generator=g_, device="cuda")
    c.k_pool.copy_(k.to(c.k_pool.dtype))
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    k_max = kv.stride
    ws = torch.empty((skv.kv_entmax_decode_step_workspace_size(kv, w.num_q_heads, k_max),),
                     dtype=torch.uint8, device="cuda")
    out, tau = skv.kv_entmax_decode_step(kv, c.q, w.sm_scale, stats, k_max=k_max, workspace=ws)
    torch.cuda.synchronize()
    B, Hq = w.batch, w.num_q_heads
    step_sel, step_cnt, step_zb = step_workspace_selection(ws, B, Hq, Hkv, kv.stride, k_max)
    zb, cz, vz = skv.kv_entmax_page_moments(kv, c.q, stats, w.sm_scale)
    sel, cnt, tau_hat = skv.kv_entmax_select(zb, cz, vz, c.seq_lens, 16, Hkv, k_max=k_max)
    out2, tau2 = skv.kv_entmax_decode_attn(kv, c.q, w.sm_scale, step_sel.cuda(), step_cnt.cuda())
    assert_no_device_error()
    # the step's own moments are the public kernel's, bit for bit; its kept pages are the public
    # selector's up to pages whose bound sits at tau_hat (a different summation order)
    for b in range(B):
        n_b = oracle.num_pages(int(c.seq_lens[b]), 16)
        assert torch.equal(step_zb[b, :, :n_b], zb.cpu()[b, :, :n_b])
    th = tau_hat.cpu().numpy()
    zbh = zb.cpu().numpy()
    for b in range(B):
        for g in range(Hkv):
            got = set(step_sel[b, g, : step_cnt[b, g]].tolist())
            want = set(sel[b, g, : cnt[b, g]].tolist())
            for p_ in got ^ want:
                near = np.abs(zbh[b, g * G_(w): (g + 1) * G_(w), p_] - th[b, g * G_(w): (g + 1) * G_(w)])
                assert near.min() <= 1e-5 * (np.abs(th[b]).max() + 1), (b, g, p_)
    # and its output is the attention over exactly the pages it kept
    assert torch.equal(out, out2) and torch.equal(tau, tau2)
    sel, cnt = step_sel.cuda(), step_cnt.cuda()
    cnt_h = cnt.cpu().numpy()
    for b in range(B):
        n = oracle.num_pages(int(c.seq_lens[b]), 16)
        assert (cnt_h[b] > 0).all() and (cnt_h[b] < n // 2).all(), cnt_h[b]
    q, K, V, table, lens = host(c)
    s_ = sel.cpu().numpy()
    chosen = [[s_[b, g, : cnt_h[b, g]] for g in range(Hkv)] for b in range(B)]
    ref, ref_tau = E.entmax_attend(q, K, V, table, lens, 16, w.sm_scale, selected=chosen)
    assert np.abs(f64(out) - ref).max() < 2e-3
    delta = E.entmax_dropped_mass(q, K, table, lens, 16, w.sm_scale, chosen)
    print(f"kept {cnt_h.sum()} of {sum(oracle.num_pages(int(x), 16) for x in lens) * Hkv} "
          f"pages, entmax dropped mass max {delta.max():.3g} mean {delta.mean():.3g}")


def test_flat_logits_take_the_global_candidate_path():
    """A zero query ties every logit: every token is a candidate (more than the shared-memory
    buffer holds) and entmax is uniform: out = mean of V, tau = -1/sqrt(n)."""
    w, c = make("bf16", 128, 4, 16, lens=(20000 + 7,), seed=44, planted=0)
    kv = skv.PagedKV.from_cache(c)
    q0 = torch.zeros_like(c.q)
    out, tau = skv.kv_entmax_decode_attn(kv, q0, w.sm_scale)
    assert_no_device_error()
    n = 20007
    q, K, V, table, lens = host(c)
    for g in range(w.num_kv_heads):
        Vt = oracle.gather_tokens(V, table, n, 16, 0, g, range(oracle.num_pages(n, 16)))
        mean = Vt.mean(axis=0)
        for h in range(g * w.group_size, (g + 1) * w.group_size):
            assert np.abs(f64(out)[0, h] - mean).max() < 1e-5
            assert f64(tau)[0, h] == pytest.approx(-1 / math.sqrt(n), abs=1e-6)


def test_entmax_step_prunes_tight_boxes_and_matches_oracle():
    """Keys tight around per-page means (the pruning workload's recipe at 4096 tokens): the
    Gaussian-aware selector keeps few pages, and the step's output is the oracle's entmax
    over exactly the pages it kept."""
    w = inputs.workload("entmax_pruning_32k", seq_len=4096, num_q_heads=8, num_kv_heads=2)
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    B, Hq, Hkv = w.batch, w.num_q_heads, w.num_kv_heads
    ws = torch.zeros((skv.kv_entmax_decode_step_workspace_size(kv, Hq, kv.stride),),
                     dtype=torch.uint8, device="cuda")
    out, tau = skv.kv_entmax_decode_step(kv, c.q, w.sm_scale, stats, k_max=kv.stride,
                                         workspace=ws)
    torch.cuda.synchronize()
    assert_no_device_error()
    M = (B * Hq * kv.stride * 4 + 255) // 256 * 256
    a = 3 * M
    cb = a + (B * Hkv * kv.stride * 4 + 255) // 256 * 256
    sel = ws[a: a + B * Hkv * kv.stride * 4].view(torch.int32).view(B, Hkv, kv.stride).cpu()
    cnt = ws[cb: cb + B * Hkv * 4].view(torch.int32).view(B, Hkv).cpu().numpy()
    n = kv.stride
    assert 0 < cnt.max() and cnt.sum() < 0.5 * B * Hkv * n, cnt
    chosen = [[sel[b, g, : cnt[b, g]].numpy() for g in range(Hkv)] for b in range(B)]
    q, K, V, table, lens = host(c)
    ref, ref_tau = E.entmax_attend(q, K, V, table, lens, w.page_size, w.sm_scale,
                                   selected=chosen)
    assert np.abs(f64(out) - ref).max() < out_tol(w)
    assert np.abs(f64(tau) - ref_tau).max() < 1e-4


def test_one_outlier_over_flat_logits():
    """One token well above thousands of tied logits: the threshold's closed form is taken about
    a pivot near the members' mean, not the outlier, so tau and the output keep float accuracy
    (sum y^2 - K mean^2 would otherwise cancel)."""
    w, c = make("bf16", 128, 4, 16, lens=(6000,), seed=45, planted=0)
    kv = skv.PagedKV.from_cache(c)
    n = 6000
    # q along the first coordinate only; every key zero there except one token's
    q0 = torch.zeros_like(c.q)
    q0[..., 0] = 1.0
    table = c.page_table[0].cpu().numpy()
    c.k_pool[:, :, :, 0] = 0
    j = 4321
    big = 2 * 0.9 / w.sm_scale                    # z_j = sm_scale * q . k_j / 2 = 0.9
    c.k_pool[table[j // 16], :, j % 16, 0] = big
    out, tau = skv.kv_entmax_decode_attn(kv, q0, w.sm_scale)
    assert_no_device_error()
    q, K, V, tab, lens = host(c)
    ref, ref_tau = E.entmax_attend(f64(q0), K, V, tab, lens, 16, w.sm_scale)
    assert np.abs(f64(tau) - ref_tau).max() < 2e-6
    assert np.abs(f64(out) - ref).max() < out_tol(w)
