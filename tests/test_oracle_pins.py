"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each test checks an oracle function against brute force on tiny inputs, a closed form,
an invariant the mathematics fixes, a library routine the operation reduces to, or a
hand-worked case under tests/golden/. They are chosen so that a plausible slip in the
oracle (a dropped term, a wrong sign or index, a transposed operand, an off-by-one on a
partial page) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_kv_cache_build_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def np_(t):
    """Exact float copy of a tensor (bf16 and fp32 values are exact in float64)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def tiny_cache(G=4, Hkv=2, D=8, PS=4, lens=(37, 20, 1), dtype="fp32", seed=0, planted=0,
               extra=0, permute=True):
    w = inputs.Workload(name="t", batch=len(lens), num_q_heads=G * Hkv, num_kv_heads=Hkv,
                        head_dim=D, page_size=PS, dtype=dtype, seed=seed,
                        seq_lens=tuple(lens), planted=planted, permute_pages=permute)
    return inputs.make_cache(w, "cpu", extra_phys_pages=extra)


def unpack(c):
    return (np_(c.q), np_(c.k_pool), np_(c.v_pool), c.page_table.numpy(),
            c.seq_lens.numpy(), c.workload.page_size)


def dense_tokens(pool, table, seq_len, PS, b, g):
    """Keys or values of (b, g) in token order, gathered one token at a time."""
    rows = []
    for t in range(int(seq_len)):
        rows.append(pool[table[b][t // PS], g, t % PS, :])
    return np.array(rows).reshape(int(seq_len), pool.shape[-1])


# ----------------------------------------------------------------------------- stats

def test_stats_brute_force_loops():
    c = tiny_cache(extra=3)
    q, K, V, table, lens, PS = unpack(c)
    mn, mx = oracle.page_stats(K, table, lens, PS)
    NP, Hkv, _, D = K.shape
    seen = set()
    for b in range(len(lens)):
        for p in range(-(-int(lens[b]) // PS)):
            P = int(table[b][p])
            seen.add(P)
            for g in range(Hkv):
                for d in range(D):
                    lo = hi = None
                    for t in range(PS):
                        if p * PS + t >= lens[b]:
                            break
                        x = K[P, g, t, d]
                        lo = x if lo is None or x < lo else lo
                        hi = x if hi is None or x > hi else hi
                    assert mn[P, g, d] == lo and mx[P, g, d] == hi
    for P in range(NP):
        if P not in seen:
            assert np.isnan(mn[P]).all() and np.isnan(mx[P]).all()


def test_stats_ignore_tokens_past_the_end():
    c = tiny_cache(lens=(13,))
    q, K, V, table, lens, PS = unpack(c)
    mn0, mx0 = oracle.page_stats(K, table, lens, PS)
    K2 = K.copy()
    last = int(table[0][3])            # logical page 3 holds token 12 only
    K2[last, :, 1:, :] = 1e6
    mn1, mx1 = oracle.page_stats(K2, table, lens, PS)
    np.testing.assert_array_equal(mn0[last], mn1[last])
    np.testing.assert_array_equal(mx0[last], mx1[last])
    # a one-token page has min == max == that token
    np.testing.assert_array_equal(mn1[last], K[last, :, 0, :])
    np.testing.assert_array_equal(mx1[last], K[last, :, 0, :])


def test_stats_and_score_golden():
    case = json.load(open(os.path.join(GOLDEN, "score_cases.json")))["cases"][0]
    PS = case["page_size"]
    D = len(case["keys"][0])
    K = np.array(case["keys"], dtype=np.float64).reshape(1, 1, PS, D)
    table = np.array([[0]])
    lens = np.array([case["seq_len"]])
    mn, mx = oracle.page_stats(K, table, lens, PS)
    np.testing.assert_array_equal(mn[0, 0], case["expected_min"])
    np.testing.assert_array_equal(mx[0, 0], case["expected_max"])
    q = np.array(case["q"], dtype=np.float64)[None]          # [1][G][D], one KV head
    s = oracle.page_scores(q, mn, mx, table, lens, PS)
    assert s[0][0, 0] == case["expected_score"]
    true_max = max(sum(q[0, h] @ K[0, 0, t] for h in range(q.shape[1]))
                   for t in range(case["seq_len"]))
    assert true_max == case["expected_true_max_qk"]


# ----------------------------------------------------------------------------- score

@pytest.mark.parametrize("G", [1, 2, 4])
def test_score_equals_per_coordinate_max_over_tokens(G):
    """max(q*mn, q*mx) is the max over [mn, mx] of a linear function, attained at an actual
    token, so the score must equal sum_h sum_d max_t q[h,d]*k[t,d] (brute force)."""
    c = tiny_cache(G=G, planted=0)
    q, K, V, table, lens, PS = unpack(c)
    mn, mx = oracle.page_stats(K, table, lens, PS)
    s = oracle.page_scores(q, mn, mx, table, lens, PS)
    Hkv, D = K.shape[1], K.shape[3]
    for b in range(len(lens)):
        for g in range(Hkv):
            for p in range(-(-int(lens[b]) // PS)):
                P = int(table[b][p])
                v = min(PS, int(lens[b]) - p * PS)
                want = 0.0
                for h in range(g * G, (g + 1) * G):
                    for d in range(D):
                        want += max(q[b, h, d] * K[P, g, t, d] for t in range(v))
                assert s[b][g, p] == pytest.approx(want, rel=1e-13, abs=1e-13)


def test_score_is_an_upper_bound_of_qk_per_head_and_per_group():
    c = tiny_cache(G=4, D=16, PS=8, lens=(200, 77), planted=5)
    q, K, V, table, lens, PS = unpack(c)
    mn, mx = oracle.page_stats(K, table, lens, PS)
    s = oracle.page_scores(q, mn, mx, table, lens, PS)
    G = 4
    # per head: score each query head on its own (one-head groups over the same pages)
    for h in range(q.shape[1]):
        g = h // G
        q1 = q[:, h:h + 1, :]
        mn1, mx1 = mn[:, g:g + 1], mx[:, g:g + 1]
        s1 = oracle.page_scores(q1, mn1, mx1, table, lens, PS)
        for b in range(len(lens)):
            Kt = dense_tokens(K, table, lens[b], PS, b, g)
            for p in range(s1[b].shape[1]):
                true = (Kt[p * PS:(p + 1) * PS] @ q[b, h]).max()
                assert s1[b][0, p] >= true - 1e-12
    for b in range(len(lens)):
        for g in range(K.shape[1]):
            Kt = dense_tokens(K, table, lens[b], PS, b, g)
            qsum = q[b, g * G:(g + 1) * G].sum(axis=0)
            for p in range(s[b].shape[1]):
                assert s[b][g, p] >= (Kt[p * PS:(p + 1) * PS] @ qsum).max() - 1e-12


def test_score_unit_queries_read_out_the_statistics():
    c = tiny_cache(G=2, D=8, lens=(40,))
    q, K, V, table, lens, PS = unpack(c)
    mn, mx = oracle.page_stats(K, table, lens, PS)
    for d in range(8):
        for sign in (+1.0, -1.0):
            qq = np.zeros_like(q)
            qq[0, 0, d] = 3.0 * sign            # only head 0 of group 0 is non-zero
            s = oracle.page_scores(qq, mn, mx, table, lens, PS)
            for p in range(s[0].shape[1]):
                P = int(table[0][p])
                want = 3.0 * (mx[P, 0, d] if sign > 0 else -mn[P, 0, d])
                assert s[0][0, p] == want
                assert s[0][1, p] == 0.0


def test_score_is_tight_on_a_one_token_page():
    c = tiny_cache(G=4, lens=(4 * 5 + 1,))
    q, K, V, table, lens, PS = unpack(c)
    mn, mx = oracle.page_stats(K, table, lens, PS)
    s = oracle.page_scores(q, mn, mx, table, lens, PS)
    P = int(table[0][5])
    for g in range(K.shape[1]):
        want = sum(q[0, h] @ K[P, g, 0] for h in range(g * 4, (g + 1) * 4))
        assert s[0][g, 5] == pytest.approx(want, rel=1e-14, abs=1e-14)


# ----------------------------------------------------------------------------- select

def test_keep_count_matches_the_workloads():
    assert oracle.keep_count(16384, ratio=1 / 50) == 328        # "~328 pages per KV group"
    assert oracle.keep_count(2048, ratio=0.3) == 615
    assert oracle.keep_count(8192, ratio=0.3) == 2458
    assert oracle.keep_count(8192, ratio=0.2) == 1639
    assert oracle.keep_count(2048, ratio=0.5) == 1024           # exact product stays put
    assert oracle.keep_count(2048, ratio=1.0) == 2048
    assert oracle.keep_count(5, ratio=0.01) == 1
    assert oracle.keep_count(0, ratio=0.3) == 0
    assert oracle.keep_count(3000, budget_tokens=2048, page_size=16) == 128
    assert oracle.keep_count(100, budget_tokens=2048, page_size=16) == 100


def test_select_golden_cases():
    for case in json.load(open(os.path.join(GOLDEN, "select_cases.json")))["cases"]:
        got = oracle.select_pages(np.array(case["scores"], dtype=np.float64), case["k"])
        assert got.tolist() == case["expected"], case


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_brute_force_sort(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    s = np.round(rng.normal(size=n), 1)            # coarse values force many ties
    for k in (0, 1, n // 3, n - 1, n, n + 4):
        want = sorted(sorted(range(n), key=lambda p: (-s[p], p))[:max(0, min(k, n))])
        assert oracle.select_pages(s, k).tolist() == want


def test_tie_band_acceptance_rule():
    s = np.array([10.0, 9.0, 8.0, 8.0000001, 1.0])
    k = 3
    ok, _ = oracle.check_selection([0, 1, 3], s, k)
    assert ok
    ok, _ = oracle.check_selection([0, 1, 2], s, k)          # 8.0 is inside the band
    assert ok
    ok, _ = oracle.check_selection([0, 1, 4], s, k)          # 1.0 is far below
    assert not ok
    ok, _ = oracle.check_selection([0, 2, 3], s, k)          # 9.0 is far above, left out
    assert not ok
    ok, _ = oracle.check_selection([1, 0, 3], s, k)          # not ascending
    assert not ok


# ----------------------------------------------------------------------------- attention

def sdpa_reference(q, K, V, table, lens, PS, scale, keep_pages=None):
    """torch.nn.functional.scaled_dot_product_attention in float64, one (b, h) at a time,
    with tokens gathered one by one and unselected pages masked out."""
    B, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for g in range(Hkv):
            Kt = torch.from_numpy(dense_tokens(K, table, lens[b], PS, b, g))
            Vt = torch.from_numpy(dense_tokens(V, table, lens[b], PS, b, g))
            mask = torch.ones(int(lens[b]), dtype=torch.bool)
            if keep_pages is not None:
                mask[:] = False
                for p in keep_pages[b][g]:
                    mask[p * PS:(p + 1) * PS] = True
                mask = mask[: int(lens[b])]
            for h in range(g * G, (g + 1) * G):
                qh = torch.from_numpy(q[b, h]).view(1, 1, 1, D)
                o = torch.nn.functional.scaled_dot_product_attention(
                    qh, Kt.view(1, 1, -1, D), Vt.view(1, 1, -1, D),
                    attn_mask=mask.view(1, 1, 1, -1), scale=scale)
                out[b, h] = o.view(D).numpy()
    return out


@pytest.mark.parametrize("G,PS", [(1, 4), (4, 4), (2, 8)])
def test_dense_attention_matches_sdpa(G, PS):
    c = tiny_cache(G=G, PS=PS, D=8, lens=(37, 20, 1), planted=3)
    q, K, V, table, lens, PS = unpack(c)
    scale = 1 / math.sqrt(8)
    out, lse = oracle.attend(q, K, V, table, lens, PS, scale)
    np.testing.assert_allclose(out, sdpa_reference(q, K, V, table, lens, PS, scale),
                               rtol=1e-12, atol=1e-12)
    # lse closed form from its definition, summed token by token
    for b in range(len(lens)):
        for h in range(q.shape[1]):
            Kt = dense_tokens(K, table, lens[b], PS, b, h // G)
            want = math.log(sum(math.exp(scale * (Kt[t] @ q[b, h])) for t in range(len(Kt))))
            assert lse[b, h] == pytest.approx(want, rel=1e-12)


def test_sparse_attention_matches_masked_sdpa():
    c = tiny_cache(G=4, PS=4, D=8, lens=(37, 23), planted=2)
    q, K, V, table, lens, PS = unpack(c)
    rng = np.random.default_rng(3)
    sel = [[np.sort(rng.choice(-(-int(n) // PS), size=3, replace=False)) for _ in range(2)]
           for n in lens]
    scale = 0.3
    out, _ = oracle.attend(q, K, V, table, lens, PS, scale, selected=sel)
    np.testing.assert_allclose(out, sdpa_reference(q, K, V, table, lens, PS, scale, sel),
                               rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    case = json.load(open(os.path.join(GOLDEN, "attention_cases.json")))["attention"][0]
    K = np.array(case["keys"]).reshape(1, 1, 2, 2)
    V = np.array(case["values"]).reshape(1, 1, 2, 2)
    q = np.array(case["q"]).reshape(1, 1, 2)
    out, lse = oracle.attend(q, K, V, np.array([[0]]), np.array([2]), 2, case["scale"])
    np.testing.assert_allclose(out[0, 0], case["expected_out"], rtol=1e-14)
    assert lse[0, 0] == pytest.approx(case["expected_lse"], rel=1e-14)
    # identical keys: the output is the plain mean of the values over the valid tokens
    c = tiny_cache(G=2, lens=(10,))
    q, K, V, table, lens, PS = unpack(c)
    K[:] = 0.7
    out, lse = oracle.attend(q, K, V, table, lens, PS, 0.5)
    for g in range(2):
        Vt = dense_tokens(V, table, 10, PS, 0, g)
        for h in (2 * g, 2 * g + 1):
            np.testing.assert_allclose(out[0, h], Vt.mean(axis=0), rtol=1e-13)
            assert lse[0, h] == pytest.approx(0.5 * 0.7 * q[0, h].sum() + math.log(10))


def test_attention_ignores_tokens_past_the_end_and_empty_sequences():
    c = tiny_cache(lens=(13, 0))
    q, K, V, table, lens, PS = unpack(c)
    out0, lse0 = oracle.attend(q, K, V, table, lens, PS, 0.4)
    last = int(table[0][3])
    K[last, :, 1:, :] = 50.0
    V[last, :, 1:, :] = -50.0
    out1, lse1 = oracle.attend(q, K, V, table, lens, PS, 0.4)
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)
    assert (out0[1] == 0).all() and np.isneginf(lse0[1]).all()


# ----------------------------------------------------------------------------- merge

def test_split_ranges_partition():
    """Consecutive runs covering the list exactly; every boundary on a 64-token tile; run
    lengths in whole tiles differing by at most one (the last tile may be partial)."""
    for PS in (16, 32, 64):
        p = 64 // PS
        for count in (0, 1, 5, 33, 615, 2048):
            for S in (1, 2, 3, 7, 19, 38, 40):
                r = oracle.split_ranges(count, S, PS)
                assert len(r) == S
                assert r[0][0] == 0 and r[-1][1] == count
                for (a0, a1), (b0, b1) in zip(r, r[1:]):
                    assert a1 == b0 and a0 <= a1
                assert all(a % p == 0 for a, _ in r)
                tiles = [-(-(b - a) // p) for a, b in r]
                T = -(-count // p)
                assert sum(tiles) == T and max(tiles) - min(tiles) <= 1
    # 615 pages of 16 tokens over 38 splits: 154 tiles; floor(s*154/38) gives splits 18 and 37
    # five tiles each (pages 288-307, and 596-614 whose last tile holds 3 pages), 16 pages else
    r = oracle.split_ranges(615, 38, 16)
    assert r[18] == (288, 308) and r[-1] == (596, 615)
    assert [b - a for a, b in r].count(16) == 36


def test_merge_golden_cases():
    for case in json.load(open(os.path.join(GOLDEN, "attention_cases.json")))["merge"]:
        m = [float(x) for x in case["m"]]
        o, lse = oracle.merge_partials(m, case["l"], case["acc"])
        np.testing.assert_allclose(o, case["expected_out"], rtol=1e-14)
        assert lse == pytest.approx(case["expected_lse"], rel=1e-14)


@pytest.mark.parametrize("seed", range(4))
def test_merge_of_any_partition_equals_unsplit_attention(seed):
    rng = np.random.default_rng(seed)
    T, D = 57, 8
    Kt, Vt, qh = rng.normal(size=(T, D)), rng.normal(size=(T, D)), rng.normal(size=D)
    scale = 0.7
    x = scale * (Kt @ qh)
    w = np.exp(x - x.max())
    want = (w @ Vt) / w.sum()
    want_lse = x.max() + math.log(w.sum())
    for S in (1, 2, 5, 9):
        cuts = np.sort(rng.integers(0, T + 1, size=S - 1))
        bounds = np.concatenate([[0], cuts, [T]])
        splits = list(zip(bounds[:-1], bounds[1:]))
        splits.append((T, T))                          # an empty split
        m, l, acc = oracle.split_partials(qh, Kt, Vt, scale, splits)
        o, lse = oracle.merge_partials(m, l, acc)
        np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-13)
        assert lse == pytest.approx(want_lse, rel=1e-13)
    m, l, acc = oracle.split_partials(qh, Kt, Vt, scale, [(0, 0), (0, 0)])
    o, lse = oracle.merge_partials(m, l, acc)
    assert (o == 0).all() and lse == -np.inf


# ----------------------------------------------------------------------------- dropped mass

def test_dropped_mass_golden():
    case = json.load(open(os.path.join(GOLDEN, "attention_cases.json")))["dropped_mass"][0]
    PS = case["page_size"]
    K = np.array(case["keys"]).reshape(2, 1, PS, 1)
    table = np.array([[0, 1]])
    q = np.array(case["q"]).reshape(1, 1, 1)
    d = oracle.dropped_mass(q, K, table, np.array([4]), PS, case["scale"],
                            [[np.array(case["selected_pages"])]])
    assert d[0, 0] == pytest.approx(case["expected_delta"], rel=1e-14)


def test_dropped_mass_mixture_identity():
    """Dense attention is the delta-mixture of attention over the kept and the dropped
    tokens, so o_sparse - o_dense = delta * (o_sparse - o_dropped) exactly."""
    c = tiny_cache(G=4, PS=4, D=8, lens=(61, 30), planted=4)
    q, K, V, table, lens, PS = unpack(c)
    scale = 1 / math.sqrt(8)
    rng = np.random.default_rng(7)
    sel, rest = [], []
    for n in lens:
        n_p = -(-int(n) // PS)
        sb, rb = [], []
        for _ in range(2):
            keep = np.sort(rng.choice(n_p, size=n_p // 3, replace=False))
            sb.append(keep)
            rb.append(np.setdiff1d(np.arange(n_p), keep))
        sel.append(sb)
        rest.append(rb)
    o_sp, _ = oracle.attend(q, K, V, table, lens, PS, scale, selected=sel)
    o_dn, _ = oracle.attend(q, K, V, table, lens, PS, scale)
    o_dr, _ = oracle.attend(q, K, V, table, lens, PS, scale, selected=rest)
    delta = oracle.dropped_mass(q, K, table, lens, PS, scale, sel)
    assert ((delta > 0) & (delta < 1)).all()
    np.testing.assert_allclose(o_sp - o_dn, delta[..., None] * (o_sp - o_dr),
                               rtol=1e-10, atol=1e-12)
    full = [[np.arange(-(-int(n) // PS)) for _ in range(2)] for n in lens]
    assert (oracle.dropped_mass(q, K, table, lens, PS, scale, full) == 0).all()


def test_dropped_mass_uniform_logits_counts_tokens():
    c = tiny_cache(G=2, PS=4, lens=(23,))
    q, K, V, table, lens, PS = unpack(c)
    q[:] = 0.0                                   # every logit is 0: uniform weights
    sel = [[np.array([0, 5]), np.array([2])]]    # page 5 holds 3 valid tokens
    d = oracle.dropped_mass(q, K, table, lens, PS, 1.0, sel)
    assert d[0, 0] == pytest.approx((23 - 4 - 3) / 23, rel=1e-14)
    assert d[0, 2] == pytest.approx((23 - 4) / 23, rel=1e-14)


def test_output_error_vanishes_with_dropped_mass():
    c = tiny_cache(G=2, PS=4, D=8, lens=(40,))
    q, K, V, table, lens, PS = unpack(c)
    q[:] = 0.0
    q[0, :, 0] = 1.0
    keep = np.array([1, 4, 6])
    drop = np.setdiff1d(np.arange(10), keep)
    errs = []
    for depth in (2.0, 10.0, 30.0):
        K2 = K.copy()
        for p in drop:
            K2[int(table[0][p]), :, :, 0] = -depth   # dropped logits pushed far below
        for p in keep:
            K2[int(table[0][p]), :, :, 0] = 0.0
        sel = [[keep, keep]]
        o_sp, _ = oracle.attend(q, K2, V, table, lens, PS, 1.0, selected=sel)
        o_dn, _ = oracle.attend(q, K2, V, table, lens, PS, 1.0)
        delta = oracle.dropped_mass(q, K2, table, lens, PS, 1.0, sel)
        err = np.abs(o_sp - o_dn).max()
        assert err <= 2 * delta.max() * np.abs(V).max() + 1e-15
        errs.append(err)
    assert errs[0] > errs[1] > errs[2] and errs[2] < 1e-10


# ----------------------------------------------------------------------------- placement

def test_physical_placement_does_not_change_results():
    c = tiny_cache(G=4, PS=4, D=8, lens=(45, 17), planted=3, extra=5)
    c2 = inputs.permute_physical(c, seed=11)
    assert not torch.equal(c.page_table, c2.page_table)
    res = []
    for cc in (c, c2):
        q, K, V, table, lens, PS = unpack(cc)
        mn, mx = oracle.page_stats(K, table, lens, PS)
        s = oracle.page_scores(q, mn, mx, table, lens, PS)
        ks = [oracle.keep_count(-(-int(n) // PS), ratio=0.3) for n in lens]
        sel = oracle.select_all_groups(s, ks)
        out, lse = oracle.attend(q, K, V, table, lens, PS, 0.35, selected=sel)
        res.append((s, sel, out, lse))
    for b in range(2):
        np.testing.assert_array_equal(res[0][0][b], res[1][0][b])
    np.testing.assert_array_equal(res[0][2], res[1][2])
    np.testing.assert_array_equal(res[0][3], res[1][3])


# ----------------------------------------------------------------------------- structured

def test_structured_selection_brute_force_and_special_cases():
    rng = np.random.default_rng(5)
    for trial in range(40):
        n = int(rng.integers(1, 60))
        s = np.round(rng.normal(size=n), 1)
        k, sink, local = (int(rng.integers(0, n + 3)) for _ in range(3))
        forced = {p for p in range(n) if p < sink or p >= n - local}
        rest = sorted((p for p in range(n) if p not in forced), key=lambda p: (-s[p], p))
        want = sorted(forced | set(rest[:max(0, min(k, n) - len(forced))]))
        got = oracle.select_structured(s, k, sink, local)
        assert got.tolist() == want, (n, k, sink, local)
    s = np.arange(10, dtype=np.float64)[::-1]            # page 0 scores highest
    # no forced pages: plain top-k
    assert oracle.select_structured(s, 3).tolist() == oracle.select_pages(s, 3).tolist()
    # the KV window keeps exactly the last k pages whatever the scores
    assert oracle.select_structured(s, 4, 0, 4).tolist() == [6, 7, 8, 9]
    # sink 1 + local 2 + one scored page (page 1 is the best unforced one)
    assert oracle.select_structured(s, 4, 1, 2).tolist() == [0, 1, 8, 9]
    # forced pages beyond k are all kept
    assert oracle.select_structured(s, 1, 2, 2).tolist() == [0, 1, 8, 9]
