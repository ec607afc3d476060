"""Pins of the entmax oracle against things other than itself: bisection on tau, closed
forms, numerical integration, and the invariants the readings imply."""

import math

import numpy as np
import pytest

from oracle import entmax as E
from oracle import kvattn as K


def bisect_tau(z, iters=200):
    lo, hi = z.max() - 1.0, z.max()
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if (np.maximum(z - mid, 0.0) ** 2).sum() >= 1.0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


@pytest.mark.parametrize("n,scale", [(1, 1.0), (2, 0.3), (7, 1.0), (100, 0.2), (100, 3.0),
                                     (5000, 1.0), (5000, 0.01)])
def test_entmax15_matches_bisection(n, scale):
    rng = np.random.default_rng(n)
    z = rng.normal(0, scale, n)
    p, tau = E.entmax15(z)
    assert tau == pytest.approx(bisect_tau(z), abs=1e-12)
    assert (p >= 0).all() and p.sum() == pytest.approx(1.0, abs=1e-12)
    np.testing.assert_allclose(p, np.maximum(z - tau, 0) ** 2, atol=0)
    assert ((p > 0) == (z > tau)).all()


def test_entmax15_two_values_closed_form():
    for a, b in [(0.3, 0.0), (1.0, 0.0), (2.5, 0.1), (0.0, 0.0), (-1.0, -1.2)]:
        p, tau = E.entmax15(np.array([a, b]))
        if a - b >= 1.0:
            np.testing.assert_allclose(p, [1.0, 0.0], atol=1e-15)
        else:
            t = ((a + b) - math.sqrt(2.0 - (a - b) ** 2)) / 2.0
            assert tau == pytest.approx(t, abs=1e-14)
            np.testing.assert_allclose(p, [(a - t) ** 2, (b - t) ** 2], atol=1e-14)


def test_entmax15_uniform_and_translation():
    p, _ = E.entmax15(np.full(9, 0.7))
    np.testing.assert_allclose(p, np.full(9, 1 / 9), atol=1e-15)
    z = np.random.default_rng(3).normal(0, 1, 50)
    np.testing.assert_allclose(E.entmax15(z + 12.5)[0], E.entmax15(z)[0], atol=1e-12)


def _cache(seed=0, NP=24, Hkv=2, PS=16, D=32, G=2, B=2):
    rng = np.random.default_rng(seed)
    k = rng.normal(0, 1, (NP, Hkv, PS, D))
    v = rng.normal(0, 1, (NP, Hkv, PS, D))
    table = np.array([rng.permutation(NP)[:20] for _ in range(B)])
    lens = np.array([20 * PS - 5, 13 * PS])[:B]
    q = rng.normal(0, 1, (B, Hkv * G, D)) * 3.0       # sharp queries: sparse supports
    return q, k, v, table, lens, PS


def test_sparse_entmax_is_exact_once_the_support_is_selected():
    q, k, v, table, lens, PS = _cache()
    scale = 1.0 / math.sqrt(q.shape[2])
    full, tau_all = E.entmax_attend(q, k, v, table, lens, PS, scale)
    B, Hq, _ = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sel_support, sel_missing = [], []
    for b in range(B):
        n = K.num_pages(lens[b], PS)
        row_s, row_m = [], []
        for g in range(Hkv):
            keep = set()
            for h in range(g * G, (g + 1) * G):
                for p in range(n):
                    toks = k[table[b][p], g, :K.valid_tokens(lens[b], PS, p)]
                    if (scale * toks @ q[b, h] / 2 > tau_all[b, h]).any():
                        keep.add(p)
            row_s.append(np.array(sorted(keep)))
            row_m.append(np.array(sorted(keep)[1:]))          # drop one support page
        sel_support.append(row_s)
        sel_missing.append(row_m)
    out, tau = E.entmax_attend(q, k, v, table, lens, PS, scale, selected=sel_support)
    np.testing.assert_allclose(out, full, atol=1e-12)
    np.testing.assert_allclose(tau, tau_all, atol=1e-12)
    assert np.abs(E.entmax_dropped_mass(q, k, table, lens, PS, scale, sel_support)).max() < 1e-12
    out2, tau2 = E.entmax_attend(q, k, v, table, lens, PS, scale, selected=sel_missing)
    assert (tau2 <= tau_all + 1e-12).all() and (tau2 < tau_all - 1e-9).any()
    d2 = E.entmax_dropped_mass(q, k, table, lens, PS, scale, sel_missing)
    assert (d2 > 1e-9).any() and (d2 >= 0).all()
    # the output error is bounded by 2 * delta * max |v| (mixture identity of the two sets)
    assert (np.abs(out2 - full).max(axis=2) <= 2 * d2 * np.abs(v).max() + 1e-12).all()


def test_gaussian_tail_matches_integration_and_threshold_solves():
    from scipy import integrate
    for mu, sigma, tau in [(0.0, 1.0, 0.5), (1.0, 0.3, 0.2), (-2.0, 2.0, 1.0), (0.0, 1.0, -3.0)]:
        f = lambda x: max(x - tau, 0.0) ** 2 * math.exp(-0.5 * ((x - mu) / sigma) ** 2) / (sigma * math.sqrt(2 * math.pi))
        ref, _ = integrate.quad(f, tau, mu + 40 * sigma, limit=200)
        assert E.gaussian_tail_sq(mu, sigma, tau) == pytest.approx(ref, rel=1e-7, abs=1e-12)
    for mu, var, N in [(0.0, 1.0, 1000), (0.5, 0.01, 32768), (-1.0, 4.0, 16)]:
        t = E.gaussian_threshold(mu, var, N)
        assert N * E.gaussian_tail_sq(mu, math.sqrt(var), t) == pytest.approx(1.0, rel=1e-9)


def test_page_moments_bound_and_special_cases():
    q, k, v, table, lens, PS = _cache(seed=1)
    scale = 0.125
    mn, mx = K.page_stats(k, table, lens, PS)
    zb, c, var, nt = E.page_moments(q, mn, mx, table, lens, PS, scale)
    G = q.shape[1] // k.shape[1]
    for b in range(len(lens)):
        for h in range(q.shape[1]):
            for p in range(len(nt[b])):
                toks = k[table[b][p], h // G, :int(nt[b][p])]
                z = scale * toks @ q[b, h] / 2
                assert zb[b][h, p] >= z.max() - 1e-12
                assert c[b][h, p] <= zb[b][h, p] + 1e-12 and var[b][h, p] >= 0
    # a one-token page: centre = the token's z, no spread
    k1 = k.copy()
    lens1 = np.array([PS + 1, PS + 1])
    mn1, mx1 = K.page_stats(k1, table, lens1, PS)
    zb1, c1, v1, nt1 = E.page_moments(q, mn1, mx1, table, lens1, PS, scale)
    for b in range(2):
        tok = k1[table[b][1], 0, 0]
        assert c1[b][0, 1] == pytest.approx(scale * tok @ q[b, 0] / 2, abs=1e-12)
        assert zb1[b][0, 1] == pytest.approx(c1[b][0, 1], abs=1e-12) and v1[b][0, 1] == 0.0
    # a two-token page symmetric about its centre: c is the tokens' mean z
    k2 = k.copy()
    P = table[0][0]
    k2[P, 0, 1] = -k2[P, 0, 0]
    lens2 = np.array([2, 2])
    mn2, mx2 = K.page_stats(k2, table, lens2, PS)
    _, c2, _, _ = E.page_moments(q, mn2, mx2, table, lens2, PS, scale)
    assert c2[0][0, 0] == pytest.approx(0.0, abs=1e-12)


def test_entmax_select_invariants_and_adaptive_budget():
    """Tight boxes (keys N(0, 0.05^2)) with three planted pages per group aligned with the
    group's queries: the selector keeps exactly the planted pages, which hold the whole
    entmax support (no mass dropped); flat unplanted keys make it keep many more pages."""
    q, k, v, table, lens, PS = _cache(seed=2, NP=64, B=1)
    rng = np.random.default_rng(6)
    G = q.shape[1] // k.shape[1]
    flat = rng.normal(0, 0.05, k.shape)
    planted = flat.copy()
    for g in range(k.shape[1]):
        qbar = q[0, g * G:(g + 1) * G].mean(axis=0)
        for P in (3, 17, 40):
            planted[P, g] += 2.0 * qbar / np.linalg.norm(qbar)
    table = np.array([rng.permutation(64)[:60]])
    lens = np.array([60 * PS])
    kept = {}
    for name, kk in (("planted", planted), ("flat", flat)):
        mn, mx = K.page_stats(kk, table, lens, PS)
        zb, c, var, nt = E.page_moments(q, mn, mx, table, lens, PS, 0.125)
        sel, tau_hat = E.entmax_select(zb[0], c[0], var[0], nt[0], G)
        for g, pages in enumerate(sel):
            assert (np.diff(pages) > 0).all()
            for h in range(g * G, (g + 1) * G):
                assert int(np.argmax(zb[0][h])) in pages
                assert set(np.nonzero(zb[0][h] > tau_hat[h])[0]) <= set(pages)
        kept[name] = sel
        if name == "planted":
            logical = sorted(int(np.nonzero(table[0] == P)[0][0]) for P in (3, 17, 40)
                             if (table[0] == P).any())
            for pages in sel:
                assert list(pages) == logical
            delta = E.entmax_dropped_mass(q, kk, table, lens, PS, 0.125, [sel])
            assert np.abs(delta).max() < 1e-12
    assert sum(map(len, kept["flat"])) > 3 * sum(map(len, kept["planted"]))
