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


def check_entmax15(E):
    """Bisection on tau and the two-value closed form (the pins above, for a planted slip)."""
    for n, scale in ((7, 1.0), (100, 0.2)):
        z = np.random.default_rng(n).normal(0, scale, n)
        p, tau = E.entmax15(z)
        assert tau == pytest.approx(bisect_tau(z), abs=1e-12)
        np.testing.assert_allclose(p, np.maximum(z - tau, 0) ** 2, atol=1e-12)
    p, tau = E.entmax15(np.array([0.3, 0.0]))
    t = (0.3 - math.sqrt(2.0 - 0.09)) / 2.0
    np.testing.assert_allclose(p, [(0.3 - t) ** 2, t * t], atol=1e-14)


def test_entmax_attend_two_tokens_closed_form():
    """One page of two tokens, q.k = a and b, V the unit rows: with z = scale * q.k / 2 the
    output is ((z1 - t)^2, (z2 - t)^2), t the two-value root (or (1, 0) when z1 - z2 >= 1)."""
    check_entmax_attend_golden(E)


def check_entmax_attend_golden(E):
    PS, D = 2, 2
    for a, b, scale in ((1.0, 0.2, 0.9), (0.5, -0.5, 0.7), (3.0, 0.0, 1.0)):
        q = np.array([[[1.0, 0.0]]])
        k = np.array([[[[a, 0.0], [b, 0.0]]]])            # [NP][Hkv][PS][D]
        v = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
        out, tau = E.entmax_attend(q, k, v, np.array([[0]]), np.array([2]), PS, scale)
        z1, z2 = scale * a / 2.0, scale * b / 2.0
        if z1 - z2 >= 1.0:
            want = [1.0, 0.0]
        else:
            t = ((z1 + z2) - math.sqrt(2.0 - (z1 - z2) ** 2)) / 2.0
            want = [(z1 - t) ** 2, (z2 - t) ** 2]
            assert tau[0, 0] == pytest.approx(t, abs=1e-14)
        np.testing.assert_allclose(out[0, 0], want, atol=1e-14)


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


# ---------------------------------------------------------------------------------------
# Pins of the selector's moments and of its token weighting (hand-worked cases, quadrature,
# Monte Carlo): a slip in the within-box variance (the 1/12, the q_d^2 weights, the
# (scale/2)^2 factor) or page- instead of token-weighting of mu and sigma^2 fails here.

import json
import os

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "entmax_cases.json")


def _one_page(q, mn, mx):
    """Arrays for page_moments: one sequence, one KV head, one query head, one full page."""
    D = len(q)
    PS = 16
    qa = np.asarray(q, dtype=np.float64).reshape(1, 1, D)
    mna = np.asarray(mn, dtype=np.float64).reshape(1, 1, D)
    mxa = np.asarray(mx, dtype=np.float64).reshape(1, 1, D)
    return qa, mna, mxa, np.array([[0]]), np.array([PS]), PS


def test_page_moments_golden():
    check_page_moments_golden(E)


def check_page_moments_golden(E):
    for case in json.load(open(GOLDEN))["moments"]:
        q, mn, mx, table, lens, PS = _one_page(case["q"], case["mn"], case["mx"])
        zb, c, v, nt = E.page_moments(q, mn, mx, table, lens, PS, case["scale"])
        assert zb[0][0, 0] == pytest.approx(case["expected_zb"], abs=1e-15)
        assert c[0][0, 0] == pytest.approx(case["expected_c"], abs=1e-15)
        assert v[0][0, 0] == pytest.approx(case["expected_v"], rel=1e-14)
        assert nt[0][0] == PS


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_page_moments_match_monte_carlo_uniform_keys(seed):
    """Keys drawn uniformly in the box, coordinate by coordinate: the sample mean and
    variance of z = (scale/2) q.k land within six standard errors of c and v. The query's
    coordinates span 0.1 to 3 in magnitude with both signs and the box widths 0 to 3, so
    weighting by |q_d| or q_d, another divisor than 12, or (scale/2) unsquared all miss."""
    check_page_moments_monte_carlo(E, seed)


def check_page_moments_monte_carlo(E, seed):
    rng = np.random.default_rng(100 + seed)
    D = 12
    q = rng.choice([-1.0, 1.0], D) * rng.uniform(0.1, 3.0, D)
    mn = rng.normal(0.0, 1.0, D)
    mx = mn + rng.uniform(0.0, 3.0, D)
    mx[0] = mn[0]                                      # one degenerate (zero-width) side
    scale = 0.35
    qa, mna, mxa, table, lens, PS = _one_page(q, mn, mx)
    zb, c, v, _ = E.page_moments(qa, mna, mxa, table, lens, PS, scale)
    n = 400_000
    keys = rng.uniform(mn, mx, size=(n, D))
    z = (scale / 2.0) * keys @ q
    se_mean = math.sqrt(v[0][0, 0] / n)
    assert abs(z.mean() - c[0][0, 0]) < 6 * se_mean
    # variance of the sample variance: (m4 - sigma^4) / n, with m4 the sample's 4th moment
    dz = z - z.mean()
    s2 = float((dz ** 2).mean())
    se_var = math.sqrt(max(float((dz ** 4).mean()) - s2 * s2, 0.0) / n)
    assert abs(s2 - v[0][0, 0]) < 6 * se_var
    assert zb[0][0, 0] >= z.max()


def _tau_by_quadrature(mu, sigma2, count):
    """tau with count * int (x - tau)^2 N(x; mu, sigma2) dx over x > tau = 1, by adaptive
    quadrature and Brent's root finder (independent of the oracle's closed form)."""
    from scipy import integrate, optimize
    s = math.sqrt(sigma2)

    def tail(t):
        f = lambda x: (x - t) ** 2 * math.exp(-0.5 * ((x - mu) / s) ** 2) / (s * math.sqrt(2 * math.pi))  # noqa: E731
        return integrate.quad(f, t, mu + 60 * s, limit=400, epsabs=1e-15, epsrel=1e-13)[0]

    return optimize.brentq(lambda t: count * tail(t) - 1.0, mu - 1.0 - 50 * s,
                           mu + 50 * s + 1.0, xtol=1e-15, rtol=1e-14)


def test_entmax_select_golden_token_weighted_threshold():
    check_select_golden(E)


def check_select_golden(E):
    for case in json.load(open(GOLDEN))["select"]:
        G = case["G"]
        zb, c, v = (np.asarray(case[k], dtype=np.float64) for k in ("zb", "c", "v"))
        nt = np.asarray(case["n_tok"], dtype=np.float64)
        assert nt.sum() == case["expected_count"]
        sel, tau_hat = E.entmax_select(zb, c, v, nt, G)
        for h in range(zb.shape[0]):
            want = _tau_by_quadrature(case["expected_mu"][h], case["expected_sigma2"][h],
                                      case["expected_count"])
            assert tau_hat[h] == pytest.approx(want, abs=1e-9)
        assert [list(map(int, pages)) for pages in sel] == [case["expected_pages"]]


def test_entmax_select_weights_pages_by_their_tokens():
    """Splitting a page into two half pages with the same box (same c and v, half the
    tokens each) changes nothing under token weighting; under page weighting it would."""
    check_token_weighting(E)


def check_token_weighting(E):
    rng = np.random.default_rng(9)
    n = 12
    c = rng.normal(0.0, 1.0, (1, n))
    v = rng.uniform(0.0, 0.2, (1, n))
    zb = c + rng.uniform(0.5, 2.0, (1, n))
    nt = rng.integers(2, 9, n).astype(np.float64) * 2.0
    _, tau = E.entmax_select(zb, c, v, nt, 1)
    split = lambda a: np.concatenate([a, a[:, :1]], axis=1)  # noqa: E731
    nt2 = np.concatenate([nt, nt[:1] / 2.0])
    nt2[0] /= 2.0
    _, tau2 = E.entmax_select(split(zb), split(c), split(v), nt2, 1)
    assert tau2[0] == pytest.approx(tau[0], abs=1e-12)
