"""Float64 oracle for entmax decoding over selected pages (test infrastructure only; see the
package header for who may import it).

The next-step row "entmax sparse attention + Gaussian-aware threshold selector", after
"EntmaxKV: Support-Aware Decoding for Entmax Attention" (abstract): alpha-entmax gives
exact zeros, so attention over selected pages is exact as soon as the selection contains
the entmax support; pages are scored against the query from page statistics before they
are read; a Gaussian-aware selector estimates the entmax threshold from those statistics,
so that the kept budget adapts to the score distribution; the dropped probability mass
delta governs the output error.

Readings taken (the page is an abstract and fixes none of these):

* alpha = 1.5. With logits x_t = scale * q . k_t and z_t = x_t / 2 (the (alpha - 1) factor),
  p_t = max(z_t - tau, 0)^2 with tau the unique value giving sum_t p_t = 1.
* Sparse entmax over a token set T normalises over T alone (tau_T). tau grows when tokens
  are added, so tau_T <= tau_all, and T holding every token with z_t > tau_all gives
  tau_T = tau_all and the full output exactly.
* Page moments for the selector, per query head h and page p (box [mn, mx] of the page's
  keys, n_p valid tokens): the upper bound zb = (scale/2) sum_d max(q_d mn_d, q_d mx_d), the
  box-centre logit c = (scale/2) q . (mn + mx)/2 and the within-page variance
  v = (scale/2)^2 sum_d q_d^2 (mx_d - mn_d)^2 / 12 (keys uniform in the box).
* Gaussian threshold: the group's tokens' z taken as N(mu, sigma^2) with mu the token-weighted
  mean of c and sigma^2 the token-weighted variance of c plus the token-weighted mean of v;
  tau_hat solves N * E[max(Z - tau, 0)^2] = 1 (N valid tokens), where for Z ~ N(mu, s^2) and
  u = (mu - tau)/s, E[max(Z - tau, 0)^2] = s^2 ((u^2 + 1) Phi(u) + u phi(u)).
* Selection: a page is kept for its (sequence, KV head) group if zb > tau_hat for some query
  head of the group, and each head's highest-bound page is always kept (the set is never
  empty); the output is ascending, as for top-k.
"""

from __future__ import annotations

import math

import numpy as np

from .kvattn import gather_tokens, num_pages, valid_tokens


def entmax15(z):
    """Exact 1.5-entmax of a 1-D array: ``(p, tau)``.

    For a support of the k largest values z_(1) >= ... >= z_(k), tau solves
    sum_{i<=k} (z_(i) - tau)^2 = 1, the smaller root tau = m - sqrt((1 - k (s - m^2)) / k)
    with m, s the mean and mean square of those k values; the support is the largest k
    whose tau lies below z_(k).
    """
    z = np.asarray(z, dtype=np.float64)
    if z.size == 0:
        return z.copy(), np.nan
    zs = np.sort(z)[::-1]
    k = np.arange(1, zs.size + 1)
    m = np.cumsum(zs) / k
    s = np.cumsum(zs * zs) / k
    disc = (1.0 - k * (s - m * m)) / k
    ok = disc >= 0
    tau_k = np.where(ok, m - np.sqrt(np.where(ok, disc, 0.0)), np.inf)
    support = np.nonzero(ok & (tau_k < zs))[0]
    tau = tau_k[support[-1]]
    p = np.maximum(z - tau, 0.0) ** 2
    return p, tau


def entmax_attend(q, k_pool, v_pool, page_table, seq_lens, page_size, scale, selected=None):
    """1.5-entmax attention of each decode query over its group's (selected) pages.

    Returns ``(out [B][Hq][D], tau [B][Hq])``; a head with no token gets out 0, tau NaN.
    """
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    tau = np.full((B, Hq), np.nan)
    for b in range(B):
        n = num_pages(seq_lens[b], page_size)
        for g in range(Hkv):
            pages = list(range(n)) if selected is None else list(selected[b][g])
            Kt = gather_tokens(k_pool, page_table, seq_lens[b], page_size, b, g, pages)
            Vt = gather_tokens(v_pool, page_table, seq_lens[b], page_size, b, g, pages)
            if Kt.shape[0] == 0:
                continue
            for h in range(g * G, (g + 1) * G):
                x = scale * (Kt @ np.asarray(q[b, h], dtype=np.float64))
                p, t = entmax15(x / 2.0)
                out[b, h] = p @ Vt
                tau[b, h] = t
    return out, tau


def entmax_dropped_mass(q, k_pool, page_table, seq_lens, page_size, scale, selected):
    """Full-entmax probability of the tokens whose pages were not selected, ``[B][Hq]``."""
    B, Hq, _ = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    delta = np.zeros((B, Hq))
    for b in range(B):
        n = num_pages(seq_lens[b], page_size)
        for g in range(Hkv):
            Kt = gather_tokens(k_pool, page_table, seq_lens[b], page_size, b, g, range(n))
            if Kt.shape[0] == 0:
                continue
            keep = np.zeros(n, dtype=bool)
            keep[np.asarray(list(selected[b][g]), dtype=np.int64)] = True
            tok_keep = np.repeat(keep, [valid_tokens(seq_lens[b], page_size, p) for p in range(n)])
            for h in range(g * G, (g + 1) * G):
                p, _ = entmax15(scale * (Kt @ np.asarray(q[b, h], dtype=np.float64)) / 2.0)
                delta[b, h] = p[~tok_keep].sum()
    return delta


def page_moments(q, mn, mx, page_table, seq_lens, page_size, scale):
    """Per query head and logical page: ``(zb, c, v, n_tok)`` as lists over b of arrays
    ``[Hq][n_b]`` (``n_tok`` ``[n_b]``) -- the upper bound, box-centre logit and within-page
    variance of z = x/2 (module readings), and the valid tokens of each page."""
    B, Hq, D = q.shape
    Hkv = mn.shape[1]
    G = Hq // Hkv
    half = scale / 2.0
    zb, c, v, nt = [], [], [], []
    for b in range(B):
        n = num_pages(seq_lens[b], page_size)
        phys = np.asarray(page_table[b][:n], dtype=np.int64)
        zb_b, c_b, v_b = np.zeros((Hq, n)), np.zeros((Hq, n)), np.zeros((Hq, n))
        for h in range(Hq):
            g = h // G
            qh = np.asarray(q[b, h], dtype=np.float64)
            lo, hi = mn[phys, g, :], mx[phys, g, :]
            zb_b[h] = half * np.maximum(qh * lo, qh * hi).sum(axis=1)
            c_b[h] = half * ((lo + hi) / 2.0) @ qh
            v_b[h] = half * half * ((hi - lo) ** 2 / 12.0) @ (qh * qh)
        zb.append(zb_b)
        c.append(c_b)
        v.append(v_b)
        nt.append(np.array([valid_tokens(seq_lens[b], page_size, p) for p in range(n)],
                           dtype=np.float64))
    return zb, c, v, nt


def gaussian_tail_sq(mu, sigma, tau):
    """E[max(Z - tau, 0)^2] for Z ~ N(mu, sigma^2) (closed form)."""
    if sigma <= 0:
        return max(mu - tau, 0.0) ** 2
    u = (mu - tau) / sigma
    Phi = 0.5 * math.erfc(-u / math.sqrt(2.0))
    phi = math.exp(-0.5 * u * u) / math.sqrt(2.0 * math.pi)
    return sigma * sigma * ((u * u + 1.0) * Phi + u * phi)


def gaussian_threshold(mu, sigma2, count):
    """tau_hat with count * E[max(Z - tau_hat, 0)^2] = 1, Z ~ N(mu, sigma2), by bisection."""
    sigma = math.sqrt(max(sigma2, 0.0))
    lo = mu - 1.0 - 40.0 * sigma            # count * E >= (mu - lo)^2 >= 1 there
    hi = mu + 40.0 * sigma + 1.0             # the tail integral is ~0 there
    if count * gaussian_tail_sq(mu, sigma, lo) < 1.0:
        return lo
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if count * gaussian_tail_sq(mu, sigma, mid) >= 1.0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def entmax_select(zb, c, v, n_tok, G):
    """Gaussian-aware selection of one sequence: ``(pages per KV group, tau_hat per head)``.

    ``zb, c, v``: ``[Hq][n]``; ``n_tok``: ``[n]``.
    """
    Hq, n = zb.shape
    Hkv = Hq // G
    tau_hat = np.full(Hq, np.nan)
    keep = np.zeros((Hkv, n), dtype=bool)
    N = n_tok.sum()
    if n == 0:
        return [np.zeros(0, dtype=np.int64) for _ in range(Hkv)], tau_hat
    for h in range(Hq):
        mu = (n_tok * c[h]).sum() / N
        var = (n_tok * (c[h] - mu) ** 2).sum() / N + (n_tok * v[h]).sum() / N
        tau_hat[h] = gaussian_threshold(mu, var, N)
        g = h // G
        keep[g] |= zb[h] > tau_hat[h]
        keep[g, int(np.argmax(zb[h]))] = True   # first maximum: the lower page index
    return [np.nonzero(keep[g])[0] for g in range(Hkv)], tau_hat
