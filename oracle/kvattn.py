"""Float64 NumPy oracle for sparse paged-KV decode attention (test infrastructure only).

Conventions shared with the library's documented interface (not with its code):

* ``k_pool``, ``v_pool``: ``[NP][Hkv][PS][D]`` -- physical page pool; page ``P`` of KV head
  ``g`` holds tokens ``0..PS-1`` of that page.
* ``page_table``: ``[B][maxP]`` integers, logical page ``p`` of sequence ``b`` lives in
  physical page ``page_table[b][p]``.
* ``seq_lens``: ``[B]`` token counts, the current decode token included.
* ``q``: ``[B][Hq][D]``; query head ``h`` reads KV head ``h // G`` with ``G = Hq // Hkv``.

Every array is widened to float64 right where it is used, so callers may hand in float32
copies of bf16 tensors (exact) without materialising a float64 copy of a large pool.

Readings taken where the pages are silent (each is also listed in the design notes):
stats and attention use only the valid tokens of a partial last page; the group score is a
sum over the group's query heads; the softmax scale is left out of the score; keep counts
round up; ties go to the lower logical page index; an empty token set gives a zero output
and lse = -inf; a split with no pages gives m = -inf, l = 0, acc = 0.
"""

from __future__ import annotations

import math

import numpy as np


# --------------------------------------------------------------------------------------
# Page geometry
# --------------------------------------------------------------------------------------

def num_pages(seq_len: int, page_size: int) -> int:
    """Logical pages of a sequence: ceil(seq_len / page_size)."""
    return -(-int(seq_len) // int(page_size))


def valid_tokens(seq_len: int, page_size: int, p: int) -> int:
    """Tokens of logical page ``p`` that lie before ``seq_len`` (0..page_size)."""
    return max(0, min(int(page_size), int(seq_len) - int(p) * int(page_size)))


# --------------------------------------------------------------------------------------
# Step a0: per-page key statistics
# --------------------------------------------------------------------------------------

def page_stats(k_pool, page_table, seq_lens, page_size):
    """Element-wise min and max of the keys of every mapped page, per KV head.

    Follows "EntmaxKV: Support-Aware Decoding for Entmax Attention", abstract: each page is
    summarised by cheap statistics that a query can score before the page is read. The
    statistic is the coordinate-wise minimum and maximum of the page's keys (the reading
    that makes the score below a true upper bound).

    Returns ``(mn, mx)``, each ``[NP][Hkv][D]`` float64. Rows of physical pages that no
    sequence maps stay NaN. Only the valid tokens of a partial last page take part.
    """
    NP, Hkv, PS, D = k_pool.shape
    assert PS == page_size
    mn = np.full((NP, Hkv, D), np.nan)
    mx = np.full((NP, Hkv, D), np.nan)
    for b in range(len(seq_lens)):
        for p in range(num_pages(seq_lens[b], PS)):
            P = int(page_table[b][p])
            v = valid_tokens(seq_lens[b], PS, p)
            keys = np.asarray(k_pool[P, :, :v, :], dtype=np.float64)   # [Hkv][v][D]
            mn[P] = keys.min(axis=1)
            mx[P] = keys.max(axis=1)
    return mn, mx


# --------------------------------------------------------------------------------------
# Step a1: query-aware page score (upper bound of q.k over the page, summed over a group)
# --------------------------------------------------------------------------------------

def page_scores(q, mn, mx, page_table, seq_lens, page_size, groups=None):
    """Score of every logical page for every KV group.

    For sequence ``b``, KV head ``g`` and logical page ``p`` (physical ``P``)::

        s[b][g][p] = sum over h in group g, sum over d of max(q[b,h,d]*mn[P,g,d],
                                                               q[b,h,d]*mx[P,g,d])

    Each inner term bounds q_d*k_d for every key of the page, so the per-head sum bounds
    q.k over the page (EntmaxKV abstract: query-aware page scoring from page statistics),
    and the per-group sum follows SparDA section 3.1 (per-head relevance summed inside a
    GQA group into one shared score). The softmax scale is left out: it does not change
    the order.

    ``groups`` optionally restricts the work to a list of ``(b, g)`` pairs.
    Returns a list over ``b`` of float64 arrays ``[Hkv][n_b]`` (NaN for groups skipped).
    """
    B, Hq, D = q.shape
    Hkv = mn.shape[1]
    G = Hq // Hkv
    out = []
    for b in range(B):
        n = num_pages(seq_lens[b], page_size)
        s = np.full((Hkv, n), np.nan)
        phys = np.asarray(page_table[b][:n], dtype=np.int64)
        for g in range(Hkv):
            if groups is not None and (b, g) not in groups:
                continue
            lo = mn[phys, g, :]                         # [n][D]
            hi = mx[phys, g, :]
            total = np.zeros(n)
            for h in range(g * G, (g + 1) * G):
                qh = np.asarray(q[b, h], dtype=np.float64)  # [D]
                total += np.maximum(qh * lo, qh * hi).sum(axis=1)
            s[g] = total
        out.append(s)
    return out


# --------------------------------------------------------------------------------------
# Step a2: keep count and top-k page selection
# --------------------------------------------------------------------------------------

def keep_count(n_pages: int, ratio: float | None = None, budget_tokens: int | None = None,
               page_size: int | None = None) -> int:
    """Pages to keep for one (sequence, KV head) group.

    A keep ratio r_KV ("Where Activation Sparsity and KV-Cache Sparsity Cross in LLM
    Decoding", Tables 16-17) keeps ceil(r * n) pages, at least one and at most n; the
    1e-9 guard keeps an exact product such as 0.5 * 2048 from rounding up past itself.
    A token budget (SparDA appendix C gives its budget in blocks) keeps
    min(n, budget_tokens // page_size) pages.
    """
    n = int(n_pages)
    if n == 0:
        return 0
    if budget_tokens is not None:
        assert page_size is not None
        return min(n, int(budget_tokens) // int(page_size))
    assert ratio is not None
    if ratio >= 1.0:
        return n
    return min(n, max(1, math.ceil(ratio * n - 1e-9)))


def select_pages(scores_1d, k: int):
    """Top-k logical pages by score, ties to the lower page index, returned ascending.

    The top-k operator of SparDA appendix A, applied to one group's page scores. Ordering is
    by (score descending, page index ascending): ``np.lexsort`` sorts by its last key first.
    """
    s = np.asarray(scores_1d, dtype=np.float64)
    n = s.shape[0]
    k = min(int(k), n)
    order = np.lexsort((np.arange(n), -s))
    return np.sort(order[:k]).astype(np.int64)


def select_structured(scores_1d, k: int, sink: int = 0, local: int = 0):
    """Forced initial and local pages joined to a top-k of the rest.

    SparDA section 3.1 describes block-sparse attention over initial blocks, a local window
    of the most recent blocks and top-k selected blocks (appendix A: B_init, B_local and
    f_top(., k) joined). Reading used here for a group of n pages and a keep count k: the
    forced set F is pages [0, sink) and [n - local, n) (clipped to [0, n)); the kept set is F
    joined with the top max(0, k - |F|) pages outside F by (score descending, page index
    ascending); the result is ascending. With sink = 0 and local = k it is the KV-window
    baseline of "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding",
    Tables 3 and 11 (keep the last pages, no scores needed).
    """
    s = np.asarray(scores_1d, dtype=np.float64)
    n = s.shape[0]
    forced = np.zeros(n, dtype=bool)
    forced[: max(0, min(int(sink), n))] = True
    if local > 0:
        forced[max(0, n - int(local)):] = True
    rest = np.nonzero(~forced)[0]
    extra = max(0, min(int(k), n) - int(forced.sum()))
    order = np.lexsort((rest, -s[rest]))
    chosen = np.concatenate([np.nonzero(forced)[0], rest[order[:extra]]])
    return np.sort(chosen).astype(np.int64)


def select_all_groups(scores, ks):
    """``select_pages`` for every (b, g): ``scores`` as returned by ``page_scores``,
    ``ks[b]`` the keep count of sequence ``b``. Returns ``sel[b][g]`` index arrays."""
    return [[select_pages(scores[b][g], ks[b]) for g in range(scores[b].shape[0])]
            for b in range(len(scores))]


# --------------------------------------------------------------------------------------
# Steps a3/a4: attention over the selected pages, split partials and their merge
# --------------------------------------------------------------------------------------

def gather_tokens(pool, page_table, seq_len, page_size, b, g, pages):
    """Valid tokens of the listed logical pages of (b, g), concatenated in list order."""
    rows = []
    for p in pages:
        P = int(page_table[b][int(p)])
        v = valid_tokens(seq_len, page_size, int(p))
        rows.append(np.asarray(pool[P, g, :v, :], dtype=np.float64))
    if not rows:
        return np.zeros((0, pool.shape[-1]))
    return np.concatenate(rows, axis=0)


def attend(q, k_pool, v_pool, page_table, seq_lens, page_size, scale, selected=None,
           groups=None):
    """Softmax attention of each decode query over the tokens of its group's pages.

    ``selected[b][g]`` lists the logical pages kept for (b, g); ``None`` keeps every page,
    which is the dense baseline ("Where Activation Sparsity and KV-Cache Sparsity Cross in
    LLM Decoding", abstract and Table 11: dense is the same attention with all pages kept).
    With x_t = scale * q.k_t and M = max x::

        o = sum_t exp(x_t - M) v_t / sum_t exp(x_t - M),   lse = M + log sum_t exp(x_t - M)

    Returns ``(out [B][Hq][D], lse [B][Hq])`` float64 (NaN for groups skipped).
    """
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    for b in range(B):
        n = num_pages(seq_lens[b], page_size)
        for g in range(Hkv):
            if groups is not None and (b, g) not in groups:
                continue
            pages = range(n) if selected is None else selected[b][g]
            K = gather_tokens(k_pool, page_table, seq_lens[b], page_size, b, g, pages)
            V = gather_tokens(v_pool, page_table, seq_lens[b], page_size, b, g, pages)
            for h in range(g * G, (g + 1) * G):
                qh = np.asarray(q[b, h], dtype=np.float64)
                if K.shape[0] == 0:
                    out[b, h] = 0.0
                    lse[b, h] = -np.inf
                    continue
                x = scale * (K @ qh)
                M = x.max()
                w = np.exp(x - M)
                L = w.sum()
                out[b, h] = (w @ V) / L
                lse[b, h] = M + np.log(L)
    return out, lse


def split_ranges(count: int, num_splits: int, page_size: int):
    """Positions of the selected-page list handled by each split.

    The list is cut into T = ceil(count / p) tiles of p = 64 / page_size pages (64 tokens);
    split ``s`` takes the whole tiles ``[floor(s*T/S), floor((s+1)*T/S))``, i.e. positions
    ``[min(count, floor(s*T/S)*p), min(count, floor((s+1)*T/S)*p))``. Runs differ by at most
    one tile; splits may be empty. This partition is part of the documented interface of the
    split-K call, so the partials can be compared split by split.
    """
    S, n = int(num_splits), int(count)
    p = 64 // int(page_size)
    T = -(-n // p) if n > 0 else 0
    return [(min(n, (s * T // S) * p), min(n, ((s + 1) * T // S) * p)) for s in range(S)]


def split_partials(q_bh, K, V, scale, token_splits):
    """(m, l, acc) of one query head for each token range of ``token_splits``.

    For the tokens t of a split: m = max x_t, l = sum exp(x_t - m), acc = sum exp(x_t - m) v_t
    with x_t = scale * q.k_t. An empty split gives (-inf, 0, 0).
    """
    qh = np.asarray(q_bh, dtype=np.float64)
    ms, ls, accs = [], [], []
    for (t0, t1) in token_splits:
        if t1 <= t0:
            ms.append(-np.inf)
            ls.append(0.0)
            accs.append(np.zeros(K.shape[1]))
            continue
        x = scale * (K[t0:t1] @ qh)
        m = x.max()
        w = np.exp(x - m)
        ms.append(m)
        ls.append(w.sum())
        accs.append(w @ V[t0:t1])
    return np.array(ms), np.array(ls), np.array(accs)


def merge_partials(m, l, acc):
    """Log-sum-exp merge of split partials into the output and its lse.

    M = max_s m_s; L = sum_s l_s exp(m_s - M); o = sum_s acc_s exp(m_s - M) / L;
    lse = M + log L. Splits with m = -inf carry no mass. All splits empty gives a zero
    output and lse = -inf. The split-K decoding of "Where Activation Sparsity and KV-Cache
    Sparsity Cross in LLM Decoding" (abstract) needs exactly this merge; the page gives no
    formula, so the standard online-softmax combination is written out.
    """
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    acc = np.asarray(acc, dtype=np.float64)
    live = np.isfinite(m)
    if not live.any():
        return np.zeros(acc.shape[-1]), -np.inf
    M = m[live].max()
    w = np.exp(m[live] - M)
    L = (l[live] * w).sum()
    o = (acc[live] * w[:, None]).sum(axis=0) / L
    return o, M + np.log(L)


# --------------------------------------------------------------------------------------
# Probe a6: dropped attention mass
# --------------------------------------------------------------------------------------

def dropped_mass(q, k_pool, page_table, seq_lens, page_size, scale, selected, groups=None):
    """Dense attention mass of the tokens whose pages were not selected.

    delta = sum_{t not selected} exp(x_t - M) / sum_{all t} exp(x_t - M), with M the max
    logit over all valid tokens ("Near-Oracle KV Selection via Pre-hoc Sparsity for
    Long-Context Inference", abstract: delta is the attention mass of the discarded
    entries; EntmaxKV abstract: the output error is controlled by delta).
    Returns ``[B][Hq]`` float64 (NaN for groups skipped; 0 for an empty sequence).
    """
    B, Hq, _ = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    delta = np.full((B, Hq), np.nan)
    for b in range(B):
        n = num_pages(seq_lens[b], page_size)
        for g in range(Hkv):
            if groups is not None and (b, g) not in groups:
                continue
            keep = np.zeros(n, dtype=bool)
            keep[np.asarray(selected[b][g], dtype=np.int64)] = True
            K = gather_tokens(k_pool, page_table, seq_lens[b], page_size, b, g, range(n))
            tok_keep = np.concatenate(
                [np.full(valid_tokens(seq_lens[b], page_size, p), keep[p]) for p in range(n)]
            ) if n else np.zeros(0, dtype=bool)
            for h in range(g * G, (g + 1) * G):
                if K.shape[0] == 0:
                    delta[b, h] = 0.0
                    continue
                x = scale * (K @ np.asarray(q[b, h], dtype=np.float64))
                w = np.exp(x - x.max())
                delta[b, h] = w[~tok_keep].sum() / w.sum()
    return delta
