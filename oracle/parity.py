"""Acceptance rule for a selected page set (test infrastructure only).

A page set chosen from float32 scores may differ from the float64 oracle's only where the
scores are too close to call: two sets are accepted as equal when they agree on every page
whose oracle score lies outside a band of ``rel`` (1e-4) relative around the k-th largest
oracle score. Inside the band either choice is correct. The set must still hold exactly k
distinct pages in ascending order.
"""

from __future__ import annotations

import numpy as np


def check_selection(sel, scores_1d, k, rel=1e-4):
    """Return ``(ok, message)`` for a candidate selection ``sel`` of one group.

    ``scores_1d`` are the oracle's float64 scores of the group's pages, ``k`` its keep count.
    """
    s = np.asarray(scores_1d, dtype=np.float64)
    n = s.shape[0]
    k = min(int(k), n)
    sel = np.asarray(sel, dtype=np.int64)
    if sel.shape[0] != k:
        return False, f"selected {sel.shape[0]} pages, expected {k}"
    if k == 0:
        return True, "empty"
    if np.any(sel < 0) or np.any(sel >= n):
        return False, "page index out of range"
    if np.any(np.diff(sel) <= 0):
        return False, "indices not strictly ascending"
    order = np.lexsort((np.arange(n), -s))
    kth = s[order[k - 1]]
    band = rel * abs(kth)
    chosen = np.zeros(n, dtype=bool)
    chosen[sel] = True
    must = s > kth + band
    never = s < kth - band
    if np.any(must & ~chosen):
        bad = np.nonzero(must & ~chosen)[0][:5]
        return False, f"pages above the tie band left out: {bad.tolist()}"
    if np.any(never & chosen):
        bad = np.nonzero(never & chosen)[0][:5]
        return False, f"pages below the tie band selected: {bad.tolist()}"
    return True, "ok"
