"""Plain CPU oracle for sparse paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously-correct reference that the CUDA library is checked
against. Only the test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` may import it. The product path (the C-ABI library and its Python
binding) never imports, calls or links anything here, and this package imports nothing
from the product: the two share no code. Inputs reach both sides from the seeded input
generator, which holds none of the method's arithmetic.

Arithmetic is NumPy float64 on the exact values the GPU is given (bf16 or fp32 tensors
widened to float64). Loops are written out in the order of the method's steps; a library
primitive (a reduction, a sort, a matrix-vector product) serves as one step and nothing is
blocked, fused or reordered beyond that.

Steps and the passages they follow (page title, then section):

* ``page_stats``  -- per-page, per-KV-head element-wise min and max of the keys over the
  page's valid tokens. "EntmaxKV: Support-Aware Decoding for Entmax Attention", abstract
  (pages are scored from cheap per-page statistics before they are loaded).
* ``page_scores`` -- for each KV group, sum over its query heads and over the head
  dimension of max(q*min, q*max): an upper bound on q.k over every token of the page.
  EntmaxKV abstract (query-aware page scoring); "SparDA: Sparse Decoupled Attention for
  Efficient Long-Context LLM Inference", section 3.1 (per-head relevance is summed within
  a GQA group into one shared score).
* ``select_structured`` -- forced initial and local-window pages joined to the top-k of
  the rest (SparDA section 3.1, appendix A); the pure KV window is its score-free case
  ("Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding", Tables 3, 11).
* ``keep_count`` / ``select_pages`` -- top-k pages per KV group under a keep ratio or a
  token budget, ties to the lower page index, output ascending. "Near-Oracle KV Selection
  via Pre-hoc Sparsity for Long-Context Inference", abstract (top-k KV selection); SparDA
  appendix A (the top-k operator f_top(., k)) and appendix C (a block budget); "Where
  Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding", Tables 16-17 (keep
  ratios r_KV).
* ``attend`` / ``split_partials`` / ``merge_partials`` -- softmax attention of the decode
  query over the tokens of the selected pages, computed per split as (m, l, acc) triples
  and merged by log-sum-exp. "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM
  Decoding", abstract and Table 11 (dense and sparse decoding read the cache through one
  split-K attention kernel; dense is the same kernel with every page kept).
* ``dropped_mass`` -- the dense attention mass of the tokens not selected. "Near-Oracle KV
  Selection via Pre-hoc Sparsity for Long-Context Inference", abstract (delta, the mass of
  the discarded entries); EntmaxKV abstract (output error is governed by delta).
* ``entmax`` -- 1.5-entmax attention over selected pages, its dropped mass, per-head page
  moments and the Gaussian-aware threshold selector ("EntmaxKV: Support-Aware Decoding for
  Entmax Attention", abstract: exact zeros make sparse decoding exact once the selection
  holds the support; the selector estimates the entmax threshold from page statistics).
* ``fp8stats`` -- the page statistics stored as E4M3 bytes with one power-of-two exponent
  per row, the minimum rounded down and the maximum rounded up so that the score stays an
  upper bound ("Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding":
  a selector key cache quantised to few bits; EntmaxKV abstract: the bound).

Parity pins (tests marked ``not gpu``): bisection on tau, two-value closed forms and
numerical integration of the Gaussian tail for entmax; PyTorch's float8_e4m3fn decoding and
rounding for
the E4M3 table and the outward rounding, the exponent's defining inequalities and the
upper-bound invariant for FP8 statistics; brute-force loops for the statistics and the
selection, closed forms and the upper-bound invariant for the score, PyTorch's
``scaled_dot_product_attention`` in float64 for attention, partition invariance for the
merge, and the exact mixture identity for delta. Every function here is pinned; none is
"parity unpinned".
"""

from .kvattn import (
    num_pages,
    valid_tokens,
    page_stats,
    page_scores,
    keep_count,
    select_pages,
    select_structured,
    select_all_groups,
    gather_tokens,
    attend,
    split_ranges,
    split_partials,
    merge_partials,
    dropped_mass,
)
from .parity import check_selection
from . import entmax, fp8stats  # noqa: F401

__all__ = [
    "num_pages",
    "valid_tokens",
    "page_stats",
    "page_scores",
    "keep_count",
    "select_pages",
    "select_structured",
    "select_all_groups",
    "gather_tokens",
    "attend",
    "split_ranges",
    "split_partials",
    "merge_partials",
    "dropped_mass",
    "check_selection",
    "entmax",
    "fp8stats",
]
