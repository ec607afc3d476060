"""Float64 oracle for FP8 (E4M3) page statistics with outward rounding (test infrastructure
only; see the package header for who may import it).

The next-step row "compressed page statistics": the per-page key minimum and maximum of
``kvattn.page_stats`` stored as one byte each, so that the score pass reads half the bytes
of bf16 statistics. Motivation: "Where Activation Sparsity and KV-Cache Sparsity Cross in
LLM Decoding" (the selector's key cache quantised to few bits); the score of
"EntmaxKV: Support-Aware Decoding for Entmax Attention" (abstract) stays an upper bound only
if the stored box contains the true one, hence the outward rounding.

Readings taken (the pages fix no format):

* E4M3 is the OCP "FN" byte: sign bit, four exponent bits with bias 7, three mantissa bits;
  exponent field 0 holds subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no infinity;
  the largest finite magnitude is 448.
* Each (physical page, KV head) row of 2*D statistics carries one power-of-two exponent e,
  the smallest integer with max|x| <= 448 * 2^e over the row (0 for an all-zero row), never
  below -126. The stored value of a byte c is value(c) * 2^e.
* The minimum is stored as the largest E4M3 value <= x / 2^e and the maximum as the smallest
  E4M3 value >= x / 2^e ("outward"), so that decoded mn <= true mn and decoded mx >= true mx.
  Zero is stored as the +0 byte 0x00, never as -0 (0x80).
"""

from __future__ import annotations

import numpy as np

from .kvattn import page_stats

E4M3_MAX = 448.0
MIN_EXPONENT = -126


def e4m3_value(code: int) -> float:
    """Value of one E4M3 byte, from the bit fields (NaN for the two NaN bytes)."""
    sign = -1.0 if code & 0x80 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return float("nan")
    if exp_field == 0:
        return sign * (mant / 8.0) * 2.0 ** -6
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


def e4m3_table() -> np.ndarray:
    """float64 value of every byte 0..255."""
    return np.array([e4m3_value(c) for c in range(256)])


def _ladder():
    """Finite values in ascending order and the byte of each (+0 stands for zero)."""
    vals, codes = [], []
    for c in range(256):
        v = e4m3_value(c)
        if np.isnan(v) or c == 0x80:
            continue
        vals.append(v)
        codes.append(c)
    order = np.argsort(vals, kind="stable")
    return np.asarray(vals)[order], np.asarray(codes, dtype=np.uint8)[order]


def row_exponent(maxabs) -> np.ndarray:
    """Smallest integer e >= -126 with maxabs <= 448 * 2^e (0 where maxabs == 0)."""
    m = np.asarray(maxabs, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.ceil(np.log2(np.where(m > 0, m, 1.0) / E4M3_MAX))
    e = e.astype(np.int64)
    # make the defining inequalities hold exactly (log2 may be off by one ulp)
    e = np.where(m > E4M3_MAX * np.exp2(e.astype(np.float64)), e + 1, e)
    e = np.where(m <= E4M3_MAX * np.exp2((e - 1).astype(np.float64)), e - 1, e)
    e = np.maximum(e, MIN_EXPONENT)
    return np.where(m > 0, e, 0)


def quantize_down(x, e) -> np.ndarray:
    """Byte of the largest E4M3 value v with v * 2^e <= x (x finite, |x| <= 448 * 2^e)."""
    vals, codes = _ladder()
    a = np.asarray(x, dtype=np.float64) / np.exp2(np.asarray(e, dtype=np.float64))
    idx = np.searchsorted(vals, a, side="right") - 1
    assert (idx >= 0).all(), "value below -448 * 2^e"
    return codes[idx]


def quantize_up(x, e) -> np.ndarray:
    """Byte of the smallest E4M3 value v with v * 2^e >= x (x finite, |x| <= 448 * 2^e)."""
    vals, codes = _ladder()
    a = np.asarray(x, dtype=np.float64) / np.exp2(np.asarray(e, dtype=np.float64))
    idx = np.searchsorted(vals, a, side="left")
    assert (idx < len(vals)).all(), "value above 448 * 2^e"
    return codes[idx]


def page_stats_fp8(k_pool, page_table, seq_lens, page_size):
    """FP8 statistics of every mapped page: ``(code_mn, code_mx, exponent, mapped)``.

    ``code_mn``/``code_mx`` are ``[NP][Hkv][D]`` uint8, ``exponent`` ``[NP][Hkv]`` int64 and
    ``mapped`` ``[NP]`` bool (rows of pages no sequence maps are left 0 and unmapped).
    """
    mn, mx = page_stats(k_pool, page_table, seq_lens, page_size)
    mapped = ~np.isnan(mn[:, 0, 0])
    NP, Hkv, D = mn.shape
    code_mn = np.zeros((NP, Hkv, D), dtype=np.uint8)
    code_mx = np.zeros((NP, Hkv, D), dtype=np.uint8)
    exponent = np.zeros((NP, Hkv), dtype=np.int64)
    rows = np.nonzero(mapped)[0]
    if rows.size:
        lo, hi = mn[rows], mx[rows]                                     # [r][Hkv][D]
        maxabs = np.maximum(np.abs(lo).max(axis=2), np.abs(hi).max(axis=2))
        e = row_exponent(maxabs)                                        # [r][Hkv]
        code_mn[rows] = quantize_down(lo, e[:, :, None])
        code_mx[rows] = quantize_up(hi, e[:, :, None])
        exponent[rows] = e
    return code_mn, code_mx, exponent, mapped


def decode_stats_fp8(code_mn, code_mx, exponent, mapped):
    """float64 ``(mn, mx)`` ``[NP][Hkv][D]`` that FP8 statistics stand for (NaN where unmapped),
    in the form ``kvattn.page_scores`` takes."""
    table = e4m3_table()
    scale = np.exp2(np.asarray(exponent, dtype=np.float64))[:, :, None]
    mn = table[np.asarray(code_mn)] * scale
    mx = table[np.asarray(code_mx)] * scale
    mn[~mapped] = np.nan
    mx[~mapped] = np.nan
    return mn, mx
