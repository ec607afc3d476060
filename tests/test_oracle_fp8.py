"""Pins of the FP8 (E4M3) page-statistics oracle against things other than itself.

* the byte table against PyTorch's float8_e4m3fn decoding (a library routine);
* outward rounding against PyTorch's round-to-nearest conversion: the nearest value is one
  of the two outward values, they bracket x, and they coincide exactly when x is on the grid;
* the row exponent against its defining inequalities, on values placed at the boundaries;
* the statistics: decoded min <= exact min, decoded max >= exact max, the brackets are one
  grid step wide, and the score from them bounds q.k over every page's tokens.
"""

import numpy as np
import pytest
import torch

from oracle import fp8stats as f8
from oracle import kvattn as K

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def torch_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def test_byte_table_matches_pytorch_e4m3fn():
    ours, ref = f8.e4m3_table(), torch_table()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def _rn(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).double().numpy()


@pytest.mark.parametrize("e", [0, -7, 5, -126])
def test_outward_rounding_brackets_round_to_nearest(e):
    rng = np.random.default_rng(7 + abs(e))
    a = np.concatenate([rng.uniform(-448, 448, 4000), rng.normal(0, 1e-2, 2000),
                        f8.e4m3_table()[np.isfinite(f8.e4m3_table())],
                        [0.0, -0.0, 448.0, -448.0, 2.0 ** -10, -(2.0 ** -10)]])
    a = a.astype(np.float32).astype(np.float64)               # values an fp32 kernel sees
    x = a * 2.0 ** e
    table = f8.e4m3_table()
    lo = table[f8.quantize_down(x, e)] * 2.0 ** e
    hi = table[f8.quantize_up(x, e)] * 2.0 ** e
    assert (lo <= x).all() and (hi >= x).all()
    on_grid = _rn(a) == a
    assert ((lo == hi) == on_grid).all()
    rn = _rn(a) * 2.0 ** e
    assert ((rn == lo) | (rn == hi)).all()
    assert (f8.quantize_down(x, e) != 0x80).all() and (f8.quantize_up(x, e) != 0x80).all()
    # lo and hi are neighbours: no grid value strictly between them
    grid = np.sort(table[np.isfinite(table)]) * 2.0 ** e
    between = np.searchsorted(grid, hi, side="left") - np.searchsorted(grid, lo, side="right")
    assert (between <= 0).all()


def test_row_exponent_inequalities():
    e_true = np.array([-126, -20, -7, -1, 0, 1, 7, 30, 100])
    m = np.concatenate([448.0 * 2.0 ** e_true,                    # exactly on the limit
                        448.0 * 2.0 ** e_true * (1 + 2.0 ** -20),  # just above: next exponent
                        [1.0, 3.0, 447.9, 448.1, 1e-30, 2.0 ** -133]])
    e = f8.row_exponent(m)
    assert (m <= 448.0 * np.exp2(e)).all()
    assert ((e == -126) | (m > 448.0 * np.exp2(e - 1))).all()
    np.testing.assert_array_equal(e[: len(e_true)], e_true)
    np.testing.assert_array_equal(e[len(e_true): 2 * len(e_true) - 1], e_true[:-1] + 1)
    assert f8.row_exponent(np.array([0.0]))[0] == 0
    assert f8.row_exponent(np.array([3.0]))[0] == -7               # 3 <= 448/128 = 3.5


def _cache(seed=0, NP=12, Hkv=2, PS=16, D=32, scale=1.0):
    rng = np.random.default_rng(seed)
    k = (rng.normal(0, 1, (NP, Hkv, PS, D)) * scale).astype(np.float32)
    k[3] *= 1e4                                                   # a page far from the others
    k[5, 0] = np.round(k[5, 0] * 4) / 4                          # on-grid values
    table = np.array([rng.permutation(NP)[:10], rng.permutation(NP)[:10]])
    lens = np.array([10 * PS - 3, 7 * PS])
    return k, table, lens


@pytest.mark.parametrize("scale", [1.0, 1e-3, 50.0])
def test_fp8_stats_contain_the_exact_box_and_bound_the_score(scale):
    k, table, lens = _cache(scale=scale)
    PS = k.shape[2]
    mn, mx = K.page_stats(k, table, lens, PS)
    cmn, cmx, e, mapped = f8.page_stats_fp8(k, table, lens, PS)
    dmn, dmx = f8.decode_stats_fp8(cmn, cmx, e, mapped)
    assert (np.isnan(mn[:, 0, 0]) == ~mapped).all()
    m = mapped
    assert (dmn[m] <= mn[m]).all() and (dmx[m] >= mx[m]).all()
    # each row fits its exponent and the exponent is the smallest that fits
    maxabs = np.maximum(np.abs(mn[m]).max(axis=2), np.abs(mx[m]).max(axis=2))
    np.testing.assert_array_equal(e[m], f8.row_exponent(maxabs))
    # one grid step at most between stored and exact values
    unit = 2.0 ** -9 * np.exp2(e[m])[:, :, None]                  # subnormal grid step
    assert (np.abs(dmn[m] - mn[m]) <= np.abs(dmn[m]) * 0.125 + unit).all()
    assert (np.abs(dmx[m] - mx[m]) <= np.abs(dmx[m]) * 0.125 + unit).all()
    # the score from FP8 statistics bounds the score from exact ones, which bounds q.k
    rng = np.random.default_rng(1)
    q = rng.normal(0, 1, (2, 4, k.shape[3]))
    s8 = K.page_scores(q, dmn, dmx, table, lens, PS)
    s = K.page_scores(q, mn, mx, table, lens, PS)
    for b in range(2):
        assert (s8[b] >= s[b] - 1e-9 * np.abs(s[b])).all()
        n = K.num_pages(lens[b], PS)
        for g in range(2):
            qsum = q[b, 2 * g: 2 * g + 2].sum(axis=0)
            for p in range(n):
                v = K.valid_tokens(lens[b], PS, p)
                true = (k[table[b][p], g, :v].astype(np.float64) @ qsum).max()
                assert s8[b][g, p] >= true - 1e-9 * abs(true)


def test_on_grid_page_is_stored_exactly():
    k, table, lens = _cache()
    PS = k.shape[2]
    k[:] = np.round(k * 4) / 4                                    # quarter steps: on grid
    cmn, cmx, e, mapped = f8.page_stats_fp8(k, table, lens, PS)
    dmn, dmx = f8.decode_stats_fp8(cmn, cmx, e, mapped)
    mn, mx = K.page_stats(k, table, lens, PS)
    m = mapped & (np.abs(mn).max(axis=(1, 2)) < 448 * 2.0 ** -2)   # rows whose scale keeps them exact
    np.testing.assert_array_equal(dmn[m], mn[m])
    np.testing.assert_array_equal(dmx[m], mx[m])
