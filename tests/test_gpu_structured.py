"""Structured page selection: forced first and last pages joined to the top-k of the rest,
and the score-free KV window. The index work must equal the oracle's rule exactly."""

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_cache_build_gb300 as skv

from gpu_helpers import assert_no_device_error, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("sink,local", [(0, 0), (1, 0), (0, 8), (1, 4), (4, 64), (3000, 0)])
@pytest.mark.parametrize("stride,ratio", [(300, 0.3), (2048, 0.2), (16384, 0.02), (40000, 0.1)])
def test_structured_selection_is_exact(sink, local, stride, ratio):
    torch.manual_seed(stride + sink)
    lens_list = [stride * 16, 17, 0, 5 * 16 + 3]
    B, Hkv = len(lens_list), 2
    s = (torch.round(torch.randn((B, Hkv, stride)) * 8) / 8).cuda()   # many ties
    lens = torch.tensor(lens_list, dtype=torch.int32, device="cuda")
    k_max = stride
    sel, cnt = skv.kv_select_structured(s, lens, 16, B, Hkv, stride, sink_pages=sink,
                                        local_pages=local, keep_ratio=ratio, k_max=k_max)
    assert_no_device_error()
    sel, cnt, sh = sel.cpu().numpy(), cnt.cpu().numpy(), s.double().cpu().numpy()
    for b, L in enumerate(lens_list):
        n = oracle.num_pages(L, 16)
        k = oracle.keep_count(n, ratio=ratio)
        for g in range(Hkv):
            want = oracle.select_structured(sh[b, g, :n], k, sink, local)
            assert cnt[b, g] == len(want)
            np.testing.assert_array_equal(sel[b, g, : cnt[b, g]], want)


def test_kv_window_needs_no_scores():
    lens_list = [1000, 40, 16, 0]
    B, Hkv, stride, win = len(lens_list), 3, 64, 12
    lens = torch.tensor(lens_list, dtype=torch.int32, device="cuda")
    keep = torch.zeros((B,), dtype=torch.int32, device="cuda")
    sel, cnt = skv.kv_select_structured(None, lens, 16, B, Hkv, stride, sink_pages=0,
                                        local_pages=win, keep=keep, k_max=win)
    assert_no_device_error()
    sel, cnt = sel.cpu().numpy(), cnt.cpu().numpy()
    for b, L in enumerate(lens_list):
        n = oracle.num_pages(L, 16)
        want = list(range(max(0, n - win), n))
        for g in range(Hkv):
            assert cnt[b, g] == len(want)
            assert sel[b, g, : cnt[b, g]].tolist() == want
