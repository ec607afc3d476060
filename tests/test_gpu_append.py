"""Token append with incremental page statistics (the cache grows one token per step).

After appending tokens one by one, across page boundaries and from an empty sequence, the
incrementally maintained statistics must equal both a full rebuild on the GPU and the
float64 oracle's statistics of the grown cache, bit for bit, and the appended rows must sit
in the pool at their positions.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_cache_build_gb300 as skv
from sparse_kv_cache_build_gb300 import inputs

from gpu_helpers import assert_no_device_error, f64, need_gpu, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype,D,G,PS", [("bf16", 128, 4, 16), ("fp32", 64, 2, 32),
                                          ("bf16", 64, 8, 64)])
def test_append_keeps_statistics_equal_to_a_rebuild(dtype, D, G, PS):
    start = (100, 15, 0, 31)
    grow = 40
    final = tuple(n + grow for n in start)
    w = workload(num_q_heads=G * 2, num_kv_heads=2, head_dim=D, page_size=PS, dtype=dtype,
                 seed=5, seq_lens=final)
    c = inputs.make_cache(w, "cuda", extra_phys_pages=3)     # every final page is mapped
    c.seq_lens.copy_(torch.tensor(start, dtype=torch.int32))
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    gen = torch.Generator(device="cuda").manual_seed(17)
    dt = c.k_pool.dtype
    appended = []
    for _ in range(grow):
        c.seq_lens += 1
        k_new = torch.randn((w.batch, 2, D), generator=gen, device="cuda").to(dt)
        v_new = torch.randn((w.batch, 2, D), generator=gen, device="cuda").to(dt)
        skv.kv_append_token(kv, k_new, v_new, stats)
        appended.append((k_new.clone(), v_new.clone()))
    assert_no_device_error()
    assert c.seq_lens.tolist() == list(final)

    rebuilt = skv.kv_build_page_stats(kv)
    table = c.page_table.cpu().numpy()
    mapped = np.unique(np.concatenate([table[b, : -(-n // PS)] for b, n in enumerate(final)]))
    got, ref = f64(stats), f64(rebuilt)
    np.testing.assert_array_equal(got[mapped], ref[mapped])
    mn, mx = oracle.page_stats(f64(c.k_pool), table, np.array(final), PS)
    np.testing.assert_array_equal(got[mapped, :, 0, :], mn[mapped])
    np.testing.assert_array_equal(got[mapped, :, 1, :], mx[mapped])
    # appended rows are in place
    for i, (k_new, v_new) in enumerate(appended):
        for b, n0 in enumerate(start):
            t = n0 + i
            P = int(table[b, t // PS])
            assert torch.equal(c.k_pool[P, :, t % PS, :], k_new[b])
            assert torch.equal(c.v_pool[P, :, t % PS, :], v_new[b])


def test_append_flags_an_unmapped_page():
    w = workload(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, dtype="bf16",
                 seed=6, seq_lens=(32,))
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    c.page_table[0, 1] = -1
    k_new = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    skv.kv_append_token(kv, k_new, k_new.clone(), stats)
    st, flags = skv.kv_check_device_errors()
    assert st == -5 and flags & 1
