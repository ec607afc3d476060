"""Seeded synthetic paged KV caches and decode queries.

This module only draws inputs: it holds none of the method's arithmetic (no statistics,
scores, selection or attention), so both the CUDA library and the float64 checker can take
their inputs from it without sharing any computation.

Recipe (one ``torch.Generator`` seeded per workload, draws made in the order below):

1. sequence lengths (fixed, or uniform integers in a range for the batched workload);
2. the physical placement of every logical page: a random permutation of a shared pool of
   ``sum_b ceil(len_b / PS)`` pages (or the identity for a contiguous table);
3. queries ``q ~ N(0, 1)`` in float32, rounded to the storage dtype;
4. keys and values ``~ N(0, 1)`` in float32, drawn page-chunk by page-chunk;
   (or, with ``page_noise``, a mean ~ N(0, 1) per (page, KV head) and coordinate plus
   ``page_noise`` times N(0, 1) per key);
5. planted salient tokens: for each (sequence, KV head), ``planted`` distinct positions drawn
   uniformly over the whole context get the key ``4 * qbar / |qbar| + N(0, 0.5^2)``, where
   ``qbar`` is the mean of the group's (rounded) query heads, so attention mass
   concentrates on them;
6. keys and values rounded to the storage dtype (bf16 by round-to-nearest-even).

The workloads stand in for the pages' real-text prefills and retrieval suites, which are
not available here: the shapes follow Llama-3.1-8B-like and Llama-3.1-70B-like decode
(32 or 64 query heads, 8 KV heads, head dim 128) at 32K, 128K and 1M tokens, plus a batch
of 32 sequences of mixed length.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


@dataclass(frozen=True)
class Workload:
    """Shape and data recipe of one synthetic decode workload."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str
    seed: int
    seq_len: int | None = None          # fixed length for every sequence
    seq_len_range: tuple[int, int] | None = None   # inclusive uniform range instead
    seq_lens: tuple[int, ...] | None = None         # explicit per-sequence lengths instead
    planted: int = 0                    # salient tokens per (sequence, KV head)
    page_noise: float | None = None     # None: keys N(0, 1); else each (page, KV head) draws a
                                        # mean ~ N(0, 1) per coordinate and its keys are that
                                        # mean + N(0, page_noise^2) (tight page boxes)
    permute_pages: bool = True          # random physical placement of pages
    keep_ratios: tuple[float, ...] = ()  # sparse keep ratios r_KV to run
    keep_pages: int | None = None       # fixed pages kept per group (instead of a ratio)
    budget_tokens: int | None = None    # token budget per group (instead of a ratio)
    description: str = ""

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload(
        name="tiny_fp32", batch=1, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
        dtype="fp32", seed=1, seq_len=4096, permute_pages=False, keep_pages=32,
        description="fp32, 8/2 heads, D 64, 4096 tokens, PS 16, contiguous table, top-32 pages"),
    "llama8b_32k": Workload(
        name="llama8b_32k", batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
        page_size=16, dtype="bf16", seed=2, seq_len=32768, planted=64, keep_ratios=(0.3,),
        description="Llama-3.1-8B-shaped decode, 32K tokens, PS 16, r_KV 0.3 (+ dense)"),
    "llama8b_128k": Workload(
        name="llama8b_128k", batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
        page_size=16, dtype="bf16", seed=3, seq_len=131072, planted=32,
        keep_ratios=(0.3, 0.2),
        description="Llama-3.1-8B-shaped decode, 128K tokens, PS 16, r_KV 0.3 and 0.2 (+ dense)"),
    "batched_serving": Workload(
        name="batched_serving", batch=32, num_q_heads=32, num_kv_heads=8, head_dim=128,
        page_size=16, dtype="bf16", seed=4, seq_len_range=(8192, 65536), budget_tokens=2048,
        description="32 sequences, lengths U[8192, 65536], shared pool, 2048-token budget"),
    "entmax_pruning_32k": Workload(
        name="entmax_pruning_32k", batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
        page_size=16, dtype="bf16", seed=6, seq_len=32768, page_noise=0.05, keep_ratios=(0.3,),
        description="8B-shaped decode, 32K tokens, PS 16, keys tight around per-page means "
                    "(within-page std 0.05): the entmax selector's boxes are tight"),
    "llama70b_1m": Workload(
        name="llama70b_1m", batch=1, num_q_heads=64, num_kv_heads=8, head_dim=128,
        page_size=64, dtype="bf16", seed=5, seq_len=1048576, planted=256,
        keep_ratios=(1.0 / 50.0,),
        description="Llama-3.1-70B-shaped decode, 1M tokens, PS 64, r_KV 1/50 (+ dense)"),
}


@dataclass
class KVCache:
    """A paged KV cache and one decode query batch, all tensors on one device."""

    workload: Workload
    k_pool: torch.Tensor        # [NP][Hkv][PS][D] storage dtype
    v_pool: torch.Tensor        # [NP][Hkv][PS][D]
    page_table: torch.Tensor    # [B][maxP] int32, -1 where unused
    seq_lens: torch.Tensor      # [B] int32
    q: torch.Tensor             # [B][Hq][D] storage dtype
    planted_positions: list = field(default_factory=list)  # [b][g] -> LongTensor

    @property
    def num_phys_pages(self) -> int:
        return self.k_pool.shape[0]

    @property
    def pages_per_seq(self) -> list[int]:
        ps = self.workload.page_size
        return [-(-int(n) // ps) for n in self.seq_lens.tolist()]


def _seq_lens(w: Workload, gen: torch.Generator, device) -> torch.Tensor:
    if w.seq_lens is not None:
        assert len(w.seq_lens) == w.batch
        return torch.tensor(list(w.seq_lens), dtype=torch.int32, device=device)
    if w.seq_len_range is not None:
        lo, hi = w.seq_len_range
        return torch.randint(lo, hi + 1, (w.batch,), generator=gen, device=device,
                             dtype=torch.int64).to(torch.int32)
    return torch.full((w.batch,), int(w.seq_len), dtype=torch.int32, device=device)


def make_cache(w: Workload, device="cpu", extra_phys_pages: int = 0) -> KVCache:
    """Draw the cache and query of workload ``w`` on ``device`` from its seed.

    ``extra_phys_pages`` appends unmapped pages to the pool (filled like the others), to
    check that nothing reads pages the table does not name.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.seed))
    dt = DTYPES[w.dtype]
    B, Hq, Hkv, D, PS = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size

    seq_lens = _seq_lens(w, gen, device)
    n_pages = [-(-int(n) // PS) for n in seq_lens.tolist()]
    mapped = sum(n_pages)
    NP = mapped + int(extra_phys_pages)
    max_p = max(n_pages) if n_pages else 0

    if w.permute_pages:
        placement = torch.randperm(NP, generator=gen, device=device)[:mapped]
    else:
        placement = torch.arange(mapped, device=device)
    page_table = torch.full((B, max(max_p, 1)), -1, dtype=torch.int32, device=device)
    off = 0
    for b in range(B):
        page_table[b, : n_pages[b]] = placement[off: off + n_pages[b]].to(torch.int32)
        off += n_pages[b]

    q32 = torch.randn((B, Hq, D), generator=gen, device=device, dtype=torch.float32)
    q = q32.to(dt)

    k_pool = torch.empty((NP, Hkv, PS, D), dtype=dt, device=device)
    v_pool = torch.empty((NP, Hkv, PS, D), dtype=dt, device=device)
    chunk = max(1, (1 << 26) // (Hkv * PS * D))     # about 64M elements per draw
    for p0 in range(0, NP, chunk):
        p1 = min(NP, p0 + chunk)
        shape = (p1 - p0, Hkv, PS, D)
        k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if w.page_noise is not None:
            mean = torch.randn((p1 - p0, Hkv, 1, D), generator=gen, device=device,
                               dtype=torch.float32)
            k = mean + float(w.page_noise) * k
        k_pool[p0:p1] = k.to(dt)
        v_pool[p0:p1] = torch.randn(shape, generator=gen, device=device,
                                    dtype=torch.float32).to(dt)

    planted_positions = []
    if w.planted > 0:
        qr = q.to(torch.float32)
        for b in range(B):
            L = int(seq_lens[b])
            per_b = []
            for g in range(Hkv):
                cnt = min(w.planted, L)
                pos = torch.randperm(L, generator=gen, device=device)[:cnt]
                qbar = qr[b, g * w.group_size:(g + 1) * w.group_size].mean(dim=0)
                direction = 4.0 * qbar / qbar.norm()
                noise = 0.5 * torch.randn((cnt, D), generator=gen, device=device,
                                          dtype=torch.float32)
                keys = (direction[None, :] + noise).to(dt)
                phys = page_table[b, (pos // PS)].to(torch.int64)
                k_pool[phys, g, pos % PS, :] = keys
                per_b.append(pos.sort().values)
            planted_positions.append(per_b)

    return KVCache(workload=w, k_pool=k_pool, v_pool=v_pool, page_table=page_table,
                   seq_lens=seq_lens, q=q, planted_positions=planted_positions)


def permute_physical(cache: KVCache, seed: int) -> KVCache:
    """Same logical cache with every physical page moved to a new random slot."""
    NP = cache.num_phys_pages
    gen = torch.Generator(device=cache.k_pool.device)
    gen.manual_seed(int(seed))
    perm = torch.randperm(NP, generator=gen, device=cache.k_pool.device)   # old -> new
    k_new = torch.empty_like(cache.k_pool)
    v_new = torch.empty_like(cache.v_pool)
    k_new[perm] = cache.k_pool
    v_new[perm] = cache.v_pool
    table = cache.page_table.clone()
    mask = table >= 0
    table[mask] = perm[table[mask].to(torch.int64)].to(torch.int32)
    return replace(cache, k_pool=k_new, v_pool=v_new, page_table=table)


def workload(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (e.g. a shorter context)."""
    w = WORKLOADS[name]
    return w.scaled(**overrides) if overrides else w
