"""Thin ctypes binding of ``libsparsekv.so`` (declared in ``include/sparsekv.h``).

Argument marshalling only: every function takes PyTorch CUDA tensors, checks their device,
dtype, shape and contiguity, and passes raw device pointers and the current CUDA stream to
the C function of the same name. All computation happens in the library's kernels; there
is no CPU fallback. If the library has not been built, every call raises.
"""

from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsparsekv.so")

KV_OK = 0
KV_BF16, KV_FP32 = 0, 1
ONE_LAUNCH = -1          # KV_SPLITS_ONE_LAUNCH: kv_decode_step as a single launch
# kv_decode_step_plan results (KV_PLAN_*)
PLANS = {0: "four kernels", 1: "score, then select + attention + merge",
         2: "score + select, then attention + merge", 3: "dense attention + merge",
         4: "dense attention, merge", 5: "one launch",
         6: "score, then select + attention, then merge",
         7: "score + select, then attention, then merge"}
STATUS = {0: "KV_OK", -1: "KV_ERR_INVALID_ARG", -2: "KV_ERR_UNSUPPORTED", -3: "KV_ERR_CUDA",
          -4: "KV_ERR_WORKSPACE", -5: "KV_ERR_BAD_INDEX", -6: "KV_ERR_TIMEOUT",
          -7: "KV_ERR_MISALIGNED"}
DEVERR = {"BAD_PAGE": 1, "BAD_LEN": 2, "BAD_SEL": 4, "KEEP": 8, "TIMEOUT": 16}

# Every symbol include/sparsekv.h declares.
EXPORTS = (
    "kv_status_string", "kv_version", "kv_build_page_stats", "kv_score_pages",
    "kv_select_topk", "kv_sparse_decode_attn", "kv_merge_splits", "kv_auto_num_splits",
    "kv_dropped_mass", "kv_dropped_mass_workspace_size", "kv_decode_step",
    "kv_decode_step_workspace_size", "kv_check_device_errors", "kv_set_wait_limit_ns",
    "kv_selftest_wait_timeout", "kv_decode_step_static", "kv_append_token",
    "kv_select_structured", "kv_select_decode_attn", "kv_score_select",
    "kv_decode_attn_merge", "kv_decode_step_plan", "kv_build_page_stats_fp8",
    "kv_score_pages_fp8", "kv_decode_step_fp8", "kv_entmax_page_moments", "kv_entmax_select",
    "kv_entmax_attn_workspace_size", "kv_entmax_decode_attn",
    "kv_entmax_decode_step_workspace_size", "kv_entmax_decode_step", "kv_workspace_size",
    "kv_decode_step_graph_create", "kv_decode_step_graph_launch", "kv_decode_step_graph_destroy",
)


class KVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} "
                         f"({_string(status)})")


class KVCacheDesc(ctypes.Structure):
    _fields_ = [
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("num_phys_pages", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
        ("page_table_stride", ctypes.c_int32),
        ("seq_lens", ctypes.c_void_p),
    ]


_lib = None


def _declare(lib):
    P, I32, F32, F64, SZ, U64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                 ctypes.c_double, ctypes.c_size_t, ctypes.c_uint64)
    D = ctypes.POINTER(KVCacheDesc)
    sig = {
        "kv_status_string": (ctypes.c_char_p, [I32]),
        "kv_version": (I32, []),
        "kv_build_page_stats": (I32, [D, P, P, I32, P]),
        "kv_workspace_size": (SZ, [I32, D, I32, I32, I32]),
        "kv_decode_step_graph_create": (I32, [D, P, I32, F32, P, F64, I32, I32, I32, P, P, P, SZ,
                                              P, P, ctypes.POINTER(P)]),
        "kv_decode_step_graph_launch": (I32, [P, P]),
        "kv_decode_step_graph_destroy": (I32, [P]),
        "kv_score_pages": (I32, [D, P, I32, P, P, I32, P]),
        "kv_select_topk": (I32, [P, I32, P, I32, I32, I32, P, F64, I32, I32, P, P, P]),
        "kv_sparse_decode_attn": (I32, [D, P, I32, F32, P, P, I32, I32, P, P, P]),
        "kv_merge_splits": (I32, [P, P, I32, I32, I32, I32, P, P, P]),
        "kv_auto_num_splits": (I32, [D, I32, I32]),
        "kv_dropped_mass": (I32, [D, P, I32, F32, P, P, I32, P, P, SZ, P]),
        "kv_dropped_mass_workspace_size": (SZ, [D, I32]),
        "kv_decode_step": (I32, [D, P, I32, F32, P, F64, I32, I32, I32, P, P, P, SZ, P]),
        "kv_decode_step_workspace_size": (SZ, [D, I32, I32, I32]),
        "kv_check_device_errors": (I32, [P, ctypes.POINTER(I32)]),
        "kv_set_wait_limit_ns": (I32, [U64]),
        "kv_selftest_wait_timeout": (I32, [U64, P]),
        "kv_decode_step_static": (I32, [D, P, I32, F32, P, F64, I32, I32, I32, P, P, P]),
        "kv_append_token": (I32, [D, P, P, P, P]),
        "kv_select_structured": (I32, [P, I32, P, I32, I32, I32, P, F64, I32, I32, I32, I32, P,
                                       P, P]),
        "kv_select_decode_attn": (I32, [D, P, I32, F32, P, I32, F64, I32, I32, I32, P, P, P, P,
                                        P, P, P, P]),
        "kv_score_select": (I32, [D, P, I32, P, F64, I32, I32, P, I32, P, P, P, P]),
        "kv_decode_attn_merge": (I32, [D, P, I32, F32, P, P, I32, I32, P, P, P, P, P, P]),
        "kv_decode_step_plan": (I32, [D, I32, F64, I32, I32, I32, ctypes.POINTER(I32)]),
        "kv_build_page_stats_fp8": (I32, [D, P, P, P]),
        "kv_score_pages_fp8": (I32, [D, P, I32, P, P, P, I32, P]),
        "kv_decode_step_fp8": (I32, [D, P, I32, F32, P, P, F64, I32, I32, I32, P, P, P, SZ, P]),
        "kv_entmax_page_moments": (I32, [D, P, I32, P, F32, P, P, P, I32, P]),
        "kv_entmax_select": (I32, [P, P, P, I32, P, I32, I32, I32, I32, I32, P, P, P, P]),
        "kv_entmax_attn_workspace_size": (SZ, [D, I32, I32]),
        "kv_entmax_decode_attn": (I32, [D, P, I32, F32, P, P, I32, P, P, P, SZ, P]),
        "kv_entmax_decode_step_workspace_size": (SZ, [D, I32, I32]),
        "kv_entmax_decode_step": (I32, [D, P, I32, F32, P, I32, P, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def lib():
    """The loaded library; raises if it was not built (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(LIB_PATH)
        _declare(handle)
        _lib = handle
    return _lib


def _string(status: int) -> str:
    try:
        return lib().kv_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - message only
        return "?"


def _check(fn: str, status: int):
    if status != KV_OK:
        raise KVError(fn, status)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


_DT = {torch.bfloat16: KV_BF16, torch.float32: KV_FP32}


@dataclass
class PagedKV:
    """The caller-owned tensors of a paged cache, and their C descriptor."""

    k_pool: torch.Tensor       # [NP][Hkv][PS][D]
    v_pool: torch.Tensor
    page_table: torch.Tensor   # [B][stride] int32
    seq_lens: torch.Tensor     # [B] int32

    def __post_init__(self):
        _need(self.k_pool, "k_pool")
        _need(self.v_pool, "v_pool", self.k_pool.dtype, self.k_pool.shape)
        _need(self.page_table, "page_table", torch.int32)
        _need(self.seq_lens, "seq_lens", torch.int32)
        if self.k_pool.dtype not in _DT:
            raise ValueError("k_pool must be bf16 or fp32")
        if self.page_table.dim() != 2 or self.seq_lens.shape != (self.page_table.shape[0],):
            raise ValueError("page_table must be [B][stride] and seq_lens [B]")
        NP, Hkv, PS, D = self.k_pool.shape
        self.desc = KVCacheDesc(
            self.k_pool.data_ptr(), self.v_pool.data_ptr(), _DT[self.k_pool.dtype], NP, Hkv,
            PS, D, self.page_table.shape[0], self.page_table.data_ptr(),
            self.page_table.shape[1], self.seq_lens.data_ptr())

    @classmethod
    def from_cache(cls, cache) -> "PagedKV":
        return cls(cache.k_pool, cache.v_pool, cache.page_table, cache.seq_lens)

    @property
    def dtype(self):
        return self.k_pool.dtype

    @property
    def batch(self):
        return self.page_table.shape[0]

    @property
    def num_kv_heads(self):
        return self.k_pool.shape[1]

    @property
    def page_size(self):
        return self.k_pool.shape[2]

    @property
    def head_dim(self):
        return self.k_pool.shape[3]

    @property
    def stride(self):
        return self.page_table.shape[1]

    def ref(self):
        return ctypes.byref(self.desc)


# -------------------------------------------------------------------------------- calls

def kv_version() -> int:
    return lib().kv_version()


def kv_build_page_stats(kv: PagedKV, stats=None, phys_pages=None, stream=None):
    """Page statistics of every mapped page, or (phys_pages: a strictly ascending int32
    tensor of physical page indices) of the mapped pages in that subset only."""
    NP, Hkv, PS, D = kv.k_pool.shape
    if stats is None:
        stats = torch.empty((NP, Hkv, 2, D), dtype=kv.dtype, device=kv.k_pool.device)
    _need(stats, "stats", kv.dtype, (NP, Hkv, 2, D))
    n_phys = 0
    if phys_pages is not None:
        _need(phys_pages, "phys_pages", torch.int32)
        n_phys = phys_pages.numel()
        if n_phys == 0:              # an empty list (whose data pointer may be NULL): no work
            return stats
    _check("kv_build_page_stats", lib().kv_build_page_stats(
        kv.ref(), _ptr(stats), _ptr(phys_pages), n_phys, _stream(stream)))
    return stats


def kv_build_page_stats_fp8(kv: PagedKV, stats=None, stats_exp=None, stream=None):
    """FP8 (E4M3) page statistics with outward rounding: (bytes [NP][Hkv][2][D] uint8,
    exponents [NP][Hkv] int8)."""
    NP, Hkv, D = kv.k_pool.shape[0], kv.num_kv_heads, kv.head_dim
    dev = kv.k_pool.device
    if stats is None:
        stats = torch.zeros((NP, Hkv, 2, D), dtype=torch.uint8, device=dev)
    if stats_exp is None:
        stats_exp = torch.zeros((NP, Hkv), dtype=torch.int8, device=dev)
    _need(stats, "stats", torch.uint8, (NP, Hkv, 2, D))
    _need(stats_exp, "stats_exp", torch.int8, (NP, Hkv))
    _check("kv_build_page_stats_fp8", lib().kv_build_page_stats_fp8(
        kv.ref(), _ptr(stats), _ptr(stats_exp), _stream(stream)))
    return stats, stats_exp


def kv_score_pages_fp8(kv: PagedKV, q, stats, stats_exp, scores=None, stream=None):
    _need(q, "q", kv.dtype)
    _need(stats, "stats", torch.uint8)
    _need(stats_exp, "stats_exp", torch.int8)
    B, Hq, _ = q.shape
    if scores is None:
        scores = torch.empty((B, kv.num_kv_heads, kv.stride), dtype=torch.float32,
                             device=q.device)
    _need(scores, "scores", torch.float32)
    _check("kv_score_pages_fp8", lib().kv_score_pages_fp8(
        kv.ref(), _ptr(q), Hq, _ptr(stats), _ptr(stats_exp), _ptr(scores), scores.shape[-1],
        _stream(stream)))
    return scores


def kv_append_token(kv: PagedKV, k_new, v_new, stats, stream=None):
    """Write the new token (position seq_lens[b] - 1) into the pools and fold its key into
    its page's min/max. k_new, v_new: [B][Hkv][D] of the cache dtype."""
    shape = (kv.batch, kv.num_kv_heads, kv.head_dim)
    _need(k_new, "k_new", kv.dtype, shape)
    _need(v_new, "v_new", kv.dtype, shape)
    _need(stats, "stats", kv.dtype)
    _check("kv_append_token", lib().kv_append_token(kv.ref(), _ptr(k_new), _ptr(v_new),
                                                    _ptr(stats), _stream(stream)))
    return stats


def kv_score_pages(kv: PagedKV, q, stats, scores=None, stream=None):
    _need(q, "q", kv.dtype)
    Hq = q.shape[1]
    if scores is None:
        scores = torch.empty((kv.batch, kv.num_kv_heads, kv.stride), dtype=torch.float32,
                             device=q.device)
    _need(scores, "scores", torch.float32)
    _check("kv_score_pages", lib().kv_score_pages(kv.ref(), _ptr(q), Hq, _ptr(stats), _ptr(scores),
                                                  scores.shape[-1], _stream(stream)))
    return scores


def max_keep_pages(stride: int, keep_ratio: float | None = None,
                   budget_pages: int | None = None) -> int:
    """An upper bound of the keep count over sequences of at most ``stride`` pages."""
    if budget_pages is not None and budget_pages > 0:
        return max(1, min(stride, int(budget_pages)))
    if keep_ratio is None or keep_ratio >= 1.0:
        return stride
    return max(1, min(stride, math.ceil(keep_ratio * stride)))


def kv_select_topk(scores, seq_lens, page_size: int, keep=None, keep_ratio: float = 0.0,
                   budget_pages: int = 0, k_max: int | None = None, sel_idx=None, sel_cnt=None,
                   stream=None):
    _need(scores, "scores", torch.float32)
    B, Hkv, stride = scores.shape
    if k_max is None:
        k_max = stride if keep is not None else max_keep_pages(stride, keep_ratio, budget_pages)
    if sel_idx is None:
        sel_idx = torch.empty((B, Hkv, k_max), dtype=torch.int32, device=scores.device)
    if sel_cnt is None:
        sel_cnt = torch.empty((B, Hkv), dtype=torch.int32, device=scores.device)
    _need(sel_idx, "sel_idx", torch.int32, (B, Hkv, k_max))
    _need(sel_cnt, "sel_cnt", torch.int32, (B, Hkv))
    if keep is not None:
        _need(keep, "keep", torch.int32, (B,))
    _check("kv_select_topk", lib().kv_select_topk(
        _ptr(scores), stride, _ptr(seq_lens), int(page_size), B, Hkv, _ptr(keep),
        float(keep_ratio), int(budget_pages), int(k_max), _ptr(sel_idx), _ptr(sel_cnt),
        _stream(stream)))
    return sel_idx, sel_cnt


def kv_select_structured(scores, seq_lens, page_size: int, batch: int, num_kv_heads: int,
                         stride: int, sink_pages: int = 0, local_pages: int = 0, keep=None,
                         keep_ratio: float = 0.0, budget_pages: int = 0, k_max: int | None = None,
                         sel_idx=None, sel_cnt=None, stream=None):
    """Forced first sink_pages and last local_pages pages joined to the top-k of the rest;
    scores may be None (the KV-window baseline when sink_pages = 0)."""
    if scores is not None:
        _need(scores, "scores", torch.float32, (batch, num_kv_heads, stride))
    dev = seq_lens.device
    if k_max is None:
        k_max = min(stride, max_keep_pages(stride, keep_ratio if keep_ratio else None,
                                           budget_pages or None) + sink_pages + local_pages)
    if sel_idx is None:
        sel_idx = torch.empty((batch, num_kv_heads, k_max), dtype=torch.int32, device=dev)
    if sel_cnt is None:
        sel_cnt = torch.empty((batch, num_kv_heads), dtype=torch.int32, device=dev)
    _need(sel_idx, "sel_idx", torch.int32, (batch, num_kv_heads, k_max))
    _need(sel_cnt, "sel_cnt", torch.int32, (batch, num_kv_heads))
    if keep is not None:
        _need(keep, "keep", torch.int32, (batch,))
    _check("kv_select_structured", lib().kv_select_structured(
        _ptr(scores), int(stride), _ptr(seq_lens), int(page_size), int(batch),
        int(num_kv_heads), _ptr(keep), float(keep_ratio), int(budget_pages), int(sink_pages),
        int(local_pages), int(k_max), _ptr(sel_idx), _ptr(sel_cnt), _stream(stream)))
    return sel_idx, sel_cnt


def kv_auto_num_splits(kv: PagedKV, num_q_heads: int, pages_per_group: int) -> int:
    r = lib().kv_auto_num_splits(kv.ref(), int(num_q_heads), int(pages_per_group))
    if r < 0:
        raise KVError("kv_auto_num_splits", r)
    return r


def kv_sparse_decode_attn(kv: PagedKV, q, sm_scale: float, sel_idx=None, sel_cnt=None,
                          num_splits: int | None = None, part_acc=None, part_ml=None,
                          stream=None):
    _need(q, "q", kv.dtype)
    B, Hq, D = q.shape
    if num_splits is None:
        bound = sel_idx.shape[-1] if sel_idx is not None else kv.stride
        num_splits = kv_auto_num_splits(kv, Hq, bound)
    S = int(num_splits)
    if part_acc is None:
        part_acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device=q.device)
    if part_ml is None:
        part_ml = torch.empty((B, Hq, S, 2), dtype=torch.float32, device=q.device)
    _need(part_acc, "part_acc", torch.float32, (B, Hq, S, D))
    _need(part_ml, "part_ml", torch.float32, (B, Hq, S, 2))
    sel_stride = 0
    if sel_idx is not None:
        _need(sel_idx, "sel_idx", torch.int32)
        _need(sel_cnt, "sel_cnt", torch.int32)
        sel_stride = sel_idx.shape[-1]
    _check("kv_sparse_decode_attn", lib().kv_sparse_decode_attn(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(sel_idx), _ptr(sel_cnt), sel_stride, S,
        _ptr(part_acc), _ptr(part_ml), _stream(stream)))
    return part_acc, part_ml


def kv_select_decode_attn(kv: PagedKV, q, sm_scale: float, scores=None, keep_ratio: float = 1.0,
                          budget_pages: int = 0, k_max: int | None = None,
                          num_splits: int | None = None, part_acc=None, part_ml=None,
                          counters=None, out=None, lse=None, sel_idx=None, sel_cnt=None,
                          merge: bool = True, stream=None):
    """Selection, split-K attention and merge in one kernel (bf16); scores=None is dense.
    counters must start at zero (they are returned to zero). merge=False: the kernel only
    writes the partials, returned as (part_acc, part_ml)."""
    _need(q, "q", kv.dtype)
    B, Hq, D = q.shape
    Hkv = kv.num_kv_heads
    if k_max is None:
        k_max = max_keep_pages(kv.stride, keep_ratio, budget_pages) if scores is not None else 1
    if num_splits is None:
        num_splits = kv_auto_num_splits(kv, Hq, k_max if scores is not None else kv.stride)
    S = int(num_splits)
    dev = q.device
    if part_acc is None:
        part_acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device=dev)
    if part_ml is None:
        part_ml = torch.empty((B, Hq, S, 2), dtype=torch.float32, device=dev)
    if merge:
        if counters is None:
            counters = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)
        if out is None:
            out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
        if lse is None:
            lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        _need(counters, "counters", torch.int32, (B, Hkv))
    else:
        counters = out = lse = None
    _need(part_acc, "part_acc", torch.float32, (B, Hq, S, D))
    _need(part_ml, "part_ml", torch.float32, (B, Hq, S, 2))
    stride = 0
    if scores is not None:
        _need(scores, "scores", torch.float32)
        stride = scores.shape[-1]
    _check("kv_select_decode_attn", lib().kv_select_decode_attn(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(scores), stride, float(keep_ratio),
        int(budget_pages), int(k_max), S, _ptr(part_acc), _ptr(part_ml), _ptr(counters),
        _ptr(out), _ptr(lse), _ptr(sel_idx), _ptr(sel_cnt), _stream(stream)))
    return (out, lse) if merge else (part_acc, part_ml)


def kv_score_select(kv: PagedKV, q, stats, keep_ratio: float = 0.0, budget_pages: int = 0,
                    k_max: int | None = None, scores=None, counters=None, sel_idx=None,
                    sel_cnt=None, stream=None):
    """kv_score_pages + kv_select_topk in one launch. counters must start at zero (they are
    returned to zero). Returns (scores, sel_idx, sel_cnt)."""
    _need(q, "q", kv.dtype)
    B, Hkv, stride, dev = kv.batch, kv.num_kv_heads, kv.stride, q.device
    if k_max is None:
        k_max = max_keep_pages(stride, keep_ratio, budget_pages)
    if scores is None:
        scores = torch.empty((B, Hkv, stride), dtype=torch.float32, device=dev)
    if counters is None:
        counters = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)
    if sel_idx is None:
        sel_idx = torch.empty((B, Hkv, k_max), dtype=torch.int32, device=dev)
    if sel_cnt is None:
        sel_cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    _need(scores, "scores", torch.float32)
    _need(counters, "counters", torch.int32, (B, Hkv))
    _need(sel_idx, "sel_idx", torch.int32, (B, Hkv, k_max))
    _need(sel_cnt, "sel_cnt", torch.int32, (B, Hkv))
    _check("kv_score_select", lib().kv_score_select(
        kv.ref(), _ptr(q), q.shape[1], _ptr(stats), float(keep_ratio), int(budget_pages),
        int(k_max), _ptr(scores), scores.shape[-1], _ptr(counters), _ptr(sel_idx),
        _ptr(sel_cnt), _stream(stream)))
    return scores, sel_idx, sel_cnt


def kv_decode_attn_merge(kv: PagedKV, q, sm_scale: float, sel_idx=None, sel_cnt=None,
                         num_splits: int | None = None, part_acc=None, part_ml=None,
                         counters=None, out=None, lse=None, stream=None):
    """kv_sparse_decode_attn + kv_merge_splits in one launch (bf16); sel_idx=None is dense.
    counters must start at zero (they are returned to zero). Returns (out, lse)."""
    _need(q, "q", kv.dtype)
    B, Hq, D = q.shape
    dev = q.device
    if num_splits is None:
        bound = sel_idx.shape[-1] if sel_idx is not None else kv.stride
        num_splits = kv_auto_num_splits(kv, Hq, bound)
    S = int(num_splits)
    if part_acc is None:
        part_acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device=dev)
    if part_ml is None:
        part_ml = torch.empty((B, Hq, S, 2), dtype=torch.float32, device=dev)
    if counters is None:
        counters = torch.zeros((B, kv.num_kv_heads), dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _need(part_acc, "part_acc", torch.float32, (B, Hq, S, D))
    _need(part_ml, "part_ml", torch.float32, (B, Hq, S, 2))
    _need(counters, "counters", torch.int32, (B, kv.num_kv_heads))
    sel_stride = 0
    if sel_idx is not None:
        _need(sel_idx, "sel_idx", torch.int32)
        _need(sel_cnt, "sel_cnt", torch.int32)
        sel_stride = sel_idx.shape[-1]
    _check("kv_decode_attn_merge", lib().kv_decode_attn_merge(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(sel_idx), _ptr(sel_cnt), sel_stride, S,
        _ptr(part_acc), _ptr(part_ml), _ptr(counters), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def kv_merge_splits(part_acc, part_ml, out=None, lse=None, stream=None):
    _need(part_acc, "part_acc", torch.float32)
    B, Hq, S, D = part_acc.shape
    _need(part_ml, "part_ml", torch.float32, (B, Hq, S, 2))
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=part_acc.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=part_acc.device)
    _need(out, "out", torch.float32, (B, Hq, D))
    _check("kv_merge_splits", lib().kv_merge_splits(
        _ptr(part_acc), _ptr(part_ml), B, Hq, S, D, _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def kv_dropped_mass_workspace_size(kv: PagedKV, num_q_heads: int) -> int:
    return int(lib().kv_dropped_mass_workspace_size(kv.ref(), int(num_q_heads)))


def kv_dropped_mass(kv: PagedKV, q, sm_scale: float, sel_idx, sel_cnt, delta=None,
                    workspace=None, stream=None):
    _need(q, "q", kv.dtype)
    B, Hq, _ = q.shape
    _need(sel_idx, "sel_idx", torch.int32)
    _need(sel_cnt, "sel_cnt", torch.int32)
    if delta is None:
        delta = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    nbytes = kv_dropped_mass_workspace_size(kv, Hq)
    if workspace is None:
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=q.device)
    _check("kv_dropped_mass", lib().kv_dropped_mass(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(sel_idx), _ptr(sel_cnt),
        sel_idx.shape[-1], _ptr(delta), _ptr(workspace), workspace.numel(), _stream(stream)))
    return delta


KV_OP = {"decode_step": 0, "dropped_mass": 1, "entmax_decode_attn": 2, "entmax_decode_step": 3}


def kv_workspace_size(op: str, kv: PagedKV, num_q_heads: int, k_max: int = 0,
                      num_splits: int = 0) -> int:
    return int(lib().kv_workspace_size(KV_OP[op], kv.ref(), int(num_q_heads), int(k_max),
                                       int(num_splits)))


def kv_decode_step_workspace_size(kv: PagedKV, num_q_heads: int, k_max: int,
                                  num_splits: int = 0) -> int:
    return int(lib().kv_decode_step_workspace_size(kv.ref(), int(num_q_heads), int(k_max),
                                                   int(num_splits)))


def kv_decode_step(kv: PagedKV, q, sm_scale: float, stats=None, keep_ratio: float = 1.0,
                   budget_pages: int = 0, k_max: int | None = None, num_splits: int = 0,
                   out=None, lse=None, workspace=None, stream=None):
    _need(q, "q", kv.dtype)
    B, Hq, D = q.shape
    if k_max is None:
        k_max = max_keep_pages(kv.stride, keep_ratio, budget_pages)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = kv_decode_step_workspace_size(kv, Hq, k_max, max(num_splits, 0))
        workspace = torch.zeros((nbytes,), dtype=torch.uint8, device=q.device)
    _check("kv_decode_step", lib().kv_decode_step(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(stats), float(keep_ratio),
        int(budget_pages), int(k_max), int(num_splits), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


class DecodeStepGraph:
    """kv_decode_step captured once (kv_decode_step_graph_create): launch() runs the step with
    the buffers given here, whose contents (q, the cache) the caller updates in place."""

    def __init__(self, kv: PagedKV, q, sm_scale: float, stats=None, keep_ratio: float = 1.0,
                 budget_pages: int = 0, k_max: int | None = None, num_splits: int = 0,
                 out=None, lse=None, workspace=None, q_host=None, out_host=None):
        """q_host / out_host: optional page-locked CPU tensors; each launch then takes the
        query from q_host and leaves the output in out_host (read and written in place by the
        kernels when the device addresses them, else copied through q and out)."""
        _need(q, "q", kv.dtype)
        for t, name in ((q_host, "q_host"), (out_host, "out_host")):
            if t is not None and (t.is_cuda or not t.is_pinned() or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous page-locked CPU tensor")
        if q_host is not None and (q_host.dtype != q.dtype or q_host.shape != q.shape):
            raise ValueError("q_host must match q")
        B, Hq, D = q.shape
        if k_max is None:
            k_max = max_keep_pages(kv.stride, keep_ratio, budget_pages)
        self.out = out if out is not None else torch.empty((B, Hq, D), dtype=torch.float32,
                                                           device=q.device)
        self.lse = lse if lse is not None else torch.empty((B, Hq), dtype=torch.float32,
                                                           device=q.device)
        if workspace is None:
            nbytes = kv_decode_step_workspace_size(kv, Hq, k_max, max(num_splits, 0))
            workspace = torch.zeros((nbytes,), dtype=torch.uint8, device=q.device)
        if out_host is not None and (out_host.dtype != torch.float32 or
                                     out_host.shape != self.out.shape):
            raise ValueError("out_host must be float32 of the output's shape")
        # the buffers must outlive the graph: keep them referenced
        self._keep = (kv, q, stats, workspace, q_host, out_host)
        handle = ctypes.c_void_p()
        _check("kv_decode_step_graph_create", lib().kv_decode_step_graph_create(
            kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(stats), float(keep_ratio),
            int(budget_pages), int(k_max), int(num_splits), _ptr(self.out), _ptr(self.lse),
            _ptr(workspace), workspace.numel(), _ptr(q_host), _ptr(out_host),
            ctypes.byref(handle)))
        self._handle = handle

    def launch(self, stream=None):
        """Runs the step; returns (output, lse), the output being out_host when given."""
        _check("kv_decode_step_graph_launch",
               lib().kv_decode_step_graph_launch(self._handle, _stream(stream)))
        out_host = self._keep[5]
        return (out_host if out_host is not None else self.out), self.lse

    def close(self):
        if getattr(self, "_handle", None) is not None and self._handle.value is not None:
            lib().kv_decode_step_graph_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kv_decode_step_plan(kv: PagedKV, num_q_heads: int, keep_ratio: float = 1.0,
                        budget_pages: int = 0, k_max: int | None = None,
                        num_splits: int = 0) -> tuple[int, int]:
    """(KV_PLAN_* value, split count) of kv_decode_step for these arguments; no launch."""
    if k_max is None:
        k_max = max_keep_pages(kv.stride, keep_ratio, budget_pages)
    splits = ctypes.c_int32(0)
    r = lib().kv_decode_step_plan(kv.ref(), int(num_q_heads), float(keep_ratio),
                                  int(budget_pages), int(k_max), int(num_splits),
                                  ctypes.byref(splits))
    if r < 0:
        raise KVError("kv_decode_step_plan", r)
    return int(r), int(splits.value)


def kv_decode_step_fp8(kv: PagedKV, q, sm_scale: float, stats=None, stats_exp=None,
                       keep_ratio: float = 1.0, budget_pages: int = 0, k_max: int | None = None,
                       num_splits: int = 0, out=None, lse=None, workspace=None, stream=None):
    """kv_decode_step scoring from FP8 statistics (kv_build_page_stats_fp8)."""
    _need(q, "q", kv.dtype)
    B, Hq, D = q.shape
    if k_max is None:
        k_max = max_keep_pages(kv.stride, keep_ratio, budget_pages)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = kv_decode_step_workspace_size(kv, Hq, k_max, max(num_splits, 0))
        workspace = torch.zeros((nbytes,), dtype=torch.uint8, device=q.device)
    _check("kv_decode_step_fp8", lib().kv_decode_step_fp8(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(stats), _ptr(stats_exp),
        float(keep_ratio), int(budget_pages), int(k_max), int(num_splits), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def kv_entmax_page_moments(kv: PagedKV, q, stats, sm_scale: float, stream=None):
    """(zb, cz, vz), each [B][Hq][stride] float32: per-head page bound, centre and variance
    of z = sm_scale * q.k / 2."""
    _need(q, "q", kv.dtype)
    B, Hq, _ = q.shape
    zb, cz, vz = (torch.full((B, Hq, kv.stride), float("nan"), dtype=torch.float32,
                             device=q.device) for _ in range(3))
    _check("kv_entmax_page_moments", lib().kv_entmax_page_moments(
        kv.ref(), _ptr(q), Hq, _ptr(stats), float(sm_scale), _ptr(zb), _ptr(cz), _ptr(vz),
        kv.stride, _stream(stream)))
    return zb, cz, vz


def kv_entmax_select(zb, cz, vz, seq_lens, page_size: int, num_kv_heads: int,
                     k_max: int | None = None, stream=None):
    """Gaussian-aware entmax page selection: (sel_idx, sel_cnt, tau_hat)."""
    for t, n in ((zb, "zb"), (cz, "cz"), (vz, "vz")):
        _need(t, n, torch.float32)
    B, Hq, stride = zb.shape
    if k_max is None:
        k_max = stride
    dev = zb.device
    sel = torch.empty((B, num_kv_heads, k_max), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, num_kv_heads), dtype=torch.int32, device=dev)
    tau = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _check("kv_entmax_select", lib().kv_entmax_select(
        _ptr(zb), _ptr(cz), _ptr(vz), stride, _ptr(seq_lens), int(page_size), B, Hq,
        int(num_kv_heads), int(k_max), _ptr(sel), _ptr(cnt), _ptr(tau), _stream(stream)))
    return sel, cnt, tau


def kv_entmax_decode_attn(kv: PagedKV, q, sm_scale: float, sel_idx=None, sel_cnt=None,
                          out=None, tau=None, workspace=None, stream=None):
    """1.5-entmax attention over the selected pages (sel_idx=None: every page): (out, tau)."""
    _need(q, "q", kv.dtype)
    B, Hq, D = q.shape
    sel_stride = sel_idx.shape[-1] if sel_idx is not None else 0
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if tau is None:
        tau = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = int(lib().kv_entmax_attn_workspace_size(kv.ref(), Hq, sel_stride))
        workspace = torch.empty((n,), dtype=torch.uint8, device=q.device)
    _check("kv_entmax_decode_attn", lib().kv_entmax_decode_attn(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(sel_idx), _ptr(sel_cnt), sel_stride,
        _ptr(out), _ptr(tau), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, tau


def kv_entmax_decode_step_workspace_size(kv: PagedKV, num_q_heads: int, k_max: int) -> int:
    return int(lib().kv_entmax_decode_step_workspace_size(kv.ref(), int(num_q_heads),
                                                          int(k_max)))


def kv_entmax_decode_step(kv: PagedKV, q, sm_scale: float, stats, k_max: int | None = None,
                          out=None, tau=None, workspace=None, stream=None):
    """Moments, Gaussian-aware selection and entmax attention in one call: (out, tau)."""
    _need(q, "q", kv.dtype)
    B, Hq, D = q.shape
    if k_max is None:
        k_max = kv.stride
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if tau is None:
        tau = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty((kv_entmax_decode_step_workspace_size(kv, Hq, k_max),),
                                dtype=torch.uint8, device=q.device)
    _check("kv_entmax_decode_step", lib().kv_entmax_decode_step(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(stats), int(k_max), _ptr(out), _ptr(tau),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, tau


def kv_check_device_errors(stream=None):
    """Synchronise the stream; return (status, raw flag mask) and clear the device word."""
    flags = ctypes.c_int32(0)
    st = lib().kv_check_device_errors(_stream(stream), ctypes.byref(flags))
    return st, flags.value


def kv_set_wait_limit_ns(limit_ns: int):
    _check("kv_set_wait_limit_ns", lib().kv_set_wait_limit_ns(int(limit_ns)))


def kv_selftest_wait_timeout(limit_ns: int, stream=None):
    _check("kv_selftest_wait_timeout", lib().kv_selftest_wait_timeout(int(limit_ns),
                                                                      _stream(stream)))


STATIC_SCRATCH_BYTES = 8 << 20     # KV_STATIC_SCRATCH_BYTES of include/sparsekv.h


def kv_decode_step_static(kv: PagedKV, q, sm_scale: float, stats=None, keep_ratio: float = 1.0,
                          budget_pages: int = 0, k_max: int | None = None, num_splits: int = 0,
                          out=None, lse=None, stream=None):
    """kv_decode_step on the library's own static scratch: for callers that cannot allocate
    device memory on the decode path. Only out and lse are the caller's; calls that overlap
    on the GPU share the scratch and must be serialised. Raises when the shape needs more
    scratch than the library holds."""
    _need(q, "q", kv.dtype)
    B, Hq, D = q.shape
    if k_max is None:
        k_max = max_keep_pages(kv.stride, keep_ratio, budget_pages)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = lib().kv_decode_step_static(
        kv.ref(), _ptr(q), Hq, float(sm_scale), _ptr(stats), float(keep_ratio),
        int(budget_pages), int(k_max), int(num_splits), _ptr(out), _ptr(lse), _stream(stream))
    if st == -4:
        raise KVError("kv_decode_step_static (the shape needs more than the "
                      f"{STATIC_SCRATCH_BYTES >> 20} MiB static scratch)", st)
    _check("kv_decode_step_static", st)
    return out, lse
