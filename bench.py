"""Decode-attention benchmark: sparse paged-KV decode step vs the dense step, on GB300.

A step is one sparse decode step over the whole batch: page scores, top-k selection,
split-K attention over the selected pages and the log-sum-exp merge (the page statistics
already exist; their build is timed separately). The dense step is the same attention
kernel with every page kept, plus the merge. Inputs are resident in HBM; L2 is flushed
(a 256 MiB write, twice the L2) before every timed step, outside the timed events.

The headline (``value``) is the 32K workload. The same line carries ``configs``: the
128K workload at both keep ratios, the batched-serving workload and the 1M workload, each
with its sparse and dense steps, FP8-statistics step, KV-window step, attention-kernel
roofline, byte bound, dropped mass and a bounded oracle baseline; and ``blocks``: the
headline sparse/dense pair timed in fresh processes, with paired ratios and resampled
intervals. ``e2e`` goes through the captured step (``kv_decode_step_graph_*``) with the
query taken from and the output returned to pinned host memory inside the timing.

Prints one JSON line. ``--impl reference`` times the float64 CPU oracle on the same
workload instead (the reference arm of this comparison).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = ("decode-attn µs/step and achieved HBM GB/s vs peak at 32K–1M ctx; "
          "sparse/dense speedup")
DEFAULT_WORKLOAD = "llama8b_32k"
PROFILE_DIR = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "sparse_kv_cache_build_gb300", "csrc")
# the attention kernel that runs for each storage dtype, and its source file
ATTN_KERNEL = {"bf16": ("split_attn_mma_kernel", os.path.join(CSRC, "attn_mma.cuh")),
               "fp32": ("split_attn_kernel", os.path.join(CSRC, "attn_impl.cuh"))}


# ----------------------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, world, device):
    """Element-wise maximum of each rank's values over the process group (any backend);
    the values themselves when there is one rank. Every rank gets the result."""
    if world <= 1:
        return [float(v) for v in values]
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def file_hash(*paths):
    """First 16 hex digits of the sha256 of the files' bytes, concatenated in order."""
    h = hashlib.sha256()
    for path in paths:
        h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def kernel_sources(source):
    """The files whose code the timed kernel compiles from: the attention kernel's header and
    the in-block top-k it selects with."""
    return (source, os.path.join(os.path.dirname(source), "cta_topk.cuh"))


def committed_traffic(workload, keep_label, source):
    """Per-launch DRAM bytes of the timed kernel from a committed ncu summary, if the
    kernel's sources have not changed since the counters were taken."""
    p = os.path.join(PROFILE_DIR, f"{os.path.basename(source).split('.')[0]}_{workload}.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("source_hash") != file_hash(*kernel_sources(source)):
        return None
    return d.get("traffic_bytes_per_launch", {}).get(keep_label)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"skv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def pct(xs, q):
    return float(np.percentile(np.asarray(xs), q))


# ----------------------------------------------------------------------------- byte account

def byte_account(w, n_pages, sel_cnt, S):
    """Algorithmic bytes: what the method must touch (not what a kernel happens to read).

    sparse step = sum_b Hkv*(k_b*PS*D*2*eb [selected K+V] + n_b*2*D*eb [page stats])
                  + B*Hq*D*eb [q] + sum_b n_b*4 [table] + sum_{b,g} k_bg*4 [indices]
    attention launch = sum_{b,g} k_bg*(2*PS*D*eb + 8) [pages + index + table entry]
                       + B*Hq*D*eb [q] + B*Hq*S*(D+2)*4 [partials written]
    attention + merge launch = sum_{b,g} k_bg*(2*PS*D*eb + 8) + q + B*Hq*(D+1)*4 [out, lse]
    dense step = sum_b Hkv*n_b*PS*D*2*eb + q + table.
    """
    eb = 2 if w.dtype == "bf16" else 4
    B, Hq, Hkv, D, PS = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size
    q_bytes = B * Hq * D * eb
    k_total = int(sel_cnt.sum())
    n_total = int(sum(n_pages))
    sparse = (k_total * PS * D * 2 * eb + n_total * Hkv * 2 * D * eb + q_bytes
              + n_total * 4 + k_total * 4)
    attn = k_total * (2 * PS * D * eb + 8) + q_bytes + B * Hq * S * (D + 2) * 4
    # the attention + merge kernel of the two-launch step: reads the selected list, the
    # table entries and pages, and (last CTA of each group) writes out and lse; its split
    # partials stay an internal round trip and are not counted
    step_attn = k_total * (2 * PS * D * eb + 8) + q_bytes + B * Hq * (D + 1) * 4
    dense = n_total * Hkv * PS * D * 2 * eb + q_bytes + n_total * 4
    return dict(sparse_step=sparse, attn_launch=attn, step_attn_launch=step_attn,
                scores_bytes=n_total * Hkv * 4, dense_step=dense, selected_pages=k_total,
                pages=n_total * Hkv)



# ----------------------------------------------------------------------------- shared timing

# Configurations measured after the headline one (workload, index of its keep ratio): the rest
# of the metric's 32K-1M range.
EXTRA_CONFIGS = (("llama8b_128k", 0), ("llama8b_128k", 1), ("batched_serving", 0),
                 ("llama70b_1m", 0))


def capture_graph(fn):
    """One CUDA graph of fn() (captured on a side stream, as torch requires)."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    return g


def time_replays(graph, steps, flush):
    """Event-timed replays of graph, L2 flushed before each (outside the events); µs."""
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    res = []
    for _ in range(steps):
        flush.zero_()
        t0.record()
        graph.replay()
        t1.record()
        torch.cuda.synchronize()
        res.append(t0.elapsed_time(t1) * 1e3)
    return res


def spread(xs):
    """Median, p10, p90 and mean. Event-timed steps on this part come in steps of about
    1.02 us, so a median can sit on either of two adjacent steps; the mean dithers between
    them."""
    return {"median": round(statistics.median(xs), 3), "p10": round(pct(xs, 10), 3),
            "p90": round(pct(xs, 90), 3), "mean": round(statistics.mean(xs), 3)}


def window_byte_account(w, k_total, n_total):
    """Algorithmic bytes of the KV-window step (the last k pages of every group, no scoring):
    selected K+V, q, table entries and indices; no statistics."""
    eb = 2 if w.dtype == "bf16" else 4
    return (k_total * w.page_size * w.head_dim * 2 * eb
            + w.batch * w.num_q_heads * w.head_dim * eb + n_total * 4 + k_total * 4)


def oracle_group_baseline(c, w, keep, budget_s, b=0, g=0):
    """The float64 oracle's sparse step (scores, top-k, attention; statistics prebuilt) on ONE
    (sequence, KV head) group of the workload, repeated for about budget_s seconds, scaled to a
    whole step by the pages of every group over the pages of this one."""
    import oracle
    PS, G = w.page_size, w.group_size
    n = oracle.num_pages(int(c.seq_lens[b]), PS)
    phys = c.page_table[b, :n].to(torch.int64)
    f32 = lambda t: t.detach().cpu().to(torch.float32).numpy()  # noqa: E731
    K = f32(c.k_pool.index_select(0, phys)[:, g:g + 1])
    V = f32(c.v_pool.index_select(0, phys)[:, g:g + 1])
    q = f32(c.q[b:b + 1, g * G:(g + 1) * G]).astype(np.float64)
    table = np.arange(n, dtype=np.int64)[None, :]
    lens = np.array([int(c.seq_lens[b])])
    mn, mx = oracle.page_stats(K, table, lens, PS)
    if "keep_pages" in keep:
        k = min(n, keep["keep_pages"])
    elif "budget_pages" in keep:
        k = oracle.keep_count(n, budget_tokens=keep["budget_pages"] * PS, page_size=PS)
    else:
        k = oracle.keep_count(n, ratio=keep["keep_ratio"])
    times, cpu_t = [], []
    t_end = time.perf_counter() + budget_s
    while not times or time.perf_counter() < t_end:
        c0, w0 = time.process_time(), time.perf_counter()
        sc = oracle.page_scores(q, mn, mx, table, lens, PS)
        sel = oracle.select_all_groups(sc, [k])
        oracle.attend(q, K, V, table, lens, PS, w.sm_scale, selected=sel)
        times.append((time.perf_counter() - w0) * 1e6)
        cpu_t.append((time.process_time() - c0) * 1e6)
    total_pages = sum(c.pages_per_seq) * w.num_kv_heads
    scale = total_pages / max(n, 1)
    cores = max(1, round(sum(cpu_t) / sum(times)))
    return {"value": round(statistics.median(times) * scale, 1), "unit": "us/step",
            "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} runs of the float64 oracle's sparse step on one (sequence, "
                      f"KV head) group of {w.name} ({n} pages, statistics prebuilt); value "
                      f"scaled to the whole step by the {total_pages} pages of all groups / "
                      f"{n}"}


def measure_config(name, keep_index, args, dev, flush, peak, peak_kind):
    """One configuration of the metric's range: the sparse step and the dense step through
    kv_decode_step (L2 flushed before each), the FP8-statistics step, the KV-window step
    through the same attention kernel, the attention kernel's roofline, the dropped mass and a
    bounded oracle baseline."""
    import sparse_kv_cache_build_gb300 as skv
    from sparse_kv_cache_build_gb300 import binding, inputs

    w = inputs.workload(name)
    label, keep = keep_setting(w, keep_index)
    c = inputs.make_cache(w, dev)
    kv = skv.PagedKV.from_cache(c)
    B, Hq, Hkv, D, PS = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size
    stats = skv.kv_build_page_stats(kv)
    stats8, exps8 = skv.kv_build_page_stats_fp8(kv)
    step_kw = dict(keep_ratio=keep.get("keep_ratio", 1.0), budget_pages=keep.get("budget_pages", 0))
    k_max = skv.max_keep_pages(kv.stride, keep.get("keep_ratio"), keep.get("budget_pages"))
    ws = torch.zeros((skv.kv_decode_step_workspace_size(kv, Hq, k_max),), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    plan, S = skv.kv_decode_step_plan(kv, Hq, k_max=k_max, **step_kw)
    dense_plan, S_dense = skv.kv_decode_step_plan(kv, Hq, keep_ratio=1.0)
    scores = torch.empty((B, Hkv, kv.stride), dtype=torch.float32, device=dev)
    sel = torch.empty((B, Hkv, k_max), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device=dev)
    ml = torch.empty((B, Hq, S, 2), dtype=torch.float32, device=dev)
    ctr = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)
    ctr2 = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)

    def sparse():
        skv.kv_decode_step(kv, c.q, w.sm_scale, stats, k_max=k_max, out=out, lse=lse,
                           workspace=ws, **step_kw)

    def dense():
        skv.kv_decode_step(kv, c.q, w.sm_scale, keep_ratio=1.0, out=out, lse=lse, workspace=ws)

    def fp8():
        skv.kv_decode_step_fp8(kv, c.q, w.sm_scale, stats8, exps8, k_max=k_max, out=out, lse=lse,
                               workspace=ws, **step_kw)

    # the KV window: the last k pages of every group, no scoring, same attention kernel
    local = k_max
    sel_w = torch.empty((B, Hkv, local), dtype=torch.int32, device=dev)
    cnt_w = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    S_w = skv.kv_auto_num_splits(kv, Hq, local)
    acc_w = torch.empty((B, Hq, S_w, D), dtype=torch.float32, device=dev)
    ml_w = torch.empty((B, Hq, S_w, 2), dtype=torch.float32, device=dev)
    ctr_w = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)

    def window():
        skv.kv_select_structured(None, c.seq_lens, PS, B, Hkv, kv.stride, sink_pages=0,
                                 local_pages=local, k_max=local, sel_idx=sel_w, sel_cnt=cnt_w)
        skv.kv_decode_attn_merge(kv, c.q, w.sm_scale, sel_w, cnt_w, num_splits=S_w,
                                 part_acc=acc_w, part_ml=ml_w, counters=ctr_w, out=out, lse=lse)

    # the step's kernels one by one with events between them (kernel durations)
    marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
    two_launch = plan in (1, 2, 6, 7)

    def marked():
        marks[0].record()
        if plan in (1, 6):
            skv.kv_score_pages(kv, c.q, stats, scores)
        else:
            skv.kv_score_select(kv, c.q, stats, k_max=k_max, scores=scores, counters=ctr,
                                sel_idx=sel, sel_cnt=cnt, **step_kw)
        marks[1].record()
        if plan in (1, 6):
            skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores, k_max=k_max, num_splits=S,
                                      part_acc=acc, part_ml=ml, counters=ctr2, out=out,
                                      lse=lse, sel_idx=sel, sel_cnt=cnt, merge=plan == 1,
                                      **step_kw)
        elif plan == 2:
            skv.kv_decode_attn_merge(kv, c.q, w.sm_scale, sel, cnt, num_splits=S, part_acc=acc,
                                     part_ml=ml, counters=ctr2, out=out, lse=lse)
        else:
            skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=S,
                                      part_acc=acc, part_ml=ml)
        marks[2].record()
        if plan in (6, 7):
            skv.kv_merge_splits(acc, ml, out, lse)

    fns = [sparse, dense, fp8, window] + ([marked] if two_launch else [])
    for _ in range(max(1, args.warmup)):
        for f in fns:
            f()
    torch.cuda.synchronize()
    st, flags = skv.kv_check_device_errors()
    if st != 0:
        raise RuntimeError(f"{name}: device error word {flags:#x} after warm-up")
    graphs = [capture_graph(f) for f in fns]
    for _ in range(args.warmup):
        for g in graphs:
            flush.zero_()
            g.replay()
    torch.cuda.synchronize()
    steps = args.steps
    sparse_us = time_replays(graphs[0], steps, flush)
    dense_us = time_replays(graphs[1], steps, flush)
    fp8_us = time_replays(graphs[2], steps, flush)
    window_us = time_replays(graphs[3], steps, flush)
    attn_us = []
    if two_launch:
        for _ in range(steps):
            flush.zero_()
            graphs[4].replay()
            torch.cuda.synchronize()
            attn_us.append(marks[1].elapsed_time(marks[2]) * 1e3)
    st, flags = skv.kv_check_device_errors()
    if st != 0:
        raise RuntimeError(f"{name}: device error word {flags:#x} after the timed region")

    # bytes, roofline, dropped mass (outside the timed regions)
    marked()
    window()
    torch.cuda.synchronize()
    sel_cnt = cnt.cpu().numpy()
    acct = byte_account(w, c.pages_per_seq, sel_cnt, S)
    w_bytes = window_byte_account(w, int(cnt_w.sum()), int(sum(c.pages_per_seq)))
    delta = float(skv.kv_dropped_mass(kv, c.q, w.sm_scale, sel, cnt).mean())
    sparse_med, dense_med = statistics.median(sparse_us), statistics.median(dense_us)
    window_med = statistics.median(window_us)
    res = {
        "workload": w.name, "description": w.description, "keep": label,
        "context_tokens": int(c.seq_lens.sum()),
        "step_path": f"kv_decode_step plan {plan}: {binding.PLANS[plan]}, {S} splits",
        "dense_path": f"kv_decode_step plan {dense_plan}: {binding.PLANS[dense_plan]}, "
                      f"{S_dense} splits",
        "sparse_us": spread(sparse_us), "dense_us": spread(dense_us),
        "speedup_vs_dense": round(dense_med / sparse_med, 3),
        "byte_bound": round(acct["dense_step"] / acct["sparse_step"], 3),
        "step_gbs": {"sparse": round(acct["sparse_step"] / (sparse_med * 1e-6) / 1e9, 1),
                     "dense": round(acct["dense_step"] / (dense_med * 1e-6) / 1e9, 1)},
        "kernel_cost_beyond_bytes_us": round(
            sparse_med - dense_med * acct["sparse_step"] / acct["dense_step"], 3),
        "fp8_stats_step_us": spread(fp8_us),
        "kv_window": {"us": spread(window_us), "pages_per_group": local,
                      "speedup_vs_dense": round(dense_med / window_med, 3),
                      "byte_bound": round(acct["dense_step"] / w_bytes, 3),
                      "path": "kv_select_structured (sink 0, last k pages, no scores), then "
                              f"kv_decode_attn_merge, {S_w} splits"},
        "dropped_mass_mean": round(delta, 5),
        "bytes": {"sparse_step": acct["sparse_step"], "dense_step": acct["dense_step"],
                  "kv_window_step": w_bytes},
    }
    if attn_us:
        roof_bytes = ((acct["step_attn_launch"] if plan in (1, 2) else acct["attn_launch"])
                      + (acct["scores_bytes"] if plan in (1, 6) else 0))
        a_us = statistics.mean(attn_us)
        ach = roof_bytes / (a_us * 1e-6) / 1e9
        dense_mean = statistics.mean(dense_us)
        res["roofline"] = {
            "kernel": "split_attn_mma_kernel" + {1: " (select + attend + merge)",
                                                 2: " (attend + merge)", 6: " (select + attend)",
                                                 7: " (attend)"}[plan],
            "bound": "hbm", "achieved": round(ach, 1), "peak": peak, "peak_kind": peak_kind,
            "unit": "GB/s", "frac": round(ach / peak, 4),
            "traffic": committed_traffic(w.name, label, ATTN_KERNEL[w.dtype][1]),
            "algorithmic_bytes_per_launch": roof_bytes, "avg_launch_us": round(a_us, 3),
            "dense_same_kernel": {
                "achieved": round(acct["dense_step"] / (dense_mean * 1e-6) / 1e9, 1),
                "frac": round(acct["dense_step"] / (dense_mean * 1e-6) / 1e9 / peak, 4),
                "avg_launch_us": round(dense_mean, 3)}}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = oracle_group_baseline(c, w, keep, args.config_cpu_seconds)
    n_step = 3 if plan in (6, 7) else (2 if plan in (1, 2) else 4)
    res["gpu_launches"] = steps * (n_step + (1 if dense_plan in (3, 5) else 2) + n_step + 2
                                   + (n_step if attn_us else 0))
    del c, kv, stats, stats8, exps8, ws, graphs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def measure_entmax_pruning(args, dev, flush):
    """The entmax step (page moments, Gaussian-aware selection, entmax over the kept pages)
    against dense entmax over every page, on the workload whose page boxes are tight enough
    for the selector to prune."""
    import sparse_kv_cache_build_gb300 as skv
    from sparse_kv_cache_build_gb300 import binding, inputs
    w = inputs.workload("entmax_pruning_32k")
    c = inputs.make_cache(w, dev)
    kv = skv.PagedKV.from_cache(c)
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    stats = skv.kv_build_page_stats(kv)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    tau = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = torch.zeros((skv.kv_entmax_decode_step_workspace_size(kv, Hq, kv.stride),),
                     dtype=torch.uint8, device=dev)
    wsd = torch.empty((int(binding.lib().kv_entmax_attn_workspace_size(kv.ref(), Hq, 0)),),
                      dtype=torch.uint8, device=dev)

    def step():
        skv.kv_entmax_decode_step(kv, c.q, w.sm_scale, stats, k_max=kv.stride, out=out, tau=tau,
                                  workspace=ws)

    def dense():
        skv.kv_entmax_decode_attn(kv, c.q, w.sm_scale, out=out, tau=tau, workspace=wsd)

    for _ in range(max(1, args.warmup)):
        step()
        dense()
    torch.cuda.synchronize()
    gs, gd = capture_graph(step), capture_graph(dense)
    for _ in range(args.warmup):
        time_replays(gs, 1, flush)
        time_replays(gd, 1, flush)
    step_us = time_replays(gs, args.steps, flush)
    dense_us = time_replays(gd, args.steps, flush)
    step()
    torch.cuda.synchronize()
    M = (B * Hq * kv.stride * 4 + 255) // 256 * 256
    cb = 3 * M + (B * Hkv * kv.stride * 4 + 255) // 256 * 256
    kept = int(ws[cb: cb + B * Hkv * 4].view(torch.int32).sum())
    st, flags = skv.kv_check_device_errors()
    if st != 0:
        raise RuntimeError(f"entmax pruning: device error word {flags:#x}")
    res = {"workload": w.name, "description": w.description, "step_us": spread(step_us),
           "dense_us": spread(dense_us),
           "speedup_vs_dense": round(statistics.median(dense_us) / statistics.median(step_us), 3),
           "kept_pages": kept, "pages": int(B * Hkv * kv.stride),
           "gpu_launches": args.steps * (5 + 3)}
    del c, kv, stats, ws, wsd
    torch.cuda.empty_cache()
    return res


def run_block_child(args):
    """One fresh-process block: the headline sparse and dense steps, replayed alternately
    (L2 flushed before each), printed as one JSON line for the parent."""
    import sparse_kv_cache_build_gb300 as skv
    from sparse_kv_cache_build_gb300 import binding, inputs
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    binding.lib()
    w = inputs.workload(args.workload)
    label, keep = keep_setting(w, args.keep_index)
    c = inputs.make_cache(w, dev)
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    step_kw = dict(keep_ratio=keep.get("keep_ratio", 1.0), budget_pages=keep.get("budget_pages", 0))
    k_max = skv.max_keep_pages(kv.stride, keep.get("keep_ratio"), keep.get("budget_pages"))
    ws = torch.zeros((skv.kv_decode_step_workspace_size(kv, w.num_q_heads, k_max),),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev)
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)

    def sparse():
        skv.kv_decode_step(kv, c.q, w.sm_scale, stats, k_max=k_max, out=out, workspace=ws,
                           **step_kw)

    def dense():
        skv.kv_decode_step(kv, c.q, w.sm_scale, keep_ratio=1.0, out=out, workspace=ws)

    for _ in range(args.warmup):
        sparse()
        dense()
    gs, gd = capture_graph(sparse), capture_graph(dense)
    for _ in range(args.warmup):
        time_replays(gs, 1, flush)
        time_replays(gd, 1, flush)
    sp, de = [], []
    for _ in range(args.steps):
        sp += time_replays(gs, 1, flush)
        de += time_replays(gd, 1, flush)
    st, flags = skv.kv_check_device_errors()
    if st != 0:
        raise RuntimeError(f"device error word {flags:#x}")
    print(json.dumps({"sparse_us": sp, "dense_us": de}), flush=True)


def run_blocks(args, n_blocks):
    """n_blocks fresh processes, each timing the headline sparse and dense steps alternately:
    per-block medians, paired dense/sparse ratios, and 95 % intervals of the mean over blocks
    from 10,000 resamples of the blocks."""
    per = []
    for i in range(n_blocks):
        cmd = [sys.executable, os.path.abspath(__file__), "--block-child", "--workload",
               args.workload, "--keep-index", str(args.keep_index), "--steps",
               str(args.block_steps), "--warmup", str(args.warmup)]
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
        if r.returncode != 0:
            raise RuntimeError(f"block {i} failed: {r.stderr[-2000:]}")
        d = json.loads(r.stdout.strip().splitlines()[-1])
        per.append((statistics.median(d["sparse_us"]), statistics.median(d["dense_us"])))
    sp = np.array([p[0] for p in per])
    de = np.array([p[1] for p in per])
    ratio = de / sp
    rng = np.random.default_rng(12345)
    idx = rng.integers(0, n_blocks, size=(10000, n_blocks))

    def ci(x):
        m = x[idx].mean(axis=1)
        return [round(float(np.percentile(m, 2.5)), 3), round(float(np.percentile(m, 97.5)), 3)]

    return {"blocks": n_blocks, "steps_per_block": args.block_steps,
            "sparse_us_per_block": [round(float(x), 3) for x in sp],
            "dense_us_per_block": [round(float(x), 3) for x in de],
            "paired_speedup_per_block": [round(float(x), 4) for x in ratio],
            "sparse_us_mean": round(float(sp.mean()), 3), "sparse_us_ci95": ci(sp),
            "dense_us_mean": round(float(de.mean()), 3), "dense_us_ci95": ci(de),
            "paired_speedup_mean": round(float(ratio.mean()), 4),
            "paired_speedup_ci95": ci(ratio),
            "method": "fresh process per block (sub-process); within a block the sparse and "
                      "dense steps alternate, L2 flushed before each; ratio = dense median / "
                      "sparse median of the block; interval = 2.5/97.5 percentiles of the mean "
                      "over 10,000 resamples of the blocks"}


# ----------------------------------------------------------------------------- our arm

def keep_setting(w, which=0):
    if w.keep_pages is not None:
        return f"top{w.keep_pages}", dict(keep_pages=w.keep_pages)
    if w.budget_tokens is not None:
        bp = w.budget_tokens // w.page_size
        return f"budget{bp}", dict(budget_pages=bp)
    r = w.keep_ratios[which]
    return f"r{r:.3g}", dict(keep_ratio=r)


def run_ours(args):
    import sparse_kv_cache_build_gb300 as skv
    from sparse_kv_cache_build_gb300 import binding, inputs

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.lib()                                      # fails loudly without the library

    w = inputs.workload(args.workload)
    label, keep = keep_setting(w, args.keep_index)
    c = inputs.make_cache(w, dev)
    kv = skv.PagedKV.from_cache(c)
    B, Hq, Hkv, D, PS = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size
    n_pages = c.pages_per_seq
    stream = torch.cuda.current_stream()

    # statistics build (once per cache; timed on its own)
    stats = torch.empty((kv.k_pool.shape[0], Hkv, 2, D), dtype=kv.dtype, device=dev)
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device=dev)   # 2x L2
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    stats_us = []
    for _ in range(3):
        flush.zero_()
        ev[0].record()
        skv.kv_build_page_stats(kv, stats)
        ev[1].record()
        torch.cuda.synchronize()
        stats_us.append(ev[0].elapsed_time(ev[1]) * 1e3)

    # buffers of the sparse and dense steps (no allocation inside a step)
    if "keep_pages" in keep:
        k_max = keep["keep_pages"]
        keep_t = torch.full((B,), k_max, dtype=torch.int32, device=dev)
        sel_kw = dict(keep=keep_t, k_max=k_max)
        step_kw = None                 # a fixed per-group keep count has no kv_decode_step form
    else:
        k_max = skv.max_keep_pages(kv.stride, keep.get("keep_ratio"), keep.get("budget_pages"))
        sel_kw = dict(keep_ratio=keep.get("keep_ratio", 0.0),
                      budget_pages=keep.get("budget_pages", 0), k_max=k_max)
        step_kw = dict(keep_ratio=keep.get("keep_ratio", 1.0),
                       budget_pages=keep.get("budget_pages", 0))
    S = skv.kv_auto_num_splits(kv, Hq, k_max)
    S_dense = skv.kv_auto_num_splits(kv, Hq, kv.stride)
    scores = torch.empty((B, Hkv, kv.stride), dtype=torch.float32, device=dev)
    sel = torch.empty((B, Hkv, k_max), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device=dev)
    ml = torch.empty((B, Hq, S, 2), dtype=torch.float32, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    acc_d = torch.empty((B, Hq, S_dense, D), dtype=torch.float32, device=dev)
    ml_d = torch.empty((B, Hq, S_dense, 2), dtype=torch.float32, device=dev)
    out_d = torch.empty_like(out)
    lse_d = torch.empty_like(lse)
    # the step's workspace starts zero-filled (its per-group counters return to zero)
    ws = torch.zeros((skv.kv_decode_step_workspace_size(kv, Hq, k_max),), dtype=torch.uint8,
                     device=dev)
    ctr = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)
    ctr2 = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)
    def plan_kernels(which, ev=None):
        """Plan `which`'s kernels one by one (ev: events recorded between them)."""
        if ev is not None:
            ev[0].record()
        if which in (1, 6):
            skv.kv_score_pages(kv, c.q, stats, scores)
        else:
            skv.kv_score_select(kv, c.q, stats, k_max=k_max, scores=scores, counters=ctr,
                                sel_idx=sel, sel_cnt=cnt, **step_kw)
        if ev is not None:
            ev[1].record()
        if which == 1:
            skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores, k_max=k_max, num_splits=S,
                                      part_acc=acc, part_ml=ml, counters=ctr2, out=out,
                                      lse=lse, sel_idx=sel, sel_cnt=cnt, **step_kw)
        elif which == 6:
            skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores, k_max=k_max, num_splits=S,
                                      part_acc=acc, part_ml=ml, sel_idx=sel, sel_cnt=cnt,
                                      merge=False, **step_kw)
        elif which == 2:
            skv.kv_decode_attn_merge(kv, c.q, w.sm_scale, sel, cnt, num_splits=S, part_acc=acc,
                                     part_ml=ml, counters=ctr2, out=out, lse=lse)
        else:
            skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=S,
                                      part_acc=acc, part_ml=ml)
        if ev is not None:
            ev[2].record()
        if which in (6, 7):
            skv.kv_merge_splits(acc, ml, out, lse)
        if ev is not None:
            ev[3].record()

    # the kernels kv_decode_step runs for this shape (KV_PLAN_*)
    plan, S_plan = (skv.kv_decode_step_plan(kv, Hq, k_max=k_max, **step_kw)
                    if step_kw is not None else (0, S))
    dense_plan, _ = skv.kv_decode_step_plan(kv, Hq, keep_ratio=1.0)
    # the staged plans: score (+ select), the attention kernel, and for plans 6 and 7 a
    # merge kernel of its own
    two_launch = plan in (1, 2, 6, 7)
    assert S_plan == S, (S_plan, S)
    # another staged form, timed beside it where the shape allows (for plans 6 and 7: the
    # same kernels with the merge in the attention kernel's last CTA)
    alt_plan = None
    if step_kw is not None:
        for cand in {1: (2,), 2: (1,), 6: (1, 7), 7: (2,)}.get(plan, (1, 2)):
            try:
                plan_kernels(cand)
                alt_plan = cand
                break
            except binding.KVError:
                continue
        torch.cuda.synchronize()

    try:
        marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
        smarks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
        in_graph_events = True
    except TypeError:
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        smarks = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        in_graph_events = False

    def plan_step(which, with_marks=False):
        """A staged plan's kernels, called one by one through the C ABI."""
        plan_kernels(which, smarks if with_marks else None)

    def two_launch_step(with_marks):
        plan_step(plan, with_marks)

    def alt_step():
        plan_step(alt_plan)

    def four_kernel_step(with_marks):
        if with_marks:
            marks[0].record()
        skv.kv_score_pages(kv, c.q, stats, scores)
        if with_marks:
            marks[1].record()
        skv.kv_select_topk(scores, c.seq_lens, PS, sel_idx=sel, sel_cnt=cnt, **sel_kw)
        if with_marks:
            marks[2].record()
        skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, sel, cnt, num_splits=S, part_acc=acc,
                                  part_ml=ml)
        if with_marks:
            marks[3].record()
        skv.kv_merge_splits(acc, ml, out, lse)
        if with_marks:
            marks[4].record()

    def step():
        """The call a user makes for one sparse decode step (one launch where possible)."""
        if step_kw is None:
            four_kernel_step(False)
        else:
            skv.kv_decode_step(kv, c.q, w.sm_scale, stats, k_max=k_max, out=out, lse=lse,
                               workspace=ws, **step_kw)

    # FP8 statistics (built once, like the bf16 ones): the same step scoring from 1-byte stats
    stats8 = exps8 = None
    if step_kw is not None:
        stats8, exps8 = skv.kv_build_page_stats_fp8(kv)

    def fp8_step():
        skv.kv_decode_step_fp8(kv, c.q, w.sm_scale, stats8, exps8, k_max=k_max, out=out,
                               lse=lse, workspace=ws, **step_kw)

    # entmax decoding (1.5-entmax): the Gaussian-aware selection step and dense entmax
    ent_ws = torch.empty((skv.kv_entmax_decode_step_workspace_size(kv, Hq, kv.stride),),
                         dtype=torch.uint8, device=dev)
    ent_dws = torch.empty((int(binding.lib().kv_entmax_attn_workspace_size(kv.ref(), Hq, 0)),),
                          dtype=torch.uint8, device=dev)
    ent_out = torch.empty_like(out)
    ent_tau = torch.empty_like(lse)

    def entmax_step():
        skv.kv_entmax_decode_step(kv, c.q, w.sm_scale, stats, k_max=kv.stride, out=ent_out,
                                  tau=ent_tau, workspace=ent_ws)

    def entmax_dense():
        skv.kv_entmax_decode_attn(kv, c.q, w.sm_scale, out=ent_out, tau=ent_tau,
                                  workspace=ent_dws)

    # the KV window: the last k pages of every group (no scoring) through the same kernel
    sel_w = torch.empty((B, Hkv, k_max), dtype=torch.int32, device=dev)
    cnt_w = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    S_w = skv.kv_auto_num_splits(kv, Hq, k_max)
    acc_w = torch.empty((B, Hq, S_w, D), dtype=torch.float32, device=dev)
    ml_w = torch.empty((B, Hq, S_w, 2), dtype=torch.float32, device=dev)
    ctr_w = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)
    out_w, lse_w = torch.empty_like(out), torch.empty_like(lse)

    def window_step():
        skv.kv_select_structured(None, c.seq_lens, PS, B, Hkv, kv.stride, sink_pages=0,
                                 local_pages=k_max, k_max=k_max, sel_idx=sel_w, sel_cnt=cnt_w)
        skv.kv_decode_attn_merge(kv, c.q, w.sm_scale, sel_w, cnt_w, num_splits=S_w,
                                 part_acc=acc_w, part_ml=ml_w, counters=ctr_w, out=out_w,
                                 lse=lse_w)

    def one_launch_step():
        """The step as one cluster launch (where the shape allows it)."""
        skv.kv_decode_step(kv, c.q, w.sm_scale, stats, k_max=k_max, out=out, lse=lse,
                           workspace=ws, num_splits=skv.ONE_LAUNCH, **step_kw)

    def dense_step():
        """The same call with every page kept: the same kernel, no scoring or selection."""
        if step_kw is None:
            skv.kv_sparse_decode_attn(kv, c.q, w.sm_scale, None, None, num_splits=S_dense,
                                      part_acc=acc_d, part_ml=ml_d)
            skv.kv_merge_splits(acc_d, ml_d, out_d, lse_d)
        else:
            skv.kv_decode_step(kv, c.q, w.sm_scale, keep_ratio=1.0, out=out_d, lse=lse_d,
                               workspace=ws)

    # warm up eagerly (this also fixes each shape's launch configuration)
    for _ in range(max(1, args.warmup)):
        step()
        dense_step()
        four_kernel_step(False)
        if step_kw is not None:
            fp8_step()
        entmax_step()
        entmax_dense()
        if step_kw is not None:
            window_step()
    torch.cuda.synchronize()
    st, flags = skv.kv_check_device_errors()
    if st != 0:
        raise RuntimeError(f"device error word {flags:#x} after warm-up")
    one_launch = plan == 5
    one_launch_ran = (step_kw is not None and
                      skv.kv_decode_step_plan(kv, Hq, k_max=k_max, num_splits=skv.ONE_LAUNCH,
                                              **step_kw)[0] == 5)

    # one CUDA graph per measured step; g_marked and g_smarked are the four-kernel and the
    # two-launch steps with event nodes between their kernels, replayed in their own flushed
    # loops to time each kernel (event nodes sit between the kernels, so their programmatic
    # launch overlap is lost there: those graphs time kernels, not steps)
    g_step, g_dense, g_four, g_marked, g_one, g_smarked, g_alt, g_fp8, g_ent, g_entd, g_win = (
        torch.cuda.CUDAGraph() for _ in range(11))
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_step, stream=side):
            step()
        with torch.cuda.graph(g_dense, stream=side):
            dense_step()
        with torch.cuda.graph(g_four, stream=side):
            four_kernel_step(False)
        with torch.cuda.graph(g_ent, stream=side):
            entmax_step()
        with torch.cuda.graph(g_entd, stream=side):
            entmax_dense()
        if in_graph_events:
            with torch.cuda.graph(g_marked, stream=side):
                four_kernel_step(True)
            if two_launch:
                with torch.cuda.graph(g_smarked, stream=side):
                    two_launch_step(True)
        if step_kw is not None:
            with torch.cuda.graph(g_one, stream=side):
                one_launch_step()
            with torch.cuda.graph(g_fp8, stream=side):
                fp8_step()
            with torch.cuda.graph(g_win, stream=side):
                window_step()
        if alt_plan is not None:
            with torch.cuda.graph(g_alt, stream=side):
                alt_step()
    stream.wait_stream(side)
    torch.cuda.synchronize()

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        for g_ in (g_step, g_dense, g_four):
            flush.zero_()
            g_.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    def timed(graph):
        res = []
        for _ in range(args.steps):
            flush.zero_()
            t0.record()
            graph.replay()
            t1.record()
            torch.cuda.synchronize()
            res.append(t0.elapsed_time(t1) * 1e3)
        return res

    # ---- timed region: K steps of each kind, L2 flushed before every step ---------------
    kern_us = {"score": [], "select": [], "attn": [], "merge": []}
    step_kern_us = {"first": [], "attention": [], "merge": []}
    barrier()
    with ClockSampler(local) as clk:
        step_us = timed(g_step)
        barrier()
        dense_us = timed(g_dense)
        barrier()
        four_us = timed(g_four)
        barrier()
        one_us = timed(g_one) if one_launch_ran else []
        barrier()
        fp8_us = timed(g_fp8) if step_kw is not None else []
        barrier()
        win_us = timed(g_win) if step_kw is not None else []
        barrier()
        ent_us = timed(g_ent)
        barrier()
        entd_us = timed(g_entd)
        barrier()
        alt_us = timed(g_alt) if alt_plan is not None else []
        barrier()
        if in_graph_events:
            for _ in range(args.steps):
                flush.zero_()
                g_marked.replay()
                torch.cuda.synchronize()
                for i, k in enumerate(kern_us):
                    kern_us[k].append(marks[i].elapsed_time(marks[i + 1]) * 1e3)
            for _ in range(args.steps if two_launch else 0):
                flush.zero_()
                g_smarked.replay()
                torch.cuda.synchronize()
                for i, k in enumerate(step_kern_us):
                    if k != "merge" or plan in (6, 7):
                        step_kern_us[k].append(smarks[i].elapsed_time(smarks[i + 1]) * 1e3)
        barrier()
    clocks = clk.summary()

    if not in_graph_events:        # per-kernel times from eager launches instead
        for _ in range(args.steps):
            flush.zero_()
            four_kernel_step(True)
            torch.cuda.synchronize()
            for i, k in enumerate(kern_us):
                kern_us[k].append(marks[i].elapsed_time(marks[i + 1]) * 1e3)
        for _ in range(args.steps if two_launch else 0):
            flush.zero_()
            two_launch_step(True)
            torch.cuda.synchronize()
            for i, k in enumerate(step_kern_us):
                if k != "merge" or plan in (6, 7):
                    step_kern_us[k].append(smarks[i].elapsed_time(smarks[i + 1]) * 1e3)

    st, flags = skv.kv_check_device_errors()
    if st != 0:
        raise RuntimeError(f"device error word {flags:#x} after the timed region")
    four_kernel_step(False)
    torch.cuda.synchronize()
    sel_cnt = cnt.cpu().numpy()
    acct = byte_account(w, n_pages, sel_cnt, S)
    # pages the entmax selector kept (read back from the step's workspace)
    entmax_step()
    torch.cuda.synchronize()
    M = (B * Hq * kv.stride * 4 + 255) // 256 * 256
    cb = 3 * M + (B * Hkv * kv.stride * 4 + 255) // 256 * 256
    ent_kept = int(ent_ws[cb: cb + B * Hkv * 4].view(torch.int32).sum())

    win_bytes = None
    if step_kw is not None:
        window_step()
        torch.cuda.synchronize()
        win_bytes = window_byte_account(w, int(cnt_w.sum()), int(sum(n_pages)))

    # dropped mass of this step (diagnostic, outside every timed region)
    delta = skv.kv_dropped_mass(kv, c.q, w.sm_scale, sel, cnt)
    delta_mean = float(delta.mean())

    # ---- end to end through the public API, host buffers, copies inside the timing -------
    # (1) the captured step (kv_decode_step_graph_*), the call a serving loop makes per token:
    #     one launch runs the step, its kernels reading the query from and writing the output
    #     to pinned host memory in place (the device addresses it); then the host waits;
    # (2) the same copies around a direct kv_decode_step call through the binding.
    q_host = c.q.detach().cpu().pin_memory()
    out_host = torch.empty((B, Hq, D), dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(c.q)
    e2e_us, e2e_direct_us = [], []
    if step_kw is not None:
        ws_g = torch.zeros_like(ws)
        sg = skv.DecodeStepGraph(kv, q_dev, w.sm_scale, stats, k_max=k_max, workspace=ws_g,
                                 q_host=q_host, out_host=out_host, **step_kw)
        for graph_call, res in ((True, e2e_us), (False, e2e_direct_us)):
            for i in range(args.warmup + min(args.steps, 500)):
                flush.zero_()
                torch.cuda.synchronize()
                h0 = time.perf_counter()
                if graph_call:
                    sg.launch()
                else:
                    q_dev.copy_(q_host, non_blocking=True)
                    g_out, _ = skv.kv_decode_step(kv, q_dev, w.sm_scale, stats, k_max=k_max,
                                                  out=out, lse=lse, workspace=ws, **step_kw)
                    out_host.copy_(g_out, non_blocking=True)
                torch.cuda.synchronize()
                if i >= args.warmup:
                    res.append((time.perf_counter() - h0) * 1e6)
        sg.close()

    # ---- max over ranks ------------------------------------------------------------------
    sparse_med = statistics.median(step_us)
    mean_us = sum(step_us) / len(step_us)
    mean_us, sparse_med = max_over_ranks([mean_us, sparse_med], world, dev)
    if rank != 0:
        return None

    peak, peak_kind = measured_peaks()
    attn_us = statistics.mean(kern_us["attn"]) if kern_us["attn"] else float("nan")
    dense_med = statistics.median(dense_us)
    step_mean = statistics.mean(step_us)
    dense_mean = statistics.mean(dense_us)
    if one_launch:
        # the step is a single kernel: its duration is the event-timed step
        roof_kernel, roof_bytes, roof_us = "fused_step_kernel", acct["sparse_step"], step_mean
        roof_source = os.path.join(CSRC, "step_fused.cu")
    elif two_launch:
        roof_kernel = ATTN_KERNEL[w.dtype][0] + {1: " (select + attend + merge)",
                                                 2: " (attend + merge)",
                                                 6: " (select + attend)", 7: " (attend)"}[plan]
        roof_bytes = ((acct["step_attn_launch"] if plan in (1, 2) else acct["attn_launch"])
                      + (acct["scores_bytes"] if plan in (1, 6) else 0))
        roof_us = statistics.mean(step_kern_us["attention"])
        roof_source = ATTN_KERNEL[w.dtype][1]
    else:
        roof_kernel, roof_bytes, roof_us = ATTN_KERNEL[w.dtype][0], acct["attn_launch"], attn_us
        roof_source = ATTN_KERNEL[w.dtype][1]
    achieved = roof_bytes / (roof_us * 1e-6) / 1e9
    # kernels per replay of each timed graph
    n_step = 1 if one_launch else ((3 if plan in (6, 7) else 2) if two_launch else 4)
    n_dense = 1 if dense_plan in (3, 5) else 2
    line = {
        "metric": METRIC,
        "value": round(sparse_med, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_us / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": w.name, "description": w.description, "batch": B,
            "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D, "page_size": PS,
            "context_tokens": int(c.seq_lens.sum()), "kv_storage": w.dtype, "keep": label,
            "step_path": f"kv_decode_step plan {plan}: {binding.PLANS[plan]}, {S} splits",
            "dense_path": f"kv_decode_step plan {dense_plan}: {binding.PLANS[dense_plan]}",
            "num_splits_four_kernel": S, "parallelism": f"replicas{world}",
            "l2": "flushed before every timed step (256 MiB write = 2x L2, outside the events)",
            "graph": "one CUDA graph per step, replayed once per timed step",
        },
        "sparse_us": {"median": round(sparse_med, 3), "p10": round(pct(step_us, 10), 3),
                      "p90": round(pct(step_us, 90), 3)},
        "dense_us": {"median": round(dense_med, 3), "p10": round(pct(dense_us, 10), 3),
                     "p90": round(pct(dense_us, 90), 3)},
        "speedup_vs_dense": round(dense_med / sparse_med, 3),
        "byte_bound": round(acct["dense_step"] / acct["sparse_step"], 3),
        "step_gbs": {"sparse": round(acct["sparse_step"] / (sparse_med * 1e-6) / 1e9, 1),
                     "dense": round(acct["dense_step"] / (dense_med * 1e-6) / 1e9, 1)},
        "one_launch_step_us": (round(statistics.median(one_us), 3) if one_us else None),
        "entmax": {"step_us": round(statistics.median(ent_us), 3),
                   "dense_us": round(statistics.median(entd_us), 3),
                   "speedup_vs_dense": round(statistics.median(entd_us)
                                             / statistics.median(ent_us), 3),
                   "kept_pages": ent_kept,
                   "path": "kv_entmax_decode_step (moments, Gaussian-aware select, logits, "
                           "threshold + output) vs kv_entmax_decode_attn over every page"},
        "fp8_stats_step_us": ({"median": round(statistics.median(fp8_us), 3),
                               "speedup_vs_dense": round(dense_med / statistics.median(fp8_us), 3),
                               "stats_bytes_per_step": acct["pages"] * (2 * D + 1)}
                              if fp8_us else None),
        "other_two_launch_step_us": ({"plan": binding.PLANS[alt_plan],
                                      "median": round(statistics.median(alt_us), 3)}
                                     if alt_us else None),
        "step_kernel_us_marked": ({k: round(statistics.mean(v), 3)
                                   for k, v in step_kern_us.items() if v} or None),
        "four_kernel_step_us": {"median": round(statistics.median(four_us), 3),
                                "kernel_us_marked": {k: round(statistics.mean(v), 3)
                                                     for k, v in kern_us.items() if v}},
        "kv_window": ({"us": spread(win_us), "pages_per_group": k_max,
                       "speedup_vs_dense": round(dense_med / statistics.median(win_us), 3),
                       "byte_bound": round(acct["dense_step"] / win_bytes, 3),
                       "path": "kv_select_structured (sink 0, last k pages, no scores), then "
                               f"kv_decode_attn_merge, {S_w} splits"} if win_us else None),
        "kernel_cost_beyond_bytes_us": round(
            sparse_med - dense_med * acct["sparse_step"] / acct["dense_step"], 3),
        "bytes": acct,
        "stats_build_us": round(statistics.median(stats_us), 3),
        "dropped_mass_mean": round(delta_mean, 5),
        "roofline": {
            "kernel": roof_kernel,
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": committed_traffic(w.name, label, roof_source),
            "algorithmic_bytes_per_launch": roof_bytes,
            "avg_launch_us": round(roof_us, 3),
            "dense_same_kernel": {
                "achieved": round(acct["dense_step"] / (dense_mean * 1e-6) / 1e9, 1),
                "frac": round(acct["dense_step"] / (dense_mean * 1e-6) / 1e9 / peak, 4),
                "avg_launch_us": round(dense_mean, 3)},
        },
        "gpu_launches": args.steps * (n_step + n_dense + 4 + (4 if in_graph_events else 0)
                                      + (n_step if two_launch else 0) + (1 if one_us else 0)
                                      + ({1: 2, 2: 2, 6: 3, 7: 3}.get(alt_plan, 0) if alt_us
                                         else 0)
                                      + (n_step if fp8_us else 0) + 4 + 2
                                      + (2 if win_us else 0)),
        "clocks": clocks,
    }
    if e2e_us:
        line["e2e"] = {"value": round(statistics.median(e2e_us), 3), "unit": "us/step",
                       "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
                       "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
                       "api": "kv_decode_step_graph_launch (the step captured once by "
                              "kv_decode_step_graph_create with q_host and out_host, pinned "
                              "host memory that the step's kernels read and write in place "
                              "over the host link; host waits)",
                       "direct_call_us": round(statistics.median(e2e_direct_us), 3),
                       "direct_call_api": "kv_decode_step through the Python binding"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(c, w, keep, budget_s=args.cpu_seconds)
    if world == 1 and not args.no_configs:
        # the rest of the metric's range, each configuration on its own (the headline cache
        # stays resident; each configuration's cache is freed before the next)
        line["configs"] = {}
        for name, ki in EXTRA_CONFIGS:
            r = measure_config(name, ki, args, dev, flush, peak, peak_kind)
            line["configs"][f"{name}:{r['keep']}"] = r
            line["gpu_launches"] += r.pop("gpu_launches")
    if world == 1 and not args.no_configs:
        r = measure_entmax_pruning(args, dev, flush)
        line["gpu_launches"] += r.pop("gpu_launches")
        line["entmax_pruning"] = r
    if world == 1 and args.blocks > 0:
        line["blocks"] = run_blocks(args, args.blocks)
    return line


# ----------------------------------------------------------------------------- oracle arm

def oracle_inputs(c):
    f32 = lambda t: t.detach().cpu().to(torch.float32).numpy()  # noqa: E731
    return (f32(c.q).astype(np.float64), f32(c.k_pool), f32(c.v_pool),
            c.page_table.cpu().numpy(), c.seq_lens.cpu().numpy())


def oracle_step(oracle, q, K, V, table, lens, mn, mx, w, keep):
    s = oracle.page_scores(q, mn, mx, table, lens, w.page_size)
    ks = []
    for b in range(w.batch):
        n = oracle.num_pages(lens[b], w.page_size)
        if "keep_pages" in keep:
            ks.append(min(n, keep["keep_pages"]))
        elif "budget_pages" in keep:
            ks.append(oracle.keep_count(n, budget_tokens=keep["budget_pages"] * w.page_size,
                                        page_size=w.page_size))
        else:
            ks.append(oracle.keep_count(n, ratio=keep["keep_ratio"]))
    sel = oracle.select_all_groups(s, ks)
    return oracle.attend(q, K, V, table, lens, w.page_size, w.sm_scale, selected=sel)


def time_oracle(c, w, keep, budget_s, min_steps=1, max_steps=None):
    import oracle
    q, K, V, table, lens = oracle_inputs(c)
    mn, mx = oracle.page_stats(K, table, lens, w.page_size)
    times, cpu_t = [], []
    t_end = time.perf_counter() + budget_s
    while (len(times) < min_steps or time.perf_counter() < t_end) and \
            (max_steps is None or len(times) < max_steps):
        c0, w0 = time.process_time(), time.perf_counter()
        oracle_step(oracle, q, K, V, table, lens, mn, mx, w, keep)
        times.append((time.perf_counter() - w0) * 1e6)
        cpu_t.append((time.process_time() - c0) * 1e6)
    cores = max(1, round(sum(cpu_t) / sum(times)))
    return times, cores


def cpu_baseline(c, w, keep, budget_s=15.0):
    times, cores = time_oracle(c, w, keep, budget_s)
    return {"value": round(statistics.median(times), 1), "unit": "us/step", "cores": cores,
            "kind": "oracle",
            "sample": f"{len(times)} full sparse decode steps of {w.name} (scores, top-k, "
                      f"attention; stats prebuilt) by the float64 NumPy oracle; cores = "
                      f"process CPU time / wall time; host has {os.cpu_count()} threads"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    from sparse_kv_cache_build_gb300 import inputs
    w = inputs.workload(args.workload)
    label, keep = keep_setting(w, args.keep_index)
    c = inputs.make_cache(w, "cpu")
    import oracle
    q, K, V, table, lens = oracle_inputs(c)
    mn, mx = oracle.page_stats(K, table, lens, w.page_size)
    for _ in range(args.warmup):
        oracle_step(oracle, q, K, V, table, lens, mn, mx, w, keep)
    times, cpu_t = [], []
    for _ in range(args.steps):
        c0, w0 = time.process_time(), time.perf_counter()
        oracle_step(oracle, q, K, V, table, lens, mn, mx, w, keep)
        times.append((time.perf_counter() - w0) * 1e6)
        cpu_t.append((time.process_time() - c0) * 1e6)
    med = statistics.median(times)
    cores = max(1, round(sum(cpu_t) / sum(times)))
    return {
        "impl": "reference", "metric": METRIC, "value": round(med, 1), "unit": "us/step",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sum(times) / len(times) / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "keep": label,
                   "context_tokens": int(c.seq_lens.sum()), "kv_storage": w.dtype},
        "cpu_baseline": {"value": round(med, 1), "unit": "us/step", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{args.steps} full sparse decode steps of {w.name} by the "
                                   "float64 NumPy oracle (stats prebuilt)"},
        "e2e": {"value": round(med, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_only_step(args):
    """kv_decode_step alone, for a profiler's launch list or capture of its kernels."""
    import sparse_kv_cache_build_gb300 as skv
    from sparse_kv_cache_build_gb300 import binding, inputs

    torch.cuda.set_device(0)
    binding.lib()
    w = inputs.workload(args.workload)
    label, keep = keep_setting(w, args.keep_index)
    c = inputs.make_cache(w, "cuda")
    kv = skv.PagedKV.from_cache(c)
    stats = skv.kv_build_page_stats(kv)
    if args.only_step.startswith("entmax"):
        flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device="cuda")
        ews = torch.empty((skv.kv_entmax_decode_step_workspace_size(kv, w.num_q_heads, kv.stride),),
                          dtype=torch.uint8, device="cuda")
        for _ in range(args.warmup + args.steps):
            flush.zero_()
            if args.only_step == "entmax_step":
                skv.kv_entmax_decode_step(kv, c.q, w.sm_scale, stats, k_max=kv.stride,
                                          workspace=ews)
            else:
                skv.kv_entmax_decode_attn(kv, c.q, w.sm_scale)
        torch.cuda.synchronize()
        st, flags = skv.kv_check_device_errors()
        if st != 0:
            raise RuntimeError(f"device error word {flags:#x}")
        print(f"{w.name} {args.only_step}: {args.warmup + args.steps} calls", flush=True)
        return
    if args.only_step == "dense" or "keep_pages" in keep:
        kw = dict(keep_ratio=1.0)
        k_max = 1
    else:
        kw = dict(keep_ratio=keep.get("keep_ratio", 1.0), budget_pages=keep.get("budget_pages", 0))
        k_max = skv.max_keep_pages(kv.stride, keep.get("keep_ratio"), keep.get("budget_pages"))
    ws = torch.zeros((skv.kv_decode_step_workspace_size(kv, w.num_q_heads, k_max),),
                     dtype=torch.uint8, device="cuda")
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device="cuda")
    for _ in range(args.warmup + args.steps):
        flush.zero_()
        skv.kv_decode_step(kv, c.q, w.sm_scale, stats, k_max=k_max, workspace=ws, **kw)
    torch.cuda.synchronize()
    st, flags = skv.kv_check_device_errors()
    if st != 0:
        raise RuntimeError(f"device error word {flags:#x}")
    plan, S = skv.kv_decode_step_plan(kv, w.num_q_heads, k_max=k_max, **kw)
    print(f"{w.name} {label if args.only_step == 'sparse' else 'dense'}: "
          f"{args.warmup + args.steps} steps, plan {plan} ({binding.PLANS[plan]}), {S} splits",
          flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--keep-index", type=int, default=0,
                    help="which keep ratio of the workload to run")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="measure the headline workload only")
    ap.add_argument("--config-cpu-seconds", type=float, default=6.0,
                    help="oracle time budget of each extra configuration's cpu_baseline")
    ap.add_argument("--blocks", type=int, default=5,
                    help="fresh-process blocks of the headline sparse/dense pair (0: none)")
    ap.add_argument("--block-steps", type=int, default=50)
    ap.add_argument("--block-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--only-step", choices=["sparse", "dense", "entmax_step", "entmax_dense"],
                    help="profiling aid: run warm-up + steps plain kv_decode_step (or entmax "
                         "step / dense entmax) calls, L2 flushed before each, and print no "
                         "benchmark line")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.block_child:
        run_block_child(args)
        return
    if args.only_step:
        run_only_step(args)
        return
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
