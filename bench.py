"""Decode-attention benchmark: sparse paged-KV decode step vs the dense step, on GB300.

A step is one sparse decode step over the whole batch: page scores, top-k selection,
split-K attention over the selected pages and the log-sum-exp merge (the page statistics
already exist; their build is timed separately). The dense step is the same attention
kernel with every page kept, plus the merge. Inputs are resident in HBM; L2 is flushed
(a 256 MiB write, twice the L2) before every timed step, outside the timed events.

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


def file_hash(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def committed_traffic(workload, keep_label, source):
    """Per-launch DRAM bytes of the timed kernel from a committed ncu summary, if the
    kernel source has not changed since the counters were taken."""
    p = os.path.join(PROFILE_DIR, f"{os.path.basename(source).split('.')[0]}_{workload}.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("source_hash") != file_hash(source):
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
    # the kernels kv_decode_step runs for this shape (KV_PLAN_*)
    plan, S_plan = (skv.kv_decode_step_plan(kv, Hq, k_max=k_max, **step_kw)
                    if step_kw is not None else (0, S))
    dense_plan, _ = skv.kv_decode_step_plan(kv, Hq, keep_ratio=1.0)
    two_launch = plan in (1, 2)
    assert S_plan == S, (S_plan, S)
    # the other two-launch form, timed beside it where the shape allows
    alt_plan = None
    if step_kw is not None:
        for cand in ((2,) if plan == 1 else (1,) if plan == 2 else (1, 2)):
            try:
                if cand == 1:
                    skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores.zero_(), k_max=k_max,
                                              num_splits=S, part_acc=acc, part_ml=ml,
                                              counters=ctr2, out=out, lse=lse, **step_kw)
                else:
                    skv.kv_score_select(kv, c.q, stats, k_max=k_max, scores=scores,
                                        counters=ctr, sel_idx=sel, sel_cnt=cnt, **step_kw)
                    skv.kv_decode_attn_merge(kv, c.q, w.sm_scale, sel, cnt, num_splits=S,
                                             part_acc=acc, part_ml=ml, counters=ctr2, out=out,
                                             lse=lse)
                alt_plan = cand
                break
            except binding.KVError:
                continue
        torch.cuda.synchronize()

    try:
        marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
        smarks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
        in_graph_events = True
    except TypeError:
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        smarks = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        in_graph_events = False

    def plan_step(which, with_marks=False):
        """A two-launch plan's kernels, called one by one through the C ABI."""
        if with_marks:
            smarks[0].record()
        if which == 1:
            skv.kv_score_pages(kv, c.q, stats, scores)
        else:
            skv.kv_score_select(kv, c.q, stats, k_max=k_max, scores=scores, counters=ctr,
                                sel_idx=sel, sel_cnt=cnt, **step_kw)
        if with_marks:
            smarks[1].record()
        if which == 1:
            skv.kv_select_decode_attn(kv, c.q, w.sm_scale, scores, k_max=k_max, num_splits=S,
                                      part_acc=acc, part_ml=ml, counters=ctr2, out=out,
                                      lse=lse, sel_idx=sel, sel_cnt=cnt, **step_kw)
        else:
            skv.kv_decode_attn_merge(kv, c.q, w.sm_scale, sel, cnt, num_splits=S, part_acc=acc,
                                     part_ml=ml, counters=ctr2, out=out, lse=lse)
        if with_marks:
            smarks[2].record()

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
    g_step, g_dense, g_four, g_marked, g_one, g_smarked, g_alt, g_fp8, g_ent, g_entd = (
        torch.cuda.CUDAGraph() for _ in range(10))
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
    step_kern_us = {"first": [], "attention": []}
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

    # dropped mass of this step (diagnostic, outside every timed region)
    delta = skv.kv_dropped_mass(kv, c.q, w.sm_scale, sel, cnt)
    delta_mean = float(delta.mean())

    # ---- end to end through the public call, host buffers, copies inside the timing -----
    q_host = c.q.detach().cpu().pin_memory()
    out_host = torch.empty((B, Hq, D), dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(c.q)
    e2e_us = []
    if step_kw is not None:
        for i in range(args.warmup + min(args.steps, 500)):
            flush.zero_()
            torch.cuda.synchronize()
            h0 = time.perf_counter()
            q_dev.copy_(q_host, non_blocking=True)
            skv.kv_decode_step(kv, q_dev, w.sm_scale, stats, k_max=k_max, out=out, lse=lse,
                               workspace=ws, **step_kw)
            out_host.copy_(out, non_blocking=True)
            torch.cuda.synchronize()
            if i >= args.warmup:
                e2e_us.append((time.perf_counter() - h0) * 1e6)

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
        roof_kernel = ATTN_KERNEL[w.dtype][0] + (" (select + attend + merge)" if plan == 1
                                                 else " (attend + merge)")
        roof_bytes = acct["step_attn_launch"] + (acct["scores_bytes"] if plan == 1 else 0)
        roof_us = statistics.mean(step_kern_us["attention"])
        roof_source = ATTN_KERNEL[w.dtype][1]
    else:
        roof_kernel, roof_bytes, roof_us = ATTN_KERNEL[w.dtype][0], acct["attn_launch"], attn_us
        roof_source = ATTN_KERNEL[w.dtype][1]
    achieved = roof_bytes / (roof_us * 1e-6) / 1e9
    # kernels per replay of each timed graph
    n_step = 1 if one_launch else (2 if two_launch else 4)
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
                                      + (2 if two_launch else 0) + (1 if one_us else 0)
                                      + (2 if alt_us else 0)
                                      + (n_step if fp8_us else 0) + 4 + 2),
        "clocks": clocks,
    }
    if e2e_us:
        line["e2e"] = {"value": round(statistics.median(e2e_us), 3), "unit": "us/step",
                       "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
                       "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
                       "api": "kv_decode_step"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(c, w, keep, budget_s=args.cpu_seconds)
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
    ap.add_argument("--only-step", choices=["sparse", "dense"],
                    help="profiling aid: run warm-up + steps plain kv_decode_step calls "
                         "(L2 flushed before each) and print no benchmark line")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.only_step:
        run_only_step(args)
        return
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
