"""The multi-GPU form of the bench is independent replicas (one per rank, no collective on
the data path); its only cross-rank steps are a barrier and the maximum of the step times
over ranks, and rank 0 alone prints (the reference arm runs on rank 0 only). These run as
two gloo ranks on the CPU."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        got = bench.max_over_ranks([10.0 * (rank + 1), 5.0 - rank, rank], world, "cpu")
        dist.barrier()
        # the reference arm: ranks other than 0 return at once, without work or output
        class A:
            workload = "tiny_fp32"
            keep_index = 0
            warmup = 0
            steps = 0
        ref = bench.run_reference(A()) if rank != 0 else None
        out.put((rank, got, ref))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks_and_rank0_only_reference():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, ref in res:
        assert got == [20.0, 5.0, 1.0]
        assert ref is None


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2], 1, "cpu") == [1.5, 2.0]
