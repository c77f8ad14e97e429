"""The N > 1 path of bench.py on the CPU: two gloo ranks (torch.distributed)
exercise the weak-scaling host logic -- per-rank batches, the max over ranks
of the timings, the whole-job value -- and the reference arm's rank-0-only
rule.  The library has no multi-GPU code: ranks are independent replicas."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_30_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [5.0, 7.5][rank]
        slowest = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        prob = W.tiny_gqa(bench.rank_seed(0, rank))
        digest = float(prob.q.float().sum()), tuple(prob.q.shape), int(prob.seq_lens.sum())
        # the reference arm runs on rank 0 only; other ranks return at once
        ran = bench.run_reference(None, rank, world) if rank != 0 else "rank0"
        out.put((rank, slowest, digest, ran))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, d0, ran0), (r1, s1, d1, ran1) = res
    assert s0 == s1 == 7.5                      # max over ranks, seen by both
    assert d0[1] == d1[1] and d0[0] != d1[0]    # same shapes, a different draw per rank
    assert ran1 is None                         # reference arm: rank 1 does no work
    # whole-job value: both ranks' bytes over the slowest step time
    assert bench.job_value(2, 10**9, 7.5) == pytest.approx(2 * 10**9 / 7.5e-3 / 1e9)


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.rank_seed(5, 0) == 5 and bench.rank_seed(5, 1) != 5
