"""Replica path across ranks, world size 2 over gloo on the CPU.

The prefill path shards without any exchange: each rank runs its own copy of
the workload. What crosses ranks is only the bench's bookkeeping: the line
reports the slowest rank's step time, and the reference arm runs on rank 0
alone while the other ranks return without work.
"""
import argparse
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        ms = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        ref = "rank0"
        if rank != 0:
            ref = bench.run_reference(argparse.Namespace(steps=1, warmup=0), rank, world)
        queue.put((rank, ms, ref))
    finally:
        dist.destroy_process_group()


def test_replicas_report_slowest_rank_and_rank0_reference():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict()
    for _ in procs:
        rank, ms, ref = queue.get(timeout=120)
        got[rank] = (ms, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == 2.5 and got[1][0] == 2.5
    assert got[1][1] is None
