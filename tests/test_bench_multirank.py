"""The benchmark's multi-rank host logic on CPU: two gloo ranks agree on the
maximum time over ranks (the N > 1 timing rule), and the committed traffic
record is tied to the kernel sources."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [31.5, 29.25][rank]
        results[rank] = bench.max_over_ranks(local_ms, world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1] == 31.5


def test_single_rank_is_identity():
    assert bench.max_over_ranks(12.5, 1) == 12.5


def test_traffic_record_matches_sources():
    # the committed summary was taken on the current kernel sources, or is reported as unknown
    t = bench.profiled_traffic("zigzag_prefill_64k_rope")
    assert t is None or t > 10**9
    assert bench.profiled_traffic("no_such_workload") is None
