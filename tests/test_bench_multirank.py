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


def _shard_main(rank, world, port, H, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        h0, h1 = bench.shard_heads(H, world, rank)
        # every rank learns every rank's range: they must tile [0, H) with no overlap
        ranges = [None] * world
        dist.all_gather_object(ranges, (h0, h1))
        results[rank] = ranges
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("H,world", [(32, 2), (7, 2)])
def test_shard_heads_gloo_tiles_the_heads(H, world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, world, port, H, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    ranges = results[0]
    assert all(results[r] == ranges for r in range(world))
    assert ranges[0][0] == 0 and ranges[-1][1] == H
    assert all(ranges[i][1] == ranges[i + 1][0] for i in range(world - 1))
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_shard_heads_single_process_cases():
    assert bench.shard_heads(32, 1, 0) == (0, 32)
    assert [bench.shard_heads(10, 4, r) for r in range(4)] == [(0, 3), (3, 6), (6, 8), (8, 10)]
    with pytest.raises(ValueError):
        bench.shard_heads(8, 2, 2)


def test_e2e_groups_split_heads():
    def heads(sl):
        return [(ix[1].start, ix[1].stop) for ix in sl]
    # default at 32 heads: small first and last groups, tiling [0, 32)
    assert heads(bench.e2e_groups(1, 32)) == [(0, 2), (2, 8), (8, 16), (16, 24), (24, 30), (30, 32)]
    # an explicit split, and equal groups when asked for another count
    assert heads(bench.e2e_groups(1, 32, 8, [4, 8, 8, 8, 4])) == [(0, 4), (4, 12), (12, 20), (20, 28), (28, 32)]
    assert heads(bench.e2e_groups(1, 32, 4)) == [(0, 8), (8, 16), (16, 24), (24, 32)]
    # a split that does not cover the heads is ignored: equal groups
    assert heads(bench.e2e_groups(1, 32, 8, [4, 4])) == [(4 * i, 4 * i + 4) for i in range(8)]
    # batch groups, or the whole tensor
    assert bench.e2e_groups(16, 8, 8) == [(slice(2 * i, 2 * i + 2),) for i in range(8)]
    assert bench.e2e_groups(4, 16, 8) == [(slice(None),)]
