"""Multi-rank host logic on CPU: GQA-group sharding and the max over ranks (gloo, 2 ranks)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from dynamic_sparse_attention_vertical_gb300.shard import gqa_shard, layers_per_ms, reduce_max


@pytest.mark.parametrize("Hq,Hkv,world", [(32, 8, 1), (32, 8, 2), (32, 8, 3), (32, 8, 8), (32, 8, 12),
                                          (8, 8, 3), (64, 4, 4)])
def test_gqa_shard_partitions_whole_groups(Hq, Hkv, world):
    g = Hq // Hkv
    shards = [gqa_shard(Hq, Hkv, r, world) for r in range(world)]
    flat = [h for s in shards for h in s]
    assert sorted(flat) == list(range(Hq))  # every head once
    for s in shards:
        assert len(s) % g == 0  # whole GQA groups
        assert {h // g for h in s} == set(range(s[0] // g, s[0] // g + len(s) // g)) if s else True
    sizes = [len(s) // g for s in shards]
    assert max(sizes) - min(sizes) <= 1


def test_gqa_shard_errors_and_helpers():
    with pytest.raises(ValueError):
        gqa_shard(30, 8, 0, 1)
    with pytest.raises(ValueError):
        gqa_shard(32, 8, 2, 2)
    assert reduce_max(3.5) == 3.5
    assert layers_per_ms(40.0, 4) == 10.0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank times its own replica; the job reports the slowest
        my_ms = 10.0 + 5.0 * rank
        dist.barrier()
        ms_max = reduce_max(my_ms, dist)
        heads = gqa_shard(32, 8, rank, world)
        gathered = [None] * world
        dist.all_gather_object(gathered, heads)
        q.put((rank, ms_max, layers_per_ms(ms_max, world), gathered))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_max_and_shards():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, per_layer, gathered in results:
        assert ms_max == 15.0  # the slower rank's time on every rank
        assert per_layer == 7.5
        assert sorted(h for s in gathered for h in s) == list(range(32))
        assert gathered[0] == list(range(0, 16)) and gathered[1] == list(range(16, 32))
