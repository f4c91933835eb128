"""The N>1 path of the benchmark on CPU: two gloo ranks, each with its own
shard (different seed, same shapes), a max-over-ranks of the step time and
the whole-job unit count — no collective touches the data."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from paged_kv_cache_313_gb300 import sharding
        from paged_kv_cache_313_gb300 import workloads as W

        w = W.tiny_fp32(sharding.shard_seed(0, rank))
        t_step = 1.0 + rank  # pretend rank 1 is slower
        mx = sharding.max_over_ranks([t_step, 10.0 * (world - rank)])
        units = sharding.total_units(w.num_decode)
        q.put((rank, w.q_decode.sum().item(), tuple(w.q_decode.shape), mx, units))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, shp0, mx0, u0), (r1, s1, shp1, mx1, u1) = res
    assert shp0 == shp1 and s0 != s1  # same shapes, different data
    assert mx0 == mx1 == [2.0, 20.0]  # max over ranks
    assert u0 == u1 == 8  # 4 decode tokens per rank x 2 ranks


def test_single_process_is_identity():
    from paged_kv_cache_313_gb300 import sharding
    assert sharding.max_over_ranks([3.0]) == [3.0]
    assert sharding.total_units(64) == 64
