"""The bench's multi-rank harness on CPU: two gloo ranks, barrier and max/sum of scalars.

Decode shards by sequence with no data-path collective; each rank times its own
batch and the harness reports the max time and the summed bytes over ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench

    d = bench.Dist()
    try:
        d.barrier()
        t_max = d.max(10.0 + rank)
        b_sum = d.sum(1000.0 * (rank + 1))
        d.barrier()
        q.put((rank, d.world, t_max, b_sum))
    finally:
        d.close()


def test_two_gloo_ranks_reduce_time_and_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, world, t_max, b_sum in res:
        assert world == 2 and t_max == 11.0 and b_sum == 3000.0


def test_single_rank_is_identity():
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    d = bench.Dist()
    assert d.world == 1 and d.max(3.5) == 3.5 and d.sum(2.0) == 2.0
    d.barrier()
    d.close()


def test_step_bytes_accounting():
    import bench
    from paged_kv_cache_91_gb300 import workloads as W

    b = W.build_batch(seed=1, context_lens=[100, 600, 1100], num_heads=8, num_kv_heads=2, head_dim=128,
                      block_size=16, dtype="f16")
    kv, call = bench.step_bytes(b, 512)
    assert kv == 1800 * 2 * 128 * 2 * 2
    tables = (7 + 38 + 69) * 4 + 3 * 4
    partials = (2 + 3) * 8 * 130 * 4 * 2
    assert call == kv + 2 * 3 * 8 * 128 * 2 + tables + partials
