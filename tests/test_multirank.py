"""World-size-2 gloo run of the multi-rank host logic used by the benchmark: disjoint
shards that cover every unit, and the max-over-ranks time reduction.  CPU only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from sparse_attention_compress_gb300.dist import max_over_ranks, shard_range


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, n_units, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, hi = shard_range(n_units, rank, world)
        t = max_over_ranks(1.5 + rank)  # each rank "measured" a different time
        dist.barrier()
        q.put((rank, lo, hi, t))
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_and_max_time():
    world, n_units = 2, 131072 + 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n_units, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    spans = [(lo, hi) for _, lo, hi, _ in res]
    assert spans[0][0] == 0 and spans[-1][1] == n_units
    assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
    assert all(t == 2.5 for *_, t in res)


@pytest.mark.parametrize("n,world", [(0, 3), (5, 8), (131072, 4), (7, 1)])
def test_shard_range_partitions(n, world):
    got = [shard_range(n, r, world) for r in range(world)]
    assert got[0][0] == 0 and got[-1][1] == n
    sizes = [hi - lo for lo, hi in got]
    assert max(sizes) - min(sizes) <= 1
