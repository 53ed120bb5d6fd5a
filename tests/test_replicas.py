"""Replica bookkeeping on CPU: sequence sharding and the cross-rank timing reductions,
with two gloo ranks (the data path itself has no collective)."""
import os
import socket

import pytest

from sparse_kv_cache_rank_gb300 import replicas


@pytest.mark.parametrize("B,world", [(1, 1), (8, 2), (7, 2), (3, 4), (16, 8), (0, 3)])
def test_shard_sequences_partition(B, world):
    spans = [replicas.shard_sequences(B, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == B
    for (a, b), (c, d) in zip(spans, spans[1:]):
        assert b == c
    sizes = [b - a for a, b in spans]
    assert max(sizes) - min(sizes) <= 1


def test_shard_sequences_rejects_bad_rank():
    with pytest.raises(ValueError):
        replicas.shard_sequences(4, 2, 2)


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = replicas.env_rank()
    mx = replicas.max_over_ranks([1.0 + rank, 10.0 - rank])
    sm = replicas.sum_over_ranks([rank + 1])
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, r, w, lr, mx, sm))


def test_two_gloo_ranks_reduce_timings():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    q = ctx.Queue()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, lr, mx, sm in res:
        assert (r, w, lr) == (rank, 2, rank)
        assert mx == [2.0, 10.0]
        assert sm == [3.0]
