"""Data-parallel replica logic on two gloo ranks (CPU): the token shards
partition the global batch, and the step time every rank reports is the max
over ranks."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp

from mixture_experts_ffn_renorm_gb300 import dp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world_size, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world_size), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world_size)
    try:
        ws, r, _ = dp.world()
        lo, hi = dp.shard_range(8193, r, ws)
        my_ms = 1.0 + r          # rank 1 is the slow one
        dp.barrier(ws)
        mx = dp.max_over_ranks(my_ms, ws)
        q.put((r, lo, hi, mx, dp.aggregate_tokens_per_s(hi - lo, ws, mx)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    (r0, lo0, hi0, mx0, v0), (r1, lo1, hi1, mx1, v1) = res
    assert (lo0, hi0, lo1, hi1) == (0, 4097, 4097, 8193)
    assert mx0 == mx1 == 2.0
    assert v0 == pytest.approx(2 * 4097 / 2e-3)


@pytest.mark.parametrize("n,w", [(10, 3), (8192, 8), (1, 4), (0, 2)])
def test_shard_range_partitions(n, w):
    spans = [dp.shard_range(n, r, w) for r in range(w)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    assert max(h - l for l, h in spans) - min(h - l for l, h in spans) <= 1
