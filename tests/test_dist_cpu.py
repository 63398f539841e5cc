"""Host logic of the multi-GPU bench path on CPU: two gloo ranks (127.0.0.1)
check the token sharding (disjoint, covering, equal per-rank batches) and the
max-over-ranks timing reduction that bench.py uses under torchrun."""

import os
import socket

import pytest


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = bench.shard_rows(20480, world, rank)
    t = bench.max_over_ranks(1.0 + rank * 0.5, world)
    bench.barrier(world)
    q.put((rank, lo, hi, t))
    dist.destroy_process_group()


def test_two_rank_sharding_and_max_timing():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, lo0, hi0, t0), (r1, lo1, hi1, t1) = out
    assert (lo0, hi0, lo1, hi1) == (0, 20480, 20480, 40960)   # each rank its own 20480-token batch
    assert t0 == t1 == 1.5                                     # the slowest rank's time on every rank


def test_env_defaults_single_process(monkeypatch):
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25
