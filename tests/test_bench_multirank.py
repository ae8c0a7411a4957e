"""bench.py's multi-rank logic with world_size 2 on the gloo backend (CPU):
replicas only, the step time is the max over ranks and the value counts the
tokens of every rank."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    step_ms = [3.0, 5.0][rank]
    mx = bench.max_over_ranks(step_ms, world)
    tokens = bench.sum_over_ranks(13312.0, world)
    bench.barrier(world)
    q.put((rank, mx, tokens, tokens / (mx / 1e3)))
    dist.destroy_process_group()


def test_two_rank_reduction():
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
    for rank, mx, tokens, value in out:
        assert mx == 5.0 and tokens == 2 * 13312.0
        assert abs(value - 2 * 13312 / 5e-3) < 1e-6
