"""The multi-rank timing logic of bench.py (replicas, max over ranks) on CPU with gloo."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    env = bench.dist_env()
    bench.barrier(ws)
    t = bench.max_over_ranks(1.5 + rank, ws)  # rank 1 is the slow one
    dist.destroy_process_group()
    q.put((rank, env, t))


@pytest.mark.parametrize("ws", [2])
def test_max_over_ranks_gloo(ws):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, t in res:
        assert env == (ws, rank, rank)
        assert t == 1.5 + (ws - 1)


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25
