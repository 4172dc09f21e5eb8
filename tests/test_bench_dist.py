"""Host logic of the multi-GPU benchmark path, on CPU with gloo (world size 2):
max-over-ranks timing and the weak-scaling whole-job value."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    env = bench.dist_env()
    t = bench.max_over_ranks(10.0 + 5 * rank, ws)
    bench.barrier(ws)
    v = bench.weak_scaling_value(1e12, t, 4, ws)
    q.put((rank, env, t, v))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo():
    ws = 2
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
    for rank, env, t, v in res:
        assert env == (ws, rank, rank)
        assert t == 15.0  # the slower rank sets the time
        # 2 ranks x 4 steps x 1 TFLOP in 15 ms
        assert v == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_rank_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.weak_scaling_value(2e12, 1000.0, 1, 1) == pytest.approx(2.0)
