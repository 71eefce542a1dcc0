"""bench.py's multi-rank host logic on CPU: two gloo ranks (no GPU).

Under torchrun every rank runs an independent replica of the decode step
(sequences shard across GPUs with no exchange step); the only communication is
the timing barrier and the max over ranks of the per-step time.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports its own step time; every rank must see the maximum
    got = bench.all_max(1.0 + rank * 0.5, w)
    out[rank] = got
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        assert dict(out) == {0: 1.5, 1: 1.5}
